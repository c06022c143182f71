"""The allocation-free decode call (kvarn_decode_attention_noalloc), for callers that
cannot allocate device memory (an engine plugin limited to the engine's own memory
pool, a process under a hard device-memory cap). Its split-K scratch lives in a static
device array of the library; this file checks, through the C ABI, that two calls in a
row give the same attention as kvarn_decode_attention, bit for bit, without taking
device memory, also at the largest cache the array takes, and that a cache too large for
the array is refused. It is named to be collected last."""
import math

import numpy as np
import pytest

from quantized_kv_cache_seal_gb300 import kvarn as K
from quantized_kv_cache_seal_gb300 import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3  # max |o - o_ref| <= TOL * ||o_ref||_2 per (sequence, head), as in the decode tests


def _fill(cache, lengths, hkv):
    ids = list(range(len(lengths)))
    toks = [workloads.TokenSource(500 + i, i, hkv).tokens(0, n) for i, n in enumerate(lengths)]
    k = np.concatenate([t[0] for t in toks])
    v = np.concatenate([t[1] for t in toks])
    cache.append(0, ids, lengths, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    return ids


def _check_twice(max_seqs, lengths, decode_ids):
    """Two noalloc calls in a row against kvarn_decode_attention on the same cache and
    queries: the same kernel and schedule run, so the outputs are bit-identical (hence
    also within the decode tolerance); the second call leaves the device's free memory
    unchanged."""
    from quantized_kv_cache_seal_gb300.cache import KVarNCache
    hq, hkv = 32, 8
    cache = KVarNCache(num_layers=1, max_seqs=max_seqs, num_q_heads=hq, num_kv_heads=hkv, k_bits=2, v_bits=2,
                       max_seq_len=max(lengths) + 128)
    _fill(cache, lengths, hkv)
    ids = list(decode_ids)
    q = torch.from_numpy(workloads.queries(9, 0, len(ids), hq)).cuda()
    scale = 1.0 / math.sqrt(128)
    ref = torch.empty_like(q)
    K.kvarn_decode_attention(cache.handle, 0, ids, q, ref, scale, torch.cuda.current_stream())
    torch.cuda.synchronize()
    refd = ref.double().cpu()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        K.kvarn_decode_attention_noalloc(cache.handle, 0, ids, q, out, scale, torch.cuda.current_stream())
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        if call == 1:
            assert free1 == free0
        assert torch.equal(out, ref)
        o = out.double().cpu()
        assert torch.isfinite(o).all()
        err = (o - refd).abs().amax(dim=-1)
        assert (err <= TOL * refd.norm(dim=-1) + 1e-7).all()
    assert cache.check_device_error() == 0


def test_noalloc_matches_decode_attention_twice():
    lengths = [1, 200, 1000, 3000, 4100]
    _check_twice(len(lengths), lengths, range(len(lengths)))


def test_noalloc_at_the_largest_cache_the_array_takes():
    """max_seqs * num_kv_heads = 128 blocks, the array's limit; the decoded sequences
    include the last one (seq 15), whose partials sit at the end of the array."""
    lengths = [300 + 97 * i for i in range(16)]
    _check_twice(16, lengths, [15, 3, 0, 9])


def test_noalloc_rejects_a_cache_beyond_the_static_workspace():
    from quantized_kv_cache_seal_gb300.cache import KVarNCache
    cache = KVarNCache(num_layers=1, max_seqs=17, num_q_heads=32, num_kv_heads=8, k_bits=2, v_bits=2,
                       max_seq_len=256)
    q = torch.zeros((1, 32, 128), dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(K.KVarNError) as e:
        K.kvarn_decode_attention_noalloc(cache.handle, 0, [0], q, out, 0.1)
    assert e.value.status == 3
    assert "static workspace" in K.kvarn_last_error()
