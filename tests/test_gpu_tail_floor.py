"""GPU parity with a tail floor (anbeeld.com "KVarN KV Cache: Implementation and
Benchmarks", 2.1: BeeLlama keeps at least one full group of recent tokens exact; here
floors of one and two groups).

Group g is sealed when group g + F fills, so the exact tail holds 128 F .. 128 F + 127
tokens once the body has started, kept in a ring of 128 (F + 1) rows per head. Checked
against the oracle, through the C ABI:
* bulk append and decode steps across seal points: attention equals the oracle's over
  the GPU's records and exact regions (tests/parity.py tolerance);
* the exact tail equals the input tokens bit for bit, in position order;
* every group sealed inside a decode step equals the oracle's seal of its tokens (the
  decoupled seal protocol of tests/parity.py).
"""
import math

import numpy as np
import pytest

import oracle
from quantized_kv_cache_seal_gb300 import kvarn as K
from quantized_kv_cache_seal_gb300 import workloads
from tests import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(128)
HQ, HKV = 8, 2


def _cache(floor, max_len=2048, seqs=2, bits=2):
    from quantized_kv_cache_seal_gb300.cache import KVarNCache
    return KVarNCache(num_layers=1, max_seqs=seqs, num_q_heads=HQ, num_kv_heads=HKV, k_bits=bits, v_bits=bits,
                      max_seq_len=max_len, tail_floor=floor)


def _records(cache, seq, kvh, which, n_groups):
    if n_groups == 0:
        return np.zeros(0, np.uint8)
    return np.stack([cache.record(0, seq, g, kvh, which).cpu().numpy() for g in range(n_groups)])


def _check_attention(cache, floor, seq, q, out, label, bits=2):
    n = cache.length(0, seq)
    n_sink = min(n, 128)
    n_groups = max(max(n - 128, 0) // 128 - floor, 0)
    sk, sv = [t.cpu().numpy() for t in cache.exact_regions(0, seq)[:2]]
    tk, tv = [t.cpu().numpy() for t in cache.exact_tail(0, seq)]
    assert tk.shape[1] == max(n - 128, 0) - 128 * n_groups
    r = HQ // HKV
    for h in range(HKV):
        ref = oracle.attention(q[h * r:(h + 1) * r], SCALE, sk[h, :n_sink], sv[h, :n_sink],
                               _records(cache, seq, h, 0, n_groups), _records(cache, seq, h, 1, n_groups),
                               tk[h], tv[h], bits, bits)
        parity.check_attention(out[h * r:(h + 1) * r], ref, f"{label} seq {seq} kvh {h}")


def _tokens(seed, seq, start, count):
    k, v = workloads.torch_tokens(seed, seq, start, count, HKV)
    return k.contiguous(), v.contiguous()


@pytest.mark.parametrize("floor,bits", [(1, 2), (2, 2), (1, 3)])
def test_tail_floor_decode_parity(floor, bits):
    seed = 20 + floor + 10 * bits
    cache = _cache(floor, bits=bits)
    # seq 0: the body has started and sealed; seq 1: still inside the floor (nothing sealed)
    lengths = [128 + 128 * (floor + 2) + 120, 128 + 128 * floor - 3]
    for s, n in enumerate(lengths):
        k, v = _tokens(seed, s, 0, n)
        cache.append(0, [s], [n], k, v)
    torch.cuda.synchronize()
    qs = workloads.torch_queries(seed, 12, 2, HQ)
    for step in range(12):  # seq 0 completes a group at step 7 (120 + 8 = 128); seq 1 reaches the floor
        ks, vs = [], []
        for s in range(2):
            k, v = _tokens(seed, s, lengths[s] + step, 1)
            ks.append(k)
            vs.append(v)
        out = cache.decode_step(0, [0, 1], torch.cat(ks), torch.cat(vs), qs[step])
        torch.cuda.synchronize()
        assert cache.check_device_error() == 0
        if step in (0, 7, 8, 11):
            o = out.float().cpu().numpy()
            q = qs[step].cpu().numpy()
            for s in range(2):
                _check_attention(cache, floor, s, q[s], o[s], f"floor {floor} b{bits} step {step}", bits)
    # the exact tail is the input, bit for bit, in position order
    for s in range(2):
        n = cache.length(0, s)
        ng = max(max(n - 128, 0) // 128 - floor, 0)
        k, v = _tokens(seed, s, 0, n)
        tk, tv = cache.exact_tail(0, s)
        assert torch.equal(tk.permute(1, 0, 2).contiguous().view(torch.int16),
                           k[128 + 128 * ng:n].view(torch.int16))
        assert torch.equal(tv.permute(1, 0, 2).contiguous().view(torch.int16),
                           v[128 + 128 * ng:n].view(torch.int16))
    # the group sealed inside the decode loop: seq 0's body held floor + 2 full groups and
    # 120 tokens; step 7 completed group floor + 2, which seals group 2
    n0 = cache.length(0, 0)
    assert max(n0 - 128, 0) // 128 - floor == 3
    k, v = _tokens(seed, 0, 128 + 128 * 2, 128)
    for h in range(HKV):
        for which, x in ((0, k), (1, v)):
            rec = cache.record(0, 0, 2, h, which).cpu().numpy()
            parity.check_seal(x[:, h].cpu().numpy(), rec, bits, which, label=f"floor {floor} seal kvh {h} side {which}")


def test_tail_floor_bulk_seals_match_published_records():
    """A seal depends only on its group's tokens: a cache with a floor of one group and one
    without seal the same groups into identical records (the floor only delays them)."""
    a, b = _cache(0, seqs=1), _cache(1, seqs=1)
    n = 128 + 128 * 5 + 17
    k, v = _tokens(30, 0, 0, n)
    a.append(0, [0], [n], k, v)
    for c0 in range(0, n, 200):  # the floored cache in chunks, so its seals read the tail ring
        c = min(200, n - c0)
        b.append(0, [0], [c], k[c0:c0 + c].contiguous(), v[c0:c0 + c].contiguous())
    torch.cuda.synchronize()
    for g in range(4):  # groups 0..3 are sealed in both (b: 5 full groups - 1)
        for h in range(HKV):
            for which in (0, 1):
                assert torch.equal(a.record(0, 0, g, h, which), b.record(0, 0, g, h, which)), (g, h, which)
    with pytest.raises(K.KVarNError):
        b.record(0, 0, 4, 0, 0)
