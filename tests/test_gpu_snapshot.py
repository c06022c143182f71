"""Cache snapshots on the GPU: save, restore into another cache, and go on.

A restored cache must hold the same bytes (records of every sealed group, the exact
sink and tail regions) and then give bit-identical results for every later call:
decode steps that seal new groups, decode attention and prefill attention. The
snapshot is an interface addition (the pages have no counterpart); its correctness is
equality with the cache it came from.
"""
import os

import pytest

from quantized_kv_cache_seal_gb300 import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

HQ, HKV = 8, 2


def _cache(floor=0):
    from quantized_kv_cache_seal_gb300.cache import KVarNCache
    return KVarNCache(num_layers=2, max_seqs=3, num_q_heads=HQ, num_kv_heads=HKV, k_bits=4, v_bits=2,
                      max_seq_len=2048, tail_floor=floor)


def _fill(cache, lengths, seed):
    for layer in (0, 1):
        for s, n in enumerate(lengths):
            if n == 0:
                continue
            k, v = workloads.torch_tokens(seed + layer, s, 0, n, HKV)
            cache.append(layer, [s], [n], k.contiguous(), v.contiguous())


def _same_state(a, b, lengths, floor=0):
    for layer in (0, 1):
        for s in range(len(lengths)):
            n = a.length(layer, s)
            assert b.length(layer, s) == n
            for g in range(max(max(n - 128, 0) // 128 - floor, 0)):
                for h in range(HKV):
                    for which in (0, 1):
                        assert torch.equal(a.record(layer, s, g, h, which), b.record(layer, s, g, h, which))
            for ra, rb in zip(a.exact_regions(layer, s), b.exact_regions(layer, s)):
                assert torch.equal(ra.view(torch.int16), rb.view(torch.int16))


def _steps(cache, lengths, seed, steps):
    outs = []
    for st in range(steps):
        ks, vs = [], []
        for s in range(len(lengths)):
            k, v = workloads.torch_tokens(seed, s, 5000 + st, 1, HKV)
            ks.append(k)
            vs.append(v)
        q = workloads.torch_queries(seed, steps, len(lengths), HQ)[st].contiguous()
        outs.append(cache.decode_step(0, list(range(len(lengths))), torch.cat(ks).contiguous(),
                                      torch.cat(vs).contiguous(), q))
    q = workloads.torch_queries(seed + 1, 40, 1, HQ)[:, 0].contiguous()
    outs.append(cache.prefill_attention(1, [1], [40], q))
    outs.append(cache.decode_attention(1, [0, 1, 2], workloads.torch_queries(seed + 2, 1, 3, HQ)[0].contiguous()))
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("floor", [0, 1])
def test_restore_into_another_cache_is_bit_identical(floor):
    lengths = [1000, 384 + 127, 90]  # the second one seals on its first decode step (floor 0)
    a, b = _cache(floor), _cache(floor)
    _fill(a, lengths, 10)
    _fill(b, [300, 0, 700], 20)  # different state, replaced by the load
    img = a.snapshot()
    b.restore(img)
    torch.cuda.synchronize()
    assert b.check_device_error() == 0
    _same_state(a, b, lengths, floor)
    oa = _steps(a, lengths, 30, 3)
    ob = _steps(b, lengths, 30, 3)
    for i, (x, y) in enumerate(zip(oa, ob)):
        assert torch.equal(x, y), f"call {i}"
    _same_state(a, b, lengths, floor)  # including the groups sealed after the restore
    assert a.check_device_error() == 0 and b.check_device_error() == 0


def test_save_to_file_and_load(tmp_path):
    lengths = [700, 260, 1300]
    a, c = _cache(), _cache()
    _fill(a, lengths, 40)
    path = os.path.join(tmp_path, "cache.kvarn")
    a.save(path)
    c.load(path)
    _same_state(a, c, lengths)
    for x, y in zip(_steps(a, lengths, 50, 2), _steps(c, lengths, 50, 2)):
        assert torch.equal(x, y)
