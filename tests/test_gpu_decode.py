"""GPU parity of decode attention over sealed groups (calls through the C ABI).

anbeeld.com "KVarN KV Cache: Implementation and Benchmarks", sections 1 and 2.1: sink
and tail exact, sealed groups read from their records with the rotated query, output
rotated back once. Each GPU output is compared with the oracle's fp64 attention over
the GPU's own records and exact regions (tests/parity.py); the records themselves are
checked against the oracle's seal of the same fp16 tokens.
"""
import math

import numpy as np
import pytest

import oracle
from quantized_kv_cache_seal_gb300 import workloads
from tests import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(128)


def _cache(hq, hkv, kb, vb, max_seqs, max_len, pool=None):
    from quantized_kv_cache_seal_gb300.cache import KVarNCache
    return KVarNCache(num_layers=2, max_seqs=max_seqs, num_q_heads=hq, num_kv_heads=hkv, k_bits=kb, v_bits=vb,
                      max_seq_len=max_len, pool_groups=pool)


def oracle_attention_from_gpu(cache, layer, seq, q_np, heads=None):
    """fp64 attention of q [Hq][d] over the GPU's records and exact regions of (layer, seq)."""
    cfg = cache.cfg
    n = cache.length(layer, seq)
    n_sink = min(n, 128)
    n_groups = max(n - 128, 0) // 128
    n_tail = max(n - 128, 0) % 128
    sk, sv, tk, tv = [t.cpu().numpy() for t in cache.exact_regions(layer, seq)]
    r = cfg.num_q_heads // cfg.num_kv_heads
    out = np.full((cfg.num_q_heads, 128), np.nan)
    for h in (range(cfg.num_kv_heads) if heads is None else heads):
        kr = np.stack([cache.record(layer, seq, g, h, 0).cpu().numpy() for g in range(n_groups)]) \
            if n_groups else np.zeros(0, np.uint8)
        vr = np.stack([cache.record(layer, seq, g, h, 1).cpu().numpy() for g in range(n_groups)]) \
            if n_groups else np.zeros(0, np.uint8)
        if n == 0:
            out[h * r:(h + 1) * r] = 0.0
            continue
        out[h * r:(h + 1) * r] = oracle.attention(q_np[h * r:(h + 1) * r], SCALE, sk[h, :n_sink], sv[h, :n_sink],
                                                  kr, vr, tk[h, :n_tail], tv[h, :n_tail], cfg.k_bits, cfg.v_bits)
    return out


def check_exact_regions(cache, layer, seq, k_all, v_all):
    """The sink and tail hold the appended fp16 bits unchanged."""
    n = cache.length(layer, seq)
    sk, sv, tk, tv = [t.cpu().numpy() for t in cache.exact_regions(layer, seq)]
    ns = min(n, 128)
    assert np.array_equal(sk[:, :ns].view(np.uint16), k_all[:ns].transpose(1, 0, 2).view(np.uint16))
    assert np.array_equal(sv[:, :ns].view(np.uint16), v_all[:ns].transpose(1, 0, 2).view(np.uint16))
    if n > 128:
        nt = (n - 128) % 128
        start = n - nt
        assert np.array_equal(tk[:, :nt].view(np.uint16), k_all[start:n].transpose(1, 0, 2).view(np.uint16))
        assert np.array_equal(tv[:, :nt].view(np.uint16), v_all[start:n].transpose(1, 0, 2).view(np.uint16))


def test_c1_single_head_293_tokens():
    """128 sink + one sealed group + 37 tail tokens, one KV head, one query head, 2/2 bits."""
    wl = workloads.workloads()["c1_single_head_293"]
    cache = _cache(1, 1, 2, 2, 1, 1024)
    src = workloads.TokenSource(wl.seed, 0, 1)
    k, v = src.tokens(0, 293)
    cache.append(0, [0], [293], torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    q = workloads.queries(wl.seed, 0, 1, 1)
    out = cache.decode_attention(0, [0], torch.from_numpy(q).cuda())
    torch.cuda.synchronize()
    assert cache.check_device_error() == 0
    check_exact_regions(cache, 0, 0, k, v)
    for which, x in ((0, k), (1, v)):
        parity.check_seal(x[128:256, 0], cache.record(0, 0, 0, 0, which).cpu().numpy(), 2, which, label="c1")
    ref = oracle_attention_from_gpu(cache, 0, 0, q[0])
    parity.check_attention(out.cpu().numpy()[0], ref, "c1")
    # end to end against the oracle's own cache (its own seal): same tolerance
    oc = oracle.OracleCache(1, 2, 2)
    oc.append(0, k, v)
    parity.check_attention(out.cpu().numpy()[0], oc.attend(0, q[0], SCALE), "c1 oracle cache", tol=2e-2)


LENGTHS = [0, 1, 127, 128, 129, 255, 256, 300, 1000, 1535]


@pytest.mark.parametrize("kb,vb", [(2, 2), (4, 2), (2, 4), (4, 4), (8, 8), (8, 2), (3, 3), (5, 5), (6, 6), (6, 5),
                                   (5, 4), (3, 2)])
def test_mixed_lengths(kb, vb):
    """Sink only, group boundaries, several groups, ragged tails; r = 4."""
    hq, hkv = 8, 2
    cache = _cache(hq, hkv, kb, vb, len(LENGTHS), 2048)
    ids = list(range(len(LENGTHS)))
    srcs = [workloads.TokenSource(40 + i, i, hkv) for i in ids]
    toks = [s.tokens(0, n) for s, n in zip(srcs, LENGTHS)]
    k = np.concatenate([t[0] for t in toks])
    v = np.concatenate([t[1] for t in toks])
    cache.append(1, ids, LENGTHS, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    q = workloads.queries(5, kb * 10 + vb, len(ids), hq)
    out = cache.decode_attention(1, ids, torch.from_numpy(q).cuda()).cpu().numpy()
    assert cache.check_device_error() == 0
    for i, n in enumerate(LENGTHS):
        check_exact_regions(cache, 1, i, *toks[i])
        ref = oracle_attention_from_gpu(cache, 1, i, q[i])
        parity.check_attention(out[i], ref, f"seq {i} n {n}")
    # every record of one sequence against the oracle's seal
    n = LENGTHS[-1]
    for g in range((n - 128) // 128):
        for h in range(hkv):
            for which, x in ((0, toks[-1][0]), (1, toks[-1][1])):
                parity.check_seal(x[128 + 128 * g:256 + 128 * g, h], cache.record(1, len(ids) - 1, g, h, which)
                                  .cpu().numpy(), kb if which == 0 else vb, which, label=f"g{g} h{h} w{which}")


def test_decode_step_streaming_equals_bulk():
    """Fused decode steps (append + seal + attend) across three seals per sequence:
    every output matches the oracle over the GPU records, and the records sealed one
    token at a time are byte-identical to those of a bulk append (pseudo-decode,
    fig1.dev 'Practical takeaway')."""
    hq, hkv = 8, 2
    starts = [250, 300, 383]
    steps = 260
    cache = _cache(hq, hkv, 2, 2, 3, 1024)
    bulk = _cache(hq, hkv, 2, 2, 3, 1024)
    srcs = [workloads.TokenSource(60 + i, i, hkv) for i in range(3)]
    toks = [src.tokens(0, st + steps) for src, st in zip(srcs, starts)]
    k0 = np.concatenate([t[0][:st] for t, st in zip(toks, starts)])
    v0 = np.concatenate([t[1][:st] for t, st in zip(toks, starts)])
    cache.append(0, [0, 1, 2], starts, torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda())
    for step in range(steps):
        kn = np.stack([t[0][st + step] for t, st in zip(toks, starts)])
        vn = np.stack([t[1][st + step] for t, st in zip(toks, starts)])
        q = workloads.queries(77, step, 3, hq)
        out = cache.decode_step(0, [0, 1, 2], torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(),
                                torch.from_numpy(q).cuda())
        if step % 23 == 0 or any((st + step - 128) % 128 == 127 for st in starts):
            o = out.cpu().numpy()
            for i in range(3):
                parity.check_attention(o[i], oracle_attention_from_gpu(cache, 0, i, q[i]), f"step {step} seq {i}")
    torch.cuda.synchronize()
    assert cache.check_device_error() == 0
    kall = np.concatenate([t[0] for t in toks])
    vall = np.concatenate([t[1] for t in toks])
    bulk.append(0, [0, 1, 2], [st + steps for st in starts], torch.from_numpy(kall).cuda(),
                torch.from_numpy(vall).cuda())
    for i, st in enumerate(starts):
        n = st + steps
        assert cache.length(0, i) == n
        check_exact_regions(cache, 0, i, *toks[i])
        for g in range((n - 128) // 128):
            for h in range(hkv):
                for which in (0, 1):
                    a = cache.record(0, i, g, h, which).cpu().numpy()
                    b = bulk.record(0, i, g, h, which).cpu().numpy()
                    assert np.array_equal(a, b), (i, g, h, which)


def test_decode_step_equals_append_then_attend():
    hq, hkv = 8, 2
    a = _cache(hq, hkv, 4, 2, 2, 1024)
    b = _cache(hq, hkv, 4, 2, 2, 1024)
    srcs = [workloads.TokenSource(90 + i, i, hkv) for i in range(2)]
    starts = [254, 383]
    toks = [s.tokens(0, st + 3) for s, st in zip(srcs, starts)]
    k0 = np.concatenate([t[0][:st] for t, st in zip(toks, starts)])
    v0 = np.concatenate([t[1][:st] for t, st in zip(toks, starts)])
    for c in (a, b):
        c.append(0, [0, 1], starts, torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda())
    for step in range(3):
        kn = torch.from_numpy(np.stack([t[0][st + step] for t, st in zip(toks, starts)])).cuda()
        vn = torch.from_numpy(np.stack([t[1][st + step] for t, st in zip(toks, starts)])).cuda()
        q = torch.from_numpy(workloads.queries(91, step, 2, hq)).cuda()
        oa = a.decode_step(0, [0, 1], kn, vn, q).cpu().numpy().astype(np.float64)
        b.append(0, [0, 1], [1, 1], kn, vn)
        ob = b.decode_attention(0, [0, 1], q).cpu().numpy().astype(np.float64)
        for i in range(2):
            nrm = np.linalg.norm(ob[i], axis=-1).min()
            assert np.abs(oa[i] - ob[i]).max() <= 2e-3 * nrm
    for i, st in enumerate(starts):
        for g in range((st + 3 - 128) // 128):
            for h in range(hkv):
                for which in (0, 1):
                    assert np.array_equal(a.record(0, i, g, h, which).cpu().numpy(),
                                          b.record(0, i, g, h, which).cpu().numpy())


def test_repeated_calls_are_deterministic():
    cache = _cache(8, 2, 2, 2, 2, 2048)
    src = [workloads.TokenSource(5 + i, i, 2) for i in range(2)]
    toks = [s.tokens(0, 1500) for s in src]
    cache.append(0, [0, 1], [1500, 1500], torch.from_numpy(np.concatenate([t[0] for t in toks])).cuda(),
                 torch.from_numpy(np.concatenate([t[1] for t in toks])).cuda())
    q = torch.from_numpy(workloads.queries(3, 0, 2, 8)).cuda()
    o1 = cache.decode_attention(0, [0, 1], q).clone()
    for _ in range(5):
        o2 = cache.decode_attention(0, [0, 1], q)
        assert torch.equal(o1, o2)
    # another batch order changes the split boundaries, not the result beyond rounding
    o3 = cache.decode_attention(0, [1, 0], q.flip(0)).flip(0).double()
    ref = o1.double()
    for i in range(2):
        for hh in range(8):
            assert (o3[i, hh] - ref[i, hh]).abs().max() <= 2e-3 * ref[i, hh].norm()
