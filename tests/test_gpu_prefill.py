"""GPU parity of prefill (many-query) attention against the oracle, through the C ABI.

Each query token attends causally to the cache as it stands after its chunk's append
(anbeeld.com "KVarN KV Cache: Implementation and Benchmarks", 2.1 and section 1: the
sink and tail exact, sealed groups from their records). The oracle's prefill attention
runs over the GPU's own records and exact regions (the decoupled protocol of
tests/parity.py), so seal parity and attention parity are checked apart; the records
themselves are checked against the oracle's seal in the seal and decode tests.
Cases: prompts from scratch (queries in the sink, inside sealed groups, in the tail),
chunks on top of a cache (also one whose paired query tiles see different units),
every query head ratio (1, 2, 4), widths 2..8 with the odd ones and the presets, a
tail floor, empty query lists, the fused append + attention, a second layer with
interleaved pool slots and norm spikes at the Phi-4 shape, and sampled rows of the
Qwen3-4B 4096-token prefill.
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


def _cache(hq, hkv, kb, vb, seqs=3, max_len=2048, floor=0):
    from quantized_kv_cache_seal_gb300.cache import KVarNCache
    return KVarNCache(num_layers=1, max_seqs=seqs, num_q_heads=hq, num_kv_heads=hkv, k_bits=kb, v_bits=vb,
                      max_seq_len=max_len, tail_floor=floor)


def _records(cache, seq, kvh, which, n_groups, layer=0):
    if n_groups == 0:
        return np.zeros(0, np.uint8)
    return np.stack([cache.record(layer, seq, g, kvh, which).cpu().numpy() for g in range(n_groups)])


def _check(cache, seq, q, out, kb, vb, floor=0, rows=None, label="", layer=0, heads=None):
    """q, out: [n_q][Hq][128] for the last n_q tokens of `seq`; rows: the query rows to
    check (all by default); heads: the KV heads to check (all by default)."""
    n = cache.length(layer, seq)
    n_q, hq = q.shape[0], q.shape[1]
    hkv = cache.cfg.num_kv_heads
    r = hq // hkv
    n_groups = max(max(n - 128, 0) // 128 - floor, 0)
    sk, sv = [t.cpu().numpy() for t in cache.exact_regions(layer, seq)[:2]]
    tk, tv = [t.cpu().numpy() for t in cache.exact_tail(layer, seq)]
    rows = list(range(n_q)) if rows is None else list(rows)
    pos = [n - n_q + i for i in rows]
    for h in (range(hkv) if heads is None else heads):
        ref = oracle.prefill_attention(q[rows, h * r:(h + 1) * r], pos, SCALE, sk[h, :min(n, 128)],
                                       sv[h, :min(n, 128)], _records(cache, seq, h, 0, n_groups, layer),
                                       _records(cache, seq, h, 1, n_groups, layer), tk[h], tv[h], kb, vb)
        for j, i in enumerate(rows):
            parity.check_attention(out[i, h * r:(h + 1) * r], ref[j], f"{label} seq {seq} kvh {h} token {pos[j]}")


def _tokens(seed, seq, start, count, hkv):
    k, v = workloads.torch_tokens(seed, seq, start, count, hkv)
    return k.contiguous(), v.contiguous()


def _queries(seed, count, hq):
    return workloads.torch_queries(seed, count, 1, hq)[:, 0].contiguous()


@pytest.mark.parametrize("hq,hkv", [(8, 2), (4, 2), (2, 2)])
def test_prompt_from_scratch_every_position(hq, hkv):
    """A whole prompt appended, then every token's query: queries in the sink, in each
    sealed group (masked inside the group) and in the tail, for r = 4, 2, 1."""
    cache = _cache(hq, hkv, 2, 2)
    n = 128 + 128 * 3 + 50
    k, v = _tokens(40 + hq, 0, 0, n, hkv)
    cache.append(0, [0], [n], k, v)
    q = _queries(41 + hq, n, hq)
    out = cache.prefill_attention(0, [0], [n], q)
    torch.cuda.synchronize()
    assert cache.check_device_error() == 0
    _check(cache, 0, q.cpu().numpy(), out.float().cpu().numpy(), 2, 2, label=f"r {hq // hkv}")


def test_prompt_tiles_with_one_to_six_sealed_groups():
    """A 900-token prompt: its query tiles see 0 to 6 sealed groups, so the switch from
    sealed groups to the exact blocks (where the output is rotated back) falls after an
    odd and after an even number of groups, with PV of earlier groups still in flight.
    A completion barrier that a late wait could mistake for an older phase gave errors
    of O(1) in the tiles with an even count; every row is checked."""
    hq, hkv = 8, 2
    cache = _cache(hq, hkv, 2, 2)
    n = 900
    k, v = _tokens(48, 0, 0, n, hkv)
    cache.append(0, [0], [n], k, v)
    q = _queries(49, n, hq)
    out = cache.prefill_attention(0, [0], [n], q)
    torch.cuda.synchronize()
    assert cache.check_device_error() == 0
    _check(cache, 0, q.cpu().numpy(), out.float().cpu().numpy(), 2, 2, label="900")


@pytest.mark.parametrize("hq,hkv", [(8, 2), (2, 2)])
def test_chunk_whose_tile_pairs_see_different_units(hq, hkv):
    """Adjacent query tiles run as one CTA pair over the units of the later tile. A chunk
    of 280 queries at positions 200 .. 479 of a 480-token cache (two sealed groups, the
    tail from 384): with 32-token tiles (r = 4) the first pair's tiles see one and two
    sealed groups, so the earlier tile walks a group that every one of its rows masks,
    and the tile count is odd (a padding tile without valid rows completes the last
    pair); with 128-token tiles (r = 1) the first pair's earlier tile sees none of the
    tail its partner sees. Every row is checked."""
    cache = _cache(hq, hkv, 2, 2)
    k, v = _tokens(70 + hq, 0, 0, 480, hkv)
    cache.append(0, [0], [200], k[:200].contiguous(), v[:200].contiguous())
    cache.append(0, [0], [280], k[200:].contiguous(), v[200:].contiguous())
    q = _queries(71 + hq, 280, hq)
    out = cache.prefill_attention(0, [0], [280], q)
    torch.cuda.synchronize()
    assert cache.check_device_error() == 0
    _check(cache, 0, q.cpu().numpy(), out.float().cpu().numpy(), 2, 2, label=f"pairs r {hq // hkv}")


@pytest.mark.parametrize("kb,vb", [(4, 2), (3, 3), (8, 8), (6, 5), (5, 4), (3, 2), (2, 8)])
def test_chunks_on_a_cache_at_every_width(kb, vb):
    """Three sequences in one call: a chunk on top of a longer cache (ragged tile), a
    short prompt inside the sink, and a sequence with no queries."""
    cache = _cache(8, 2, kb, vb)
    lengths = [900, 70, 400]
    for s, n in enumerate(lengths):
        k, v = _tokens(50, s, 0, n, 2)
        cache.append(0, [s], [n], k, v)
    q_lens = [150, 70, 0]
    q = _queries(51, sum(q_lens), 8)
    out = cache.prefill_attention(0, [0, 1, 2], q_lens, q)
    torch.cuda.synchronize()
    assert cache.check_device_error() == 0
    qn, on = q.cpu().numpy(), out.float().cpu().numpy()
    _check(cache, 0, qn[:150], on[:150], kb, vb, label=f"{kb}/{vb}")
    _check(cache, 1, qn[150:], on[150:], kb, vb, label=f"{kb}/{vb}")


def test_tail_floor():
    """With a floor of one group the exact tail holds 128 .. 255 tokens in its ring."""
    cache = _cache(8, 2, 2, 2, floor=1)
    n = 128 + 128 * 4 + 77
    k, v = _tokens(60, 0, 0, n, 2)
    for c0 in range(0, n, 300):  # chunked, so the ring wraps
        c = min(300, n - c0)
        cache.append(0, [0], [c], k[c0:c0 + c].contiguous(), v[c0:c0 + c].contiguous())
    q = _queries(61, 260, 8)
    out = cache.prefill_attention(0, [0], [260], q)
    torch.cuda.synchronize()
    assert cache.check_device_error() == 0
    _check(cache, 0, q.cpu().numpy(), out.float().cpu().numpy(), 2, 2, floor=1, label="floor 1")


def test_fused_prefill_equals_append_then_attention():
    """kvarn_prefill = kvarn_append + kvarn_prefill_attention, bit for bit, chunk by
    chunk; the last chunk's rows also match the oracle."""
    a, b = _cache(8, 2, 2, 2), _cache(8, 2, 2, 2)
    chunks = [200, 333, 1]
    start = 0
    for i, c in enumerate(chunks):
        k, v = _tokens(70, 0, start, c, 2)
        q = _queries(71 + i, c, 8)
        oa = a.prefill(0, [0], [c], k, v, q)
        b.append(0, [0], [c], k, v)
        ob = b.prefill_attention(0, [0], [c], q)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob), f"chunk {i}"
        start += c
    assert a.check_device_error() == 0
    _check(a, 0, q.cpu().numpy(), oa.float().cpu().numpy(), 2, 2, label="fused")


def test_last_token_prefill_matches_decode_attention():
    """The query of the newest token sees the whole cache, as decode attention does (the
    two kernels share no code; both are within the parity tolerance of the oracle)."""
    cache = _cache(8, 2, 2, 2)
    lengths = [1000, 300]
    for s, n in enumerate(lengths):
        k, v = _tokens(80, s, 0, n, 2)
        cache.append(0, [s], [n], k, v)
    q = _queries(81, 2, 8)
    pf = cache.prefill_attention(0, [0, 1], [1, 1], q)
    dc = cache.decode_attention(0, [0, 1], q)
    torch.cuda.synchronize()
    d = (pf.float() - dc.float()).abs().amax(dim=-1)
    nrm = dc.float().norm(dim=-1)
    assert bool((d <= 4e-3 * nrm + 1e-6).all())


def test_empty_calls():
    cache = _cache(8, 2, 2, 2)
    k, v = _tokens(90, 0, 0, 10, 2)
    cache.append(0, [0], [10], k, v)
    q = torch.empty((0, 8, 128), dtype=torch.float16, device="cuda")
    cache.prefill_attention(0, [0], [0], q)
    cache.prefill_attention(0, [], [], q)
    torch.cuda.synchronize()
    assert cache.check_device_error() == 0


def test_qwen3_4b_prefill_4096_sampled_rows():
    """The measured workload (Qwen3-4B attention shape: 32 query heads, 8 KV heads; a
    4096-token prompt appended in one call, 31 groups sealed, then every token's query),
    checked on sampled rows in each region."""
    cache = _cache(32, 8, 2, 2, seqs=1, max_len=4096)
    n = 4096
    k, v = _tokens(1, 0, 0, n, 8)
    q = _queries(2, n, 32)
    out = cache.prefill(0, [0], [n], k, v, q)
    torch.cuda.synchronize()
    assert cache.check_device_error() == 0
    assert bool(torch.isfinite(out.float()).all())
    rows = [0, 1, 127, 128, 200, 255, 1000, 2047, 3000, 3967, 3968, 4095]
    _check(cache, 0, q.cpu().numpy(), out.float().cpu().numpy(), 2, 2, rows=rows, label="qwen3-4b 4096")


def test_phi4_shape_second_layer_interleaved_slots_spikes():
    """Phi-4 attention shape (40 query heads, 10 KV heads), a cache of two layers whose
    sequences were appended in interleaved rounds (the pool slots of a sequence are not
    contiguous), 5 % of tokens with x10 K/V norms; prefill attention on layer 1."""
    from quantized_kv_cache_seal_gb300.cache import KVarNCache
    cache = KVarNCache(num_layers=2, max_seqs=3, num_q_heads=40, num_kv_heads=10, k_bits=4, v_bits=2,
                       max_seq_len=2048)
    lengths = [900, 1400, 700]
    done = [0, 0, 0]
    while any(d < n for d, n in zip(done, lengths)):
        for layer in (0, 1):
            ids, counts, ks, vs = [], [], [], []
            for s, n in enumerate(lengths):
                take = min(300, n - done[s])
                if take <= 0:
                    continue
                k, v = workloads.torch_tokens(100 + layer, s, done[s], take, 10, spike_frac=0.05, spike_factor=10.0)
                ids.append(s)
                counts.append(take)
                ks.append(k)
                vs.append(v)
            cache.append(layer, ids, counts, torch.cat(ks).contiguous(), torch.cat(vs).contiguous())
        done = [min(n, d + 300) for d, n in zip(done, lengths)]
    from quantized_kv_cache_seal_gb300 import kvarn as K
    # group 0 of sequence 1 was sealed in the first round, group 1 in the second
    p0, _ = K.kvarn_group_record(cache.handle, 1, 1, 0, 0, 0)
    p1, _ = K.kvarn_group_record(cache.handle, 1, 1, 1, 0, 0)
    assert p1 - p0 != K.kvarn_cache_stats(cache.handle).slot_bytes  # not adjacent in the pool
    # one call over the sequences in the order 2, 0, 1; rows follow the call's order
    q_lens = [200, 130, 64]
    q = _queries(101, sum(q_lens), 40)
    out = cache.prefill_attention(1, [2, 0, 1], q_lens, q)
    torch.cuda.synchronize()
    assert cache.check_device_error() == 0
    qn, on = q.cpu().numpy(), out.float().cpu().numpy()
    _check(cache, 2, qn[:200], on[:200], 4, 2, label="phi4 l1", layer=1, heads=[0, 9])
    _check(cache, 0, qn[200:330], on[200:330], 4, 2, label="phi4 l1", layer=1, heads=[3])
    _check(cache, 1, qn[330:], on[330:], 4, 2, label="phi4 l1", layer=1, heads=[5, 7])
