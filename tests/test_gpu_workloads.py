"""GPU parity on the model-shaped workloads, at their full sizes, checked on samples.

The workloads (quantized_kv_cache_seal_gb300.workloads) stand in for the decode loops
the KVarN pages evaluate (fig1.dev "Key result": Qwen3-4B, Llama-3.1-8B, Phi-4-14B;
anbeeld.com "KVarN KV Cache: Implementation and Benchmarks", sections 1 and 2.1 for the
sink / sealed body / tail regions). Each case builds the cache through the C ABI
(bulk append, then decode steps that append, seal and attend in one launch) and checks:

* attention: for sampled (sequence, KV head) blocks, the GPU output against the
  oracle's fp64 attention over the GPU's own records and exact regions
  (tests/parity.py: max |err| <= 2e-3 ||o||_2 per head);
* seals done inside a decode step: the record against the oracle's seal of the same
  fp16 tokens, with the decoupled protocol of tests/parity.py (the pseudo-decode check:
  streaming one token at a time seals what a bulk seal of those tokens would).

Inputs are drawn on the device (workloads.torch_tokens / torch_queries); the tokens a
check needs are copied back, so GPU and oracle see the same fp16 bits.
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
WL = workloads.workloads()


def _cache(w, max_len, layers=1):
    from quantized_kv_cache_seal_gb300.cache import KVarNCache
    return KVarNCache(num_layers=layers, max_seqs=w.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                      k_bits=w.k_bits, v_bits=w.v_bits, max_seq_len=max_len)


def _records(cache, layer, seq, kvh, which, n_groups):
    """All records of one (sequence, KV head, side) as a host array [n_groups][bytes]."""
    if n_groups == 0:
        return np.zeros(0, np.uint8)
    base = cache.mem.data_ptr()
    offs = []
    n = 0
    for g in range(n_groups):
        ptr, n = K.kvarn_group_record(cache.handle, layer, seq, g, kvh, which)
        offs.append(ptr - base)
    idx = torch.tensor(offs, device=cache.mem.device, dtype=torch.int64)[:, None] + \
        torch.arange(n, device=cache.mem.device, dtype=torch.int64)[None, :]
    return cache.mem[idx].cpu().numpy()


def _oracle_block(cache, layer, seq, kvh, q_heads):
    """fp64 attention of the r query heads q_heads [r][d] of KV head kvh over the GPU's state."""
    cfg = cache.cfg
    n = cache.length(layer, seq)
    n_sink = min(n, 128)
    n_groups = max(n - 128, 0) // 128
    n_tail = max(n - 128, 0) % 128
    sk, sv, tk, tv = [t[kvh].cpu().numpy() for t in cache.exact_regions(layer, seq)]
    kr = _records(cache, layer, seq, kvh, 0, n_groups)
    vr = _records(cache, layer, seq, kvh, 1, n_groups)
    return oracle.attention(q_heads, SCALE, sk[:n_sink], sv[:n_sink], kr, vr, tk[:n_tail], tv[:n_tail],
                            cfg.k_bits, cfg.v_bits)


def _check_blocks(cache, layer, out, q, samples, label):
    r = cache.cfg.num_q_heads // cache.cfg.num_kv_heads
    out = out.float().cpu().numpy()
    q = q.cpu().numpy()
    worst = 0.0
    for seq, kvh in samples:
        ref = _oracle_block(cache, layer, seq, kvh, q[seq, kvh * r:(kvh + 1) * r])
        worst = max(worst, parity.check_attention(out[seq, kvh * r:(kvh + 1) * r], ref,
                                                  f"{label} seq {seq} kvh {kvh}"))
    return worst


def _prefill(cache, w, lengths, chunk=8192, rounds=None):
    """Bulk-append the prefixes, in rounds over the sequences (so that the pool slots of
    different sequences interleave)."""
    done = [0] * w.batch
    while any(d < n for d, n in zip(done, lengths)):
        ids, counts, ks, vs = [], [], [], []
        for s in range(w.batch):
            take = min(chunk, lengths[s] - done[s])
            if take <= 0:
                continue
            k, v = workloads.torch_tokens(w.seed, s, done[s], take, w.num_kv_heads, spike_frac=w.spike_frac,
                                          spike_factor=w.spike_factor)
            ids.append(s)
            counts.append(take)
            ks.append(k)
            vs.append(v)
            done[s] += take
        cache.append(0, ids, counts, torch.cat(ks).contiguous(), torch.cat(vs).contiguous())
    torch.cuda.synchronize()


def _step_tokens(w, lengths, step):
    """The decode step's new token of every sequence, fp16 [B][Hkv][d] each."""
    ks, vs = [], []
    for s in range(w.batch):
        k, v = workloads.torch_tokens(w.seed, s, lengths[s] + step, 1, w.num_kv_heads, spike_frac=w.spike_frac,
                                      spike_factor=w.spike_factor)
        ks.append(k)
        vs.append(v)
    return torch.cat(ks).contiguous(), torch.cat(vs).contiguous()


def _check_new_seal(cache, w, seq, kvh, g, label):
    """Record of body group g (sealed during the decode loop) against the oracle's seal."""
    start = 128 + 128 * g
    k, v = workloads.torch_tokens(w.seed, seq, start, 128, w.num_kv_heads, spike_frac=w.spike_frac,
                                  spike_factor=w.spike_factor)
    for which, x in ((0, k), (1, v)):
        rec = cache.record(0, seq, g, kvh, which).cpu().numpy()
        parity.check_seal(x[:, kvh].cpu().numpy(), rec, w.k_bits if which == 0 else w.v_bits, which,
                          label=f"{label} seq {seq} g {g} kvh {kvh} side {which}")


def test_c2_qwen3_4b_decode_seals_at_step_128():
    """C2: one 4096-token sequence, then decode steps; the step whose token completes a
    group seals it and attends to the new record."""
    w = WL["c2_qwen3_4b_4k"]
    lengths = list(w.context)
    cache = _cache(w, lengths[0] + 512)
    _prefill(cache, w, lengths)
    qs = workloads.torch_queries(w.seed, 130, w.batch, w.num_q_heads)
    samples = [(0, h) for h in range(w.num_kv_heads)]
    for step in range(130):
        k, v = _step_tokens(w, lengths, step)
        out = cache.decode_step(0, [0], k, v, qs[step])
        if step in (0, 126, 127, 128, 129):
            assert cache.check_device_error() == 0
            _check_blocks(cache, 0, out, qs[step], samples, f"c2 step {step}")
    assert cache.length(0, 0) == 4096 + 130
    # 4096 = 128 sink + 31 groups, no tail: the token of step 127 completed group 31
    for h in range(w.num_kv_heads):
        _check_new_seal(cache, w, 0, h, 31, "c2")


def test_c3_llama31_8b_headline_shape_sampled():
    """C3 (the benchmark's workload): batch 16 at 32k with ragged tails, two decode steps,
    outputs checked on sampled blocks, including the sequence with the longest tail."""
    w = WL["c3_llama31_8b_32k"]
    lengths = list(w.context)
    cache = _cache(w, max(lengths) + 256)
    _prefill(cache, w, lengths)
    qs = workloads.torch_queries(w.seed, 2, w.batch, w.num_q_heads)
    longest = int(np.argmax([n % 128 for n in lengths]))
    samples = [(0, 0), (5, 3), (longest, 7), (15, 5)]
    for step in range(2):
        k, v = _step_tokens(w, lengths, step)
        out = cache.decode_step(0, list(range(w.batch)), k, v, qs[step])
        assert cache.check_device_error() == 0
        _check_blocks(cache, 0, out, qs[step], samples, f"c3 step {step}")


@pytest.mark.parametrize("name", ["c4_long_64k_k4v2", "c4_long_64k_k4v4"])
def test_c4_long_context_fused_seals(name):
    """C4: 8 sequences at 64k in phase, K 4-bit; 128 decode steps, so that every sequence
    seals group 511 of every KV head inside the same step (64 seals in one launch)."""
    w = WL[name]
    lengths = list(w.context)
    cache = _cache(w, lengths[0] + 256)
    _prefill(cache, w, lengths)
    qs = workloads.torch_queries(w.seed, 128, w.batch, w.num_q_heads)
    for step in range(128):
        k, v = _step_tokens(w, lengths, step)
        out = cache.decode_step(0, list(range(w.batch)), k, v, qs[step])
        if step in (0, 127):
            assert cache.check_device_error() == 0
            _check_blocks(cache, 0, out, qs[step], [(0, 0), (3, 5), (7, 7)], f"{name} step {step}")
    # 65536 = 128 + 511 * 128 + 0: the token of step 127 completed group 511
    for seq, kvh in ((0, 0), (4, 2), (7, 7)):
        _check_new_seal(cache, w, seq, kvh, 511, name)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_c5_phi4_ragged_paged_spikes(bits):
    """C5: 40/10 heads, batch 64, lengths 1k..16k, 5 % of tokens with x10 K/V norms, pool
    slots of different sequences interleaved; one decode step and one attention call."""
    w = WL[f"c5_phi4_14b_ragged_b{bits}"]
    lengths = list(w.context)
    cache = _cache(w, max(lengths) + 256)
    _prefill(cache, w, lengths, chunk=1024)
    # the pages of a sequence are not contiguous in the pool: group 6 ends the first
    # 1024-token round, group 7 comes after the other sequences' first rounds
    big = int(np.argmax(lengths))
    p0, _ = K.kvarn_group_record(cache.handle, 0, big, 6, 0, 0)
    p1, _ = K.kvarn_group_record(cache.handle, 0, big, 7, 0, 0)
    slot = K.kvarn_cache_stats(cache.handle).slot_bytes
    assert p1 - p0 != slot
    qs = workloads.torch_queries(w.seed, 2, w.batch, w.num_q_heads)
    rng = np.random.default_rng(bits)
    samples = [(int(s), int(h)) for s, h in zip(rng.integers(0, w.batch, 6), rng.integers(0, w.num_kv_heads, 6))]
    samples.append((int(np.argmin(lengths)), 9))
    samples.append((int(np.argmax(lengths)), 0))
    k, v = _step_tokens(w, lengths, 0)
    out = cache.decode_step(0, list(range(w.batch)), k, v, qs[0])
    assert cache.check_device_error() == 0
    _check_blocks(cache, 0, out, qs[0], samples, f"c5 b{bits} step")
    out = cache.decode_attention(0, list(range(w.batch)), qs[1])
    assert cache.check_device_error() == 0
    _check_blocks(cache, 0, out, qs[1], samples, f"c5 b{bits} attend")
