"""GPU parity on the model-shaped workloads, at their full sizes and decode lengths.

The workloads (quantized_kv_cache_seal_gb300.workloads) stand in for the decode loops
the KVarN pages evaluate (fig1.dev "Key result": Qwen3-4B, Llama-3.1-8B, Phi-4-14B;
"Practical takeaway": the pseudo-decode check, which re-quantises the cache block by
block as decoding proceeds and makes later tokens read the sealed blocks;
anbeeld.com "KVarN KV Cache: Implementation and Benchmarks", sections 1 and 2.1 for the
sink / sealed body / tail regions). Each case builds the cache through the C ABI
(bulk append, then decode steps that append, seal and attend in one launch) and checks:

* attention: for (sequence, KV head) blocks, the GPU output against the oracle's fp64
  attention over the GPU's own records and exact regions (tests/parity.py:
  max |err| <= 2e-3 ||o||_2 per head);
* every seal done inside the decode loop: the record against the oracle's seal of the
  same fp16 tokens, with the decoupled protocol of tests/parity.py (streaming one token
  at a time seals what a bulk seal of those tokens would).

Inputs are drawn on the device (workloads.torch_tokens / torch_queries); the tokens a
check needs are copied back, so GPU and oracle see the same fp16 bits. The oracle runs
in host threads (its C entry points release the interpreter lock).
"""
import concurrent.futures
import math
import os

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
POOL = concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))
CHECKED = {"blocks": 0}  # attention checks done (each test asserts its own count)


def _all(fn, jobs):
    """Run fn(*job) for every job on the host threads; return the results in order."""
    return list(POOL.map(lambda j: fn(*j), jobs))


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


def _block_state(cache, layer, seq, kvh):
    """The GPU's state of one (sequence, KV head) block as host arrays."""
    n = cache.length(layer, seq)
    n_sink = min(n, 128)
    n_groups = max(n - 128, 0) // 128
    n_tail = max(n - 128, 0) % 128
    sk, sv, tk, tv = [t[kvh].cpu().numpy() for t in cache.exact_regions(layer, seq)]
    kr = _records(cache, layer, seq, kvh, 0, n_groups)
    vr = _records(cache, layer, seq, kvh, 1, n_groups)
    return sk[:n_sink], sv[:n_sink], kr, vr, tk[:n_tail], tv[:n_tail]


def _check_blocks(cache, layer, out, q, samples, label):
    """Attention of the given (sequence, KV head) blocks against the oracle's."""
    cfg = cache.cfg
    r = cfg.num_q_heads // cfg.num_kv_heads
    out = out.float().cpu().numpy()
    q = q.cpu().numpy()
    jobs = []
    for seq, kvh in samples:
        st = _block_state(cache, layer, seq, kvh)
        jobs.append((seq, kvh, st))

    def one(seq, kvh, st):
        ref = oracle.attention(q[seq, kvh * r:(kvh + 1) * r], SCALE, *st, cfg.k_bits, cfg.v_bits)
        return parity.check_attention(out[seq, kvh * r:(kvh + 1) * r], ref, f"{label} seq {seq} kvh {kvh}")

    CHECKED["blocks"] += len(jobs)
    return max(_all(one, jobs)) if jobs else 0.0


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


def _decode_tokens(w, lengths, steps):
    """The new tokens of decode steps 0 .. steps - 1, fp16 [steps][B][Hkv][d] each (token
    t of a sequence depends only on its position, so drawing them at once gives the same
    bits as drawing them step by step)."""
    ks, vs = [], []
    for s in range(w.batch):
        k, v = workloads.torch_tokens(w.seed, s, lengths[s], steps, w.num_kv_heads, spike_frac=w.spike_frac,
                                      spike_factor=w.spike_factor)
        ks.append(k)
        vs.append(v)
    return torch.stack(ks, 1).contiguous(), torch.stack(vs, 1).contiguous()


def _check_seals(cache, w, groups, label):
    """Records of body groups sealed during the decode loop, (sequence, group) pairs,
    every KV head and both sides, against the oracle's seal of the same fp16 tokens."""
    jobs = []
    for seq, g in groups:
        k, v = workloads.torch_tokens(w.seed, seq, 128 + 128 * g, 128, w.num_kv_heads, spike_frac=w.spike_frac,
                                      spike_factor=w.spike_factor)
        k, v = k.cpu().numpy(), v.cpu().numpy()
        for kvh in range(w.num_kv_heads):
            for which, x in ((0, k), (1, v)):
                rec = cache.record(0, seq, g, kvh, which).cpu().numpy()
                jobs.append((x[:, kvh].copy(), rec, w.k_bits if which == 0 else w.v_bits, which,
                             f"{label} seq {seq} g {g} kvh {kvh} side {which}"))
    _all(lambda x, rec, bits, which, lab: parity.check_seal(x, rec, bits, which, label=lab), jobs)
    return len(jobs)


def _sealing(lengths, step):
    """Sequences whose token of decode step `step` completes a group (no tail floor)."""
    return [s for s, n in enumerate(lengths) if n + step >= 128 and (n + step - 128) % 128 == 127]


def test_c2_qwen3_4b_all_256_steps_two_seals():
    """C2: one 4096-token sequence, then all 256 decode steps of the workload; the tokens
    of steps 127 and 255 complete groups 31 and 32, which are sealed in those steps and
    attended to at once. Attention of every KV head is checked around both seals and at
    other steps; both seals are checked on every KV head and side."""
    w = WL["c2_qwen3_4b_4k"]
    lengths = list(w.context)
    steps = w.decode_steps
    assert steps == 256
    cache = _cache(w, lengths[0] + steps)
    _prefill(cache, w, lengths)
    qs = workloads.torch_queries(w.seed, steps, w.batch, w.num_q_heads)
    kn, vn = _decode_tokens(w, lengths, steps)
    samples = [(0, h) for h in range(w.num_kv_heads)]
    checked = {0, 1, 63, 126, 127, 128, 200, 254, 255}
    for step in range(steps):
        out = cache.decode_step(0, [0], kn[step], vn[step], qs[step])
        if step in checked:
            assert cache.check_device_error() == 0
            _check_blocks(cache, 0, out, qs[step], samples, f"c2 step {step}")
    assert cache.length(0, 0) == 4096 + 256
    assert [st for st in range(steps) if _sealing(lengths, st)] == [127, 255]
    assert _check_seals(cache, w, [(0, 31), (0, 32)], "c2") == 2 * 2 * w.num_kv_heads


def test_c3_llama31_8b_every_block_at_a_sealing_step():
    """C3 (the benchmark's workload): batch 16 at 32k with ragged tails. 128 decode steps,
    in which every sequence seals once, at a step of its own. All 128 (sequence, KV head)
    blocks are checked at the first step that contains a fused seal and at the last
    step (which contains one too); sampled blocks at every other sealing step; every seal
    of the run on every KV head and side."""
    w = WL["c3_llama31_8b_32k"]
    lengths = list(w.context)
    steps = 128
    before = CHECKED["blocks"]
    cache = _cache(w, max(lengths) + steps)
    _prefill(cache, w, lengths)
    qs = workloads.torch_queries(w.seed, steps, w.batch, w.num_q_heads)
    kn, vn = _decode_tokens(w, lengths, steps)
    seal_steps = {st: _sealing(lengths, st) for st in range(steps) if _sealing(lengths, st)}
    assert sorted(s for v in seal_steps.values() for s in v) == list(range(w.batch))  # each seals once
    first, last = min(seal_steps), max(seal_steps)
    every = [(s, h) for s in range(w.batch) for h in range(w.num_kv_heads)]
    rng = np.random.default_rng(3)
    ids = list(range(w.batch))
    for step in range(steps):
        out = cache.decode_step(0, ids, kn[step], vn[step], qs[step])
        if step in (first, last) or step in seal_steps or step == 0:
            assert cache.check_device_error() == 0
            if step in (first, last):
                samples = every
            else:
                samples = [(s, int(rng.integers(0, w.num_kv_heads))) for s in seal_steps.get(step, [])]
                samples += [(int(rng.integers(0, w.batch)), int(rng.integers(0, w.num_kv_heads)))]
            _check_blocks(cache, 0, out, qs[step], samples, f"c3 step {step}")
    assert CHECKED["blocks"] - before >= 2 * len(every)
    groups = [(s, (lengths[s] + st - 128) // 128) for st, seqs in seal_steps.items() for s in seqs]
    assert _check_seals(cache, w, groups, "c3") == w.batch * w.num_kv_heads * 2


@pytest.mark.parametrize("name", ["c4_long_64k_k4v2", "c4_long_64k_k4v4"])
def test_c4_long_reasoning_2048_steps_every_seal(name):
    """C4: 8 sequences at 64k in phase, K 4-bit; all 2048 decode steps of the workload,
    which seal 16 groups per sequence (steps 127, 255, ..., 2047: all 8 sequences and 8 KV
    heads seal in the same launch). The pseudo-decode check: every one of those 1024
    (sequence, group) seals is checked on every KV head and side against the oracle's
    seal of the same tokens; attention is checked on sampled blocks at steps around the
    first and the last seal and in between."""
    w = WL[name]
    lengths = list(w.context)
    steps = w.decode_steps
    assert steps == 2048
    cache = _cache(w, lengths[0] + steps)
    _prefill(cache, w, lengths)
    qs = workloads.torch_queries(w.seed, steps, w.batch, w.num_q_heads)
    kn, vn = _decode_tokens(w, lengths, steps)
    ids = list(range(w.batch))
    checked = {0: [(0, 0), (3, 5), (7, 7)], 127: [(1, 1), (6, 4)], 128: [(2, 3), (5, 6)],
               1023: [(4, 2)], 1024: [(0, 7)], 2047: [(0, 0), (3, 5), (7, 7)]}
    for step in range(steps):
        out = cache.decode_step(0, ids, kn[step], vn[step], qs[step])
        if step in checked:
            assert cache.check_device_error() == 0
            _check_blocks(cache, 0, out, qs[step], checked[step], f"{name} step {step}")
    seal_steps = [st for st in range(steps) if _sealing(lengths, st)]
    assert seal_steps == list(range(127, steps, 128)) and len(seal_steps) == 16
    groups = [(s, 511 + i) for i in range(16) for s in range(w.batch)]
    assert _check_seals(cache, w, groups, name) == 16 * w.batch * w.num_kv_heads * 2


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_c5_phi4_ragged_paged_spikes(bits):
    """C5: 40/10 heads, batch 64, lengths 1k..16k, 5 % of tokens with x10 K/V norms, pool
    slots of different sequences interleaved; four decode steps (sampled blocks checked at
    each, with the sequences that seal in them) and one attention call; the seals made in
    those steps checked on every KV head and side."""
    w = WL[f"c5_phi4_14b_ragged_b{bits}"]
    lengths = list(w.context)
    steps = 4
    cache = _cache(w, max(lengths) + 256)
    _prefill(cache, w, lengths, chunk=1024)
    # the pages of a sequence are not contiguous in the pool: group 6 ends the first
    # 1024-token round, group 7 comes after the other sequences' first rounds
    big = int(np.argmax(lengths))
    p0, _ = K.kvarn_group_record(cache.handle, 0, big, 6, 0, 0)
    p1, _ = K.kvarn_group_record(cache.handle, 0, big, 7, 0, 0)
    slot = K.kvarn_cache_stats(cache.handle).slot_bytes
    assert p1 - p0 != slot
    qs = workloads.torch_queries(w.seed, steps + 1, w.batch, w.num_q_heads)
    kn, vn = _decode_tokens(w, lengths, steps)
    rng = np.random.default_rng(bits)
    ids = list(range(w.batch))
    groups = []
    for step in range(steps):
        out = cache.decode_step(0, ids, kn[step], vn[step], qs[step])
        assert cache.check_device_error() == 0
        samples = [(int(s), int(h)) for s, h in zip(rng.integers(0, w.batch, 5), rng.integers(0, w.num_kv_heads, 5))]
        samples.append((int(np.argmin(lengths)), 9))
        samples.append((int(np.argmax(lengths)), 0))
        sealing = _sealing(lengths, step)
        samples += [(s, int(rng.integers(0, w.num_kv_heads))) for s in sealing]
        groups += [(s, (lengths[s] + step - 128) // 128) for s in sealing]
        _check_blocks(cache, 0, out, qs[step], samples, f"c5 b{bits} step {step}")
    out = cache.decode_attention(0, ids, qs[steps])
    assert cache.check_device_error() == 0
    _check_blocks(cache, 0, out, qs[steps], samples, f"c5 b{bits} attend")
    if groups:
        _check_seals(cache, w, groups, f"c5 b{bits}")
