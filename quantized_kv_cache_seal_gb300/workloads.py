"""Seeded synthetic inputs for the KVarN cache: K/V token streams, queries, lengths.

This module holds no KVarN arithmetic (no rotation, normalisation, rounding or
packing). It only draws numbers, so that the CUDA path and the CPU oracle are
fed the very same fp16 bits. The value recipe stands in for the post-RoPE K/V
of the models the KVarN pages evaluate (Qwen3-4B, Llama-3.1-8B, Phi-4-14B; the
fig1.dev summary, "Key result"), which are not available here:

* per (layer, KV head, side) a channel scale s_j ~ lognormal(0, 0.5), fixed over
  tokens, with two distinct outlier channels multiplied by 20;
* per token a norm factor n_t ~ lognormal(0, 0.7), shared by K and V and by all
  KV heads of that token;
* x_tj = N(0, 1) * s_j * n_t, cast to fp16 with round-to-nearest-even;
* optionally a fraction of (sequence, token) positions whose K and V are
  multiplied by a spike factor (token-norm imbalance stress);
* queries N(0, 1) in fp16.

Everything is generated with ``numpy.random.default_rng(seed)`` so that runs are
reproducible on any host.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

HEAD_DIM = 128
GROUP = 128
SINK = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode workload: head layout, batch, context lengths and bit widths."""

    name: str
    num_q_heads: int
    num_kv_heads: int
    batch: int
    k_bits: int
    v_bits: int
    seed: int
    # context lengths at the start of the decode loop (one per sequence)
    context: tuple
    decode_steps: int
    spike_frac: float = 0.0
    spike_factor: float = 10.0
    head_dim: int = HEAD_DIM
    paged_random: bool = False

    @property
    def gqa(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def _lengths_c3(seed: int, batch: int) -> tuple:
    rng = np.random.default_rng(seed)
    tails = rng.integers(0, GROUP, size=batch)  # U{0..127}
    return tuple(int(32768 + t) for t in tails)


def _lengths_c5(seed: int, batch: int) -> tuple:
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(1024, 16385, size=batch))


def workloads() -> dict:
    """The five workloads: parity case, three model-shaped decode loops, ragged batch."""
    w = {}
    # single KV head, 128 sink + one sealed group + 37 tail tokens = 293 tokens
    w["c1_single_head_293"] = Workload("c1_single_head_293", 1, 1, 1, 2, 2, 0, (293,), 0)
    # Qwen3-4B heads, 4096 context, 256 decode steps
    w["c2_qwen3_4b_4k"] = Workload("c2_qwen3_4b_4k", 32, 8, 1, 2, 2, 1, (4096,), 256)
    # Llama-3.1-8B heads, batch 16, 32k context with ragged tails
    w["c3_llama31_8b_32k"] = Workload("c3_llama31_8b_32k", 32, 8, 16, 2, 2, 2,
                                      _lengths_c3(2, 16), 256)
    # long reasoning, 64k context, K 4-bit / V 2-bit and 4/4
    w["c4_long_64k_k4v2"] = Workload("c4_long_64k_k4v2", 32, 8, 8, 4, 2, 3, (65536,) * 8, 2048)
    w["c4_long_64k_k4v4"] = Workload("c4_long_64k_k4v4", 32, 8, 8, 4, 4, 3, (65536,) * 8, 2048)
    # Phi-4-14B heads, batch 64, ragged 1k..16k, 5% x10 token-norm spikes
    for b in (2, 4, 8):
        w[f"c5_phi4_14b_ragged_b{b}"] = Workload(
            f"c5_phi4_14b_ragged_b{b}", 40, 10, 64, b, b, 4, _lengths_c5(4, 64), 64,
            spike_frac=0.05, paged_random=True)
    return w


class TokenSource:
    """Deterministic K/V stream for one (layer, sequence): token t's K/V do not depend
    on how many tokens are drawn at once, so bulk and streaming appends see the same bits.

    Tokens are produced in blocks of ``block`` tokens from a per-block seeded generator.
    """

    def __init__(self, seed: int, seq: int, num_kv_heads: int, head_dim: int = HEAD_DIM,
                 spike_frac: float = 0.0, spike_factor: float = 10.0, block: int = 1024):
        self.seed = seed
        self.seq = seq
        self.hkv = num_kv_heads
        self.d = head_dim
        self.spike_frac = spike_frac
        self.spike_factor = spike_factor
        self.block = block
        # per (kv head, side) channel scales with two outlier channels
        rng = np.random.default_rng([seed, 7919, seq])
        s = rng.lognormal(0.0, 0.5, size=(2, num_kv_heads, head_dim))
        for side in range(2):
            for h in range(num_kv_heads):
                out = rng.choice(head_dim, size=2, replace=False)
                s[side, h, out] *= 20.0
        self.chan_scale = s
        self._cache = {}

    def _block(self, b: int):
        if b in self._cache:
            return self._cache[b]
        rng = np.random.default_rng([self.seed, 104729, self.seq, b])
        n = self.block
        norms = rng.lognormal(0.0, 0.7, size=(n,))
        if self.spike_frac > 0:
            spikes = rng.random(n) < self.spike_frac
            norms = np.where(spikes, norms * self.spike_factor, norms)
        g = rng.standard_normal(size=(2, n, self.hkv, self.d))
        x = g * self.chan_scale[:, None, :, :] * norms[None, :, None, None]
        x = np.clip(x, -65504.0, 65504.0).astype(np.float16)
        if len(self._cache) > 8:
            self._cache.clear()
        self._cache[b] = x
        return x

    def tokens(self, start: int, count: int):
        """Return (K, V) fp16 arrays of shape [count][Hkv][d] for positions start..start+count."""
        k = np.empty((count, self.hkv, self.d), np.float16)
        v = np.empty((count, self.hkv, self.d), np.float16)
        pos = start
        out = 0
        while out < count:
            b, off = divmod(pos, self.block)
            take = min(self.block - off, count - out)
            blk = self._block(b)
            k[out:out + take] = blk[0, off:off + take]
            v[out:out + take] = blk[1, off:off + take]
            out += take
            pos += take
        return k, v


def queries(seed: int, step: int, batch: int, num_q_heads: int, head_dim: int = HEAD_DIM):
    """N(0,1) fp16 queries [batch][Hq][d] for one decode step."""
    rng = np.random.default_rng([seed, 15485863, step])
    return rng.standard_normal(size=(batch, num_q_heads, head_dim)).astype(np.float16)


def group_matrices(seed: int, count: int, head_dim: int = HEAD_DIM, group: int = GROUP,
                   spike_frac: float = 0.0):
    """``count`` independent fp16 [group][head_dim] matrices with the K/V value recipe."""
    rng = np.random.default_rng([seed, 2038074743])
    s = rng.lognormal(0.0, 0.5, size=(count, 1, head_dim))
    for i in range(count):
        out = rng.choice(head_dim, size=2, replace=False)
        s[i, 0, out] *= 20.0
    n = rng.lognormal(0.0, 0.7, size=(count, group, 1))
    if spike_frac > 0:
        n = np.where(rng.random((count, group, 1)) < spike_frac, n * 10.0, n)
    x = rng.standard_normal(size=(count, group, head_dim)) * s * n
    return np.clip(x, -65504.0, 65504.0).astype(np.float16)


def random_slot_permutation(seed: int, n: int) -> np.ndarray:
    """A random order in which pool slots are handed out (non-contiguous pages)."""
    return np.random.default_rng([seed, 32452843]).permutation(n).astype(np.int32)


def tiny_matrix(seed: int, rows: int, cols: int, scale: Optional[float] = 1.0):
    """Small fp16 matrix for brute-force checks."""
    rng = np.random.default_rng([seed, 49979687])
    return (rng.standard_normal(size=(rows, cols)) * scale).astype(np.float16)


def torch_tokens(seed: int, seq: int, start: int, count: int, num_kv_heads: int, head_dim: int = HEAD_DIM,
                 spike_frac: float = 0.0, spike_factor: float = 10.0, device="cuda"):
    """Same value recipe as TokenSource, drawn on the device with torch (for the
    multi-gigabyte prefills of the full-size workloads). Token t of sequence ``seq``
    depends only on (seed, seq, t // 4096), so chunked generation is reproducible.
    Returns fp16 (K, V), each [count][Hkv][d]."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + int(seq) * 7919 + 17)
    s = torch.empty((2, num_kv_heads, head_dim), device=device).log_normal_(0.0, 0.5, generator=g)
    for side in range(2):
        for h in range(num_kv_heads):
            out = torch.randperm(head_dim, generator=g, device=device)[:2]
            s[side, h, out] *= 20.0
    blk = 4096
    ks, vs = [], []
    pos = start
    end = start + count
    while pos < end:
        b = pos // blk
        gb = torch.Generator(device=device)
        gb.manual_seed(int(seed) * 1000003 + int(seq) * 7919 + 104729 * (b + 1))
        norms = torch.empty((blk,), device=device).log_normal_(0.0, 0.7, generator=gb)
        if spike_frac > 0:
            spikes = torch.rand((blk,), device=device, generator=gb) < spike_frac
            norms = torch.where(spikes, norms * spike_factor, norms)
        lo = pos - b * blk
        hi = min(blk, end - b * blk)
        x = torch.randn((2, blk, num_kv_heads, head_dim), device=device, generator=gb)[:, lo:hi]
        x = x * s[:, None] * norms[None, lo:hi, None, None]
        x = x.clamp_(-65504.0, 65504.0).to(torch.float16)
        ks.append(x[0])
        vs.append(x[1])
        pos = b * blk + hi
    return torch.cat(ks).contiguous(), torch.cat(vs).contiguous()


def torch_queries(seed: int, steps: int, batch: int, num_q_heads: int, head_dim: int = HEAD_DIM, device="cuda"):
    """N(0,1) fp16 queries [steps][batch][Hq][d] drawn on the device."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 15485863 + 3)
    return torch.randn((steps, batch, num_q_heads, head_dim), device=device, generator=g).to(torch.float16)
