"""ctypes binding and cache-region model for the KVarN CPU oracle (test infrastructure).

Sources (page title, section):
  * anbeeld.com "KVarN KV Cache: Implementation and Benchmarks", 2.1 "Sink, Body,
    And Tail": the first 128 tokens stay exact, later tokens form groups of 128
    that are quantised when the group's last token arrives, and the newest
    partial group (the tail) stays exact.
  * same page, section 1, and fig1.dev "KVarN ...", "What it is": rotation,
    16 Sinkhorn iterations, round-to-nearest; attention in the rotated frame.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvarn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkvarn_oracle.so")
_lock = threading.Lock()
_lib = None

GROUP = 128
SINK = 128
HEAD_DIM = 128
ITERS = 16

__all__ = [
    "build", "lib", "half_to_double", "double_to_half", "hadamard", "rotate", "sinkhorn",
    "record_bytes", "header_bytes", "pack", "unpack", "seal", "codes_for_grid", "read_header", "quantize",
    "dequant", "attention", "prefill_attention", "OracleCache", "bits_per_element", "GROUP", "SINK", "ITERS",
]


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (plain -O2, no CUDA)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            L.kvo_half_to_double.argtypes = [ctypes.c_uint16]
            L.kvo_half_to_double.restype = D
            L.kvo_double_to_half.argtypes = [D]
            L.kvo_double_to_half.restype = ctypes.c_uint16
            L.kvo_double_to_half_sat.argtypes = [D]
            L.kvo_double_to_half_sat.restype = ctypes.c_uint16
            L.kvo_hadamard.argtypes = [I, P]
            L.kvo_rotate.argtypes = [P, I, I, P]
            L.kvo_sinkhorn.argtypes = [P, I, I, I, P, P, P, P, P]
            L.kvo_header_bytes.argtypes = [I, I]
            L.kvo_header_bytes.restype = ctypes.c_size_t
            L.kvo_payload_bytes.argtypes = [I, I, I]
            L.kvo_payload_bytes.restype = ctypes.c_size_t
            L.kvo_record_bytes.argtypes = [I, I, I]
            L.kvo_record_bytes.restype = ctypes.c_size_t
            L.kvo_pack.argtypes = [P, I, I, I, I, P]
            L.kvo_unpack.argtypes = [P, I, I, I, I, P]
            L.kvo_read_header.argtypes = [P, I, I, P, P, P, P]
            L.kvo_quantize.argtypes = [P, I, I, I, P, P, P, P, P, P]
            L.kvo_codes_for_grid.argtypes = [P, I, I, I, P, P, D, D, P, P]
            L.kvo_seal.argtypes = [P, I, I, I, I, I, P, P, P]
            L.kvo_seal.restype = I
            L.kvo_dequant.argtypes = [P, I, I, I, I, I, P]
            L.kvo_attention.argtypes = [I, I, I, I, I, P, D, I, P, P, I, P, P, I, P, P, P, P]
            L.kvo_attention.restype = I
            _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def half_to_double(bits: int) -> float:
    return lib().kvo_half_to_double(int(bits) & 0xFFFF)


def double_to_half(x: float, saturate: bool = False) -> int:
    f = lib().kvo_double_to_half_sat if saturate else lib().kvo_double_to_half
    return int(f(float(x)))


def hadamard(d: int) -> np.ndarray:
    H = np.empty((d, d), np.float64)
    lib().kvo_hadamard(d, _p(H))
    return H


def rotate(X: np.ndarray) -> np.ndarray:
    X = _c(X, np.float64)
    T, d = X.shape
    Y = np.empty_like(X)
    lib().kvo_rotate(_p(X), T, d, _p(Y))
    return Y


def sinkhorn(Y: np.ndarray, iters: int = ITERS, trace: bool = False):
    """Returns (a, c, Z) or, with trace, (a, c, Z, row_dev, col_dev)."""
    Y = _c(Y, np.float64)
    T, d = Y.shape
    a = np.empty(T)
    c = np.empty(d)
    Z = np.empty_like(Y)
    rd = np.empty(max(iters, 1))
    cd = np.empty(max(iters, 1))
    lib().kvo_sinkhorn(_p(Y), T, d, iters, _p(a), _p(c), _p(Z),
                       _p(rd) if trace else None, _p(cd) if trace else None)
    if trace:
        return a, c, Z, rd[:iters], cd[:iters]
    return a, c, Z


def header_bytes(T: int = GROUP, d: int = HEAD_DIM) -> int:
    return int(lib().kvo_header_bytes(T, d))


def record_bytes(bits: int, T: int = GROUP, d: int = HEAD_DIM) -> int:
    return int(lib().kvo_record_bytes(T, d, bits))


def pack(codes: np.ndarray, bits: int, side: int) -> np.ndarray:
    codes = _c(codes, np.uint8)
    T, d = codes.shape
    out = np.zeros(int(lib().kvo_payload_bytes(T, d, bits)), np.uint8)
    lib().kvo_pack(_p(codes), T, d, bits, side, _p(out))
    return out


def unpack(payload: np.ndarray, bits: int, side: int, T: int = GROUP, d: int = HEAD_DIM) -> np.ndarray:
    payload = _c(payload, np.uint8)
    codes = np.empty((T, d), np.uint8)
    lib().kvo_unpack(_p(payload), T, d, bits, side, _p(codes))
    return codes


def read_header(record: np.ndarray, T: int = GROUP, d: int = HEAD_DIM):
    """(delta, m, a[T], c[d]) of a record, as doubles."""
    record = _c(record, np.uint8)
    delta = ctypes.c_double()
    m = ctypes.c_double()
    a = np.empty(T)
    c = np.empty(d)
    lib().kvo_read_header(_p(record), T, d, ctypes.byref(delta), ctypes.byref(m), _p(a), _p(c))
    return delta.value, m.value, a, c


def quantize(Y: np.ndarray, bits: int, a16: np.ndarray, c16: np.ndarray):
    """Grid + round-to-nearest given stored scales: (delta32, m32, codes, t)."""
    Y = _c(Y, np.float64)
    T, d = Y.shape
    a16 = _c(a16, np.float64)
    c16 = _c(c16, np.float64)
    dl = ctypes.c_float()
    m = ctypes.c_float()
    codes = np.empty((T, d), np.uint8)
    t = np.empty((T, d))
    lib().kvo_quantize(_p(Y), T, d, bits, _p(a16), _p(c16), ctypes.byref(dl), ctypes.byref(m),
                       _p(codes), _p(t))
    return dl.value, m.value, codes, t


def codes_for_grid(Y: np.ndarray, bits: int, a16, c16, m: float, delta: float):
    """(codes, t) for a given grid and stored scales."""
    Y = _c(Y, np.float64)
    T, d = Y.shape
    codes = np.empty((T, d), np.uint8)
    t = np.empty((T, d))
    lib().kvo_codes_for_grid(_p(Y), T, d, bits, _p(_c(a16, np.float64)), _p(_c(c16, np.float64)),
                             float(m), float(delta), _p(codes), _p(t))
    return codes, t


def seal(x_half: np.ndarray, bits: int, side: int, iters: int = ITERS, return_scales: bool = False):
    """Seal one fp16 group matrix x [T][d] (token rows). side 0 = K, 1 = V."""
    x = _c(np.asarray(x_half, np.float16).view(np.uint16), np.uint16)
    T, d = x.shape
    rec = np.zeros(record_bytes(bits, T, d), np.uint8)
    a = np.empty(T)
    c = np.empty(d)
    rc = lib().kvo_seal(_p(x), T, d, bits, side, iters, _p(rec), _p(a), _p(c))
    if rc != 0:
        raise ValueError("kvo_seal: bad arguments")
    if return_scales:
        return rec, a, c
    return rec


def dequant(record: np.ndarray, bits: int, side: int, frame: int = 0, T: int = GROUP,
            d: int = HEAD_DIM) -> np.ndarray:
    """frame 0 = original (rotated back), 1 = rotated frame."""
    record = _c(record, np.uint8)
    out = np.empty((T, d))
    lib().kvo_dequant(_p(record), T, d, bits, side, frame, _p(out))
    return out


def attention(q_half, scale, sink_k, sink_v, k_records, v_records, tail_k, tail_v,
              k_bits, v_bits, T: int = GROUP, return_lse: bool = False):
    """Decode attention for one (sequence, KV head). q_half: [r][d] fp16.
    sink_*/tail_*: [n][d] fp16. *_records: [n_groups][record bytes] uint8."""
    q = _c(np.asarray(q_half, np.float16).view(np.uint16), np.uint16)
    r, d = q.shape
    sk = _c(np.asarray(sink_k, np.float16).reshape(-1, d).view(np.uint16), np.uint16)
    sv = _c(np.asarray(sink_v, np.float16).reshape(-1, d).view(np.uint16), np.uint16)
    tk = _c(np.asarray(tail_k, np.float16).reshape(-1, d).view(np.uint16), np.uint16)
    tv = _c(np.asarray(tail_v, np.float16).reshape(-1, d).view(np.uint16), np.uint16)
    kr = _c(np.asarray(k_records, np.uint8).reshape(-1), np.uint8)
    vr = _c(np.asarray(v_records, np.uint8).reshape(-1), np.uint8)
    ng = kr.size // record_bytes(k_bits, T, d) if kr.size else 0
    out = np.empty((r, d))
    lse = np.empty(r)
    rc = lib().kvo_attention(d, T, r, k_bits, v_bits, _p(q), float(scale),
                             sk.shape[0], _p(sk), _p(sv), ng, _p(kr), _p(vr),
                             tk.shape[0], _p(tk), _p(tv), _p(out), _p(lse))
    if rc != 0:
        raise ValueError("kvo_attention: bad arguments")
    return (out, lse) if return_lse else out


def prefill_attention(q_half, positions, scale, sink_k, sink_v, k_records, v_records, tail_k, tail_v,
                      k_bits, v_bits, T: int = GROUP):
    """Many-query (prefill) attention for one (sequence, KV head), by its plain definition.

    q_half: [n_q][r][d] fp16, the queries of the tokens at `positions` (ints). The keys
    are the cache as it stands: sink tokens at positions 0 .. n_sink - 1, sealed group g
    at positions 128 + T g .. 128 + T g + T - 1 (its record dequantised and rotated back,
    anbeeld.com "KVarN KV Cache: Implementation and Benchmarks", 2.1 and section 1), then
    the exact tail. The query at position P attends to the keys at positions <= P
    (causal), with a plain fp64 softmax. Returns [n_q][r][d] fp64.
    """
    q = np.asarray(q_half, np.float16).astype(np.float64)
    n_q, r, d = q.shape
    kr = np.asarray(k_records, np.uint8).reshape(-1, record_bytes(k_bits, T, d)) if np.size(k_records) else []
    vr = np.asarray(v_records, np.uint8).reshape(-1, record_bytes(v_bits, T, d)) if np.size(v_records) else []
    parts_k = [np.asarray(sink_k, np.float16).reshape(-1, d).astype(np.float64)]
    parts_v = [np.asarray(sink_v, np.float16).reshape(-1, d).astype(np.float64)]
    if len(kr):
        assert parts_k[0].shape[0] == SINK, "sealed groups follow a full sink"
    for g in range(len(kr)):
        parts_k.append(dequant(kr[g], k_bits, 0, frame=0, T=T, d=d))
        parts_v.append(dequant(vr[g], v_bits, 1, frame=0, T=T, d=d))
    parts_k.append(np.asarray(tail_k, np.float16).reshape(-1, d).astype(np.float64))
    parts_v.append(np.asarray(tail_v, np.float16).reshape(-1, d).astype(np.float64))
    K = np.concatenate(parts_k)  # row j = the key at position j
    V = np.concatenate(parts_v)
    out = np.empty((n_q, r, d))
    for i, P in enumerate(positions):
        if not 0 <= P < K.shape[0]:
            raise ValueError("query position outside the cache")
        s = scale * (q[i] @ K[:P + 1].T)  # [r][P + 1]
        s -= s.max(axis=1, keepdims=True)
        w = np.exp(s)
        out[i] = (w @ V[:P + 1]) / w.sum(axis=1, keepdims=True)
    return out


def bits_per_element(bits: int, T: int = GROUP, d: int = HEAD_DIM) -> float:
    """Body bits per cached element of the record format: payload plus metadata."""
    return record_bytes(bits, T, d) * 8.0 / (T * d)


class OracleCache:
    """Reference model of one layer's KVarN cache for a set of sequences.

    Region rules (anbeeld.com, 2.1): positions 0..127 are the sink (exact fp16);
    body group g covers positions [128 + 128 g, 256 + 128 g) and is sealed when its
    last token arrives; the partial newest group (the tail) stays exact fp16.
    With tail_floor F > 0 (the BeeLlama floor of the same section, F = 1 there) the
    exact tail never drops below F full groups: the oldest exact group is sealed only
    once F + 1 full groups are exact, i.e. group g seals when group g + F fills.
    K and V of each KV head are sealed as separate 128 x d matrices.
    """

    def __init__(self, num_kv_heads: int, k_bits: int, v_bits: int, head_dim: int = HEAD_DIM,
                 iters: int = ITERS, tail_floor: int = 0):
        self.hkv = num_kv_heads
        self.kb = k_bits
        self.vb = v_bits
        self.d = head_dim
        self.iters = iters
        self.floor = tail_floor
        self.seqs = {}

    def _seq(self, s):
        if s not in self.seqs:
            self.seqs[s] = {
                "n": 0,
                "sink_k": np.zeros((SINK, self.hkv, self.d), np.float16),
                "sink_v": np.zeros((SINK, self.hkv, self.d), np.float16),
                "tail_k": [],  # exact tail tokens in position order, each [Hkv][d]
                "tail_v": [],
                "krec": [],  # per group: [Hkv][record] uint8
                "vrec": [],
            }
        return self.seqs[s]

    def append(self, s, k, v):
        """Append tokens k, v [n][Hkv][d] fp16 to sequence s, sealing each group due."""
        st = self._seq(s)
        for t in range(k.shape[0]):
            p = st["n"]
            if p < SINK:
                st["sink_k"][p] = k[t]
                st["sink_v"][p] = v[t]
            else:
                st["tail_k"].append(np.asarray(k[t], np.float16))
                st["tail_v"].append(np.asarray(v[t], np.float16))
                if len(st["tail_k"]) == GROUP * (self.floor + 1):
                    gk = np.stack(st["tail_k"][:GROUP])  # the oldest exact group [T][Hkv][d]
                    gv = np.stack(st["tail_v"][:GROUP])
                    st["krec"].append(np.stack([seal(gk[:, h, :], self.kb, 0, self.iters) for h in range(self.hkv)]))
                    st["vrec"].append(np.stack([seal(gv[:, h, :], self.vb, 1, self.iters) for h in range(self.hkv)]))
                    del st["tail_k"][:GROUP]
                    del st["tail_v"][:GROUP]
            st["n"] = p + 1

    def tail(self, s):
        """Exact tail tokens of sequence s, (k, v) [n_tail][Hkv][d] fp16."""
        st = self._seq(s)
        if not st["tail_k"]:
            z = np.zeros((0, self.hkv, self.d), np.float16)
            return z, z
        return np.stack(st["tail_k"]), np.stack(st["tail_v"])

    def length(self, s):
        return self._seq(s)["n"]

    def regions(self, s):
        st = self._seq(s)
        n = st["n"]
        n_sink = min(n, SINK)
        n_groups = len(st["krec"])
        n_tail = len(st["tail_k"])
        assert n_tail == max(n - SINK, 0) - GROUP * n_groups
        return n_sink, n_groups, n_tail

    def prefill_attend(self, s, q, scale, kv_heads=None):
        """q: [n_q][Hq][d] fp16, the queries of the last n_q tokens of sequence s ->
        out [n_q][Hq][d] fp64, each attending causally to the cache as it stands."""
        st = self._seq(s)
        n = st["n"]
        n_sink, n_groups, n_tail = self.regions(s)
        n_q, hq = q.shape[0], q.shape[1]
        r = hq // self.hkv
        pos = list(range(n - n_q, n))
        out = np.full((n_q, hq, self.d), np.nan)
        heads = range(self.hkv) if kv_heads is None else kv_heads
        tk, tv = self.tail(s)
        for h in heads:
            kr = np.stack([g[h] for g in st["krec"]]) if n_groups else np.zeros((0,), np.uint8)
            vr = np.stack([g[h] for g in st["vrec"]]) if n_groups else np.zeros((0,), np.uint8)
            out[:, h * r:(h + 1) * r] = prefill_attention(
                q[:, h * r:(h + 1) * r], pos, scale, st["sink_k"][:n_sink, h], st["sink_v"][:n_sink, h],
                kr, vr, tk[:, h], tv[:, h], self.kb, self.vb)
        return out

    def attend(self, s, q, scale, kv_heads=None):
        """q: [Hq][d] fp16 for sequence s -> out [Hq][d] fp64 (contiguous GQA grouping)."""
        st = self._seq(s)
        n_sink, n_groups, n_tail = self.regions(s)
        hq = q.shape[0]
        r = hq // self.hkv
        out = np.full((hq, self.d), np.nan)
        heads = range(self.hkv) if kv_heads is None else kv_heads
        tk, tv = self.tail(s)
        for h in heads:
            kr = np.stack([g[h] for g in st["krec"]]) if n_groups else np.zeros((0,), np.uint8)
            vr = np.stack([g[h] for g in st["vrec"]]) if n_groups else np.zeros((0,), np.uint8)
            out[h * r:(h + 1) * r] = attention(
                q[h * r:(h + 1) * r], scale,
                st["sink_k"][:n_sink, h], st["sink_v"][:n_sink, h], kr, vr,
                tk[:, h], tv[:, h], self.kb, self.vb)
        return out
