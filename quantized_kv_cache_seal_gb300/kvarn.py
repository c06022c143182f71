"""Thin ctypes binding of libkvarn.so (``include/kvarn.h``): argument marshalling only.

Every function carries the C name. Device buffers may be given as torch tensors
(their ``data_ptr()`` is passed) or as integer addresses; host integer arrays as
Python sequences. A non-OK status raises :class:`KVarNError`. All arithmetic runs in
the CUDA library; there is no fallback path: if the library cannot be loaded, the
import of this module fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from . import build as _build

STATUS = {0: "KVARN_OK", 1: "KVARN_EINVAL", 2: "KVARN_ENOMEM", 3: "KVARN_ECAPACITY", 4: "KVARN_ECUDA",
          5: "KVARN_ESTATE", 6: "KVARN_ETIMEOUT"}
KVARN_FLAG_HOST_ONLY = 1
KVARN_FLAG_TEST_STALL = 2

# every entry point declared in include/kvarn.h
EXPORTS = [
    "kvarn_record_bytes", "kvarn_cache_required_bytes", "kvarn_cache_create", "kvarn_cache_destroy",
    "kvarn_append", "kvarn_decode_attention", "kvarn_decode_attention_noalloc", "kvarn_decode_step", "kvarn_dequant_group",
    "kvarn_seq_release", "kvarn_seq_length", "kvarn_group_record", "kvarn_exact_regions",
    "kvarn_cache_stats", "kvarn_seal_groups", "kvarn_check_device_error", "kvarn_status_string",
    "kvarn_last_error", "kvarn_partition_units", "kvarn_device_accessible", "kvarn_prefill_attention",
    "kvarn_prefill", "kvarn_snapshot_bytes", "kvarn_snapshot_save", "kvarn_snapshot_load",
]


class KVarNError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


class kvarn_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_layers", "max_seqs", "num_q_heads", "num_kv_heads", "head_dim", "k_bits", "v_bits",
        "group_size", "sink_tokens", "sinkhorn_iters", "max_seq_len", "pool_groups", "flags", "tail_floor")]


class kvarn_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "device_bytes", "record_bytes_k", "record_bytes_v", "slot_bytes", "pool_slots_total",
        "pool_slots_used", "tokens_cached", "sealed_tokens", "exact_tokens", "sealed_bytes",
        "exact_bytes")] + [("body_bits_per_element", ctypes.c_double),
                           ("all_in_bits_per_element", ctypes.c_double)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libkvarn.so (building it first if needed) and declare the signatures."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build_if_missing else _build.LIB
    if not os.path.exists(path):
        raise OSError(f"libkvarn.so not built: {path}")
    L = ctypes.CDLL(path)
    P, I32, I64, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    IP = ctypes.POINTER(ctypes.c_int32)
    L.kvarn_record_bytes.argtypes = [I32]
    L.kvarn_record_bytes.restype = SZ
    L.kvarn_cache_required_bytes.argtypes = [ctypes.POINTER(kvarn_config), ctypes.POINTER(SZ)]
    L.kvarn_cache_create.argtypes = [ctypes.POINTER(kvarn_config), P, SZ, ctypes.POINTER(P)]
    L.kvarn_cache_destroy.argtypes = [P]
    L.kvarn_cache_destroy.restype = None
    L.kvarn_append.argtypes = [P, I32, I32, IP, IP, P, P, P]
    L.kvarn_decode_attention.argtypes = [P, I32, I32, IP, P, P, F, P]
    L.kvarn_decode_attention_noalloc.argtypes = [P, I32, I32, IP, P, P, F, P]
    L.kvarn_decode_step.argtypes = [P, I32, I32, IP, P, P, P, P, F, P]
    L.kvarn_prefill_attention.argtypes = [P, I32, I32, IP, IP, P, P, F, P]
    L.kvarn_prefill.argtypes = [P, I32, I32, IP, IP, P, P, P, P, F, P]
    L.kvarn_snapshot_bytes.argtypes = [P, ctypes.POINTER(SZ)]
    L.kvarn_snapshot_save.argtypes = [P, P, SZ, P]
    L.kvarn_snapshot_load.argtypes = [P, P, SZ, P]
    L.kvarn_dequant_group.argtypes = [P, I32, I32, I32, I32, I32, I32, I32, P, P]
    L.kvarn_seq_release.argtypes = [P, I32]
    L.kvarn_seq_length.argtypes = [P, I32, I32, ctypes.POINTER(I64)]
    L.kvarn_group_record.argtypes = [P, I32, I32, I32, I32, I32, ctypes.POINTER(P), ctypes.POINTER(SZ)]
    L.kvarn_exact_regions.argtypes = [P, I32, I32] + [ctypes.POINTER(P)] * 4
    L.kvarn_cache_stats.argtypes = [P, ctypes.POINTER(kvarn_stats)]
    L.kvarn_seal_groups.argtypes = [P, I32, I32, I32, I32, P, P, P]
    L.kvarn_check_device_error.argtypes = [P, P]
    L.kvarn_status_string.argtypes = [I32]
    L.kvarn_status_string.restype = ctypes.c_char_p
    L.kvarn_last_error.argtypes = []
    L.kvarn_last_error.restype = ctypes.c_char_p
    L.kvarn_partition_units.argtypes = [I32, IP, IP, I32, I32, I32, I32, IP, IP]
    L.kvarn_device_accessible.argtypes = [P, IP]
    for name in EXPORTS:
        fn = getattr(L, name)
        if fn.restype is ctypes.c_int:  # default: status enum
            fn.restype = I32
    _lib = L
    return L


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"expected a tensor or an address, got {type(x)}")


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


def _ints(xs: Sequence[int]):
    arr = (ctypes.c_int32 * len(xs))(*[int(v) for v in xs])
    return arr


def _check(rc: int, where: str):
    if rc != 0:
        detail = load().kvarn_last_error().decode() if rc == 4 else ""
        raise KVarNError(rc, where, detail)


def make_config(num_layers=1, max_seqs=1, num_q_heads=32, num_kv_heads=8, k_bits=2, v_bits=2,
                sinkhorn_iters=16, max_seq_len=32768, pool_groups=None, flags=0, head_dim=128,
                group_size=128, sink_tokens=128, tail_floor=0) -> kvarn_config:
    if pool_groups is None:
        pool_groups = max_seqs * num_layers * max(0, (max_seq_len - 128) // 128 - tail_floor)
    return kvarn_config(num_layers, max_seqs, num_q_heads, num_kv_heads, head_dim, k_bits, v_bits,
                        group_size, sink_tokens, sinkhorn_iters, max_seq_len, pool_groups, flags, tail_floor)


def kvarn_record_bytes(bits: int) -> int:
    return int(load().kvarn_record_bytes(bits))


def kvarn_cache_required_bytes(cfg: kvarn_config) -> int:
    n = ctypes.c_size_t()
    _check(load().kvarn_cache_required_bytes(ctypes.byref(cfg), ctypes.byref(n)), "kvarn_cache_required_bytes")
    return n.value


def kvarn_cache_create(cfg: kvarn_config, dev_mem, nbytes: int) -> int:
    h = ctypes.c_void_p()
    _check(load().kvarn_cache_create(ctypes.byref(cfg), _ptr(dev_mem), nbytes, ctypes.byref(h)),
           "kvarn_cache_create")
    return h.value


def kvarn_cache_destroy(handle: int) -> None:
    load().kvarn_cache_destroy(handle)


def kvarn_append(handle, layer, seq_ids, n_tokens, k, v, stream=None):
    _check(load().kvarn_append(handle, layer, len(seq_ids), _ints(seq_ids), _ints(n_tokens), _ptr(k), _ptr(v),
                               _stream(stream)), "kvarn_append")


def kvarn_decode_attention(handle, layer, seq_ids, q, out, softmax_scale, stream=None):
    _check(load().kvarn_decode_attention(handle, layer, len(seq_ids), _ints(seq_ids), _ptr(q), _ptr(out),
                                         float(softmax_scale), _stream(stream)), "kvarn_decode_attention")


def kvarn_decode_attention_noalloc(handle, layer, seq_ids, q, out, softmax_scale, stream=None):
    _check(load().kvarn_decode_attention_noalloc(handle, layer, len(seq_ids), _ints(seq_ids), _ptr(q), _ptr(out),
                                                 float(softmax_scale), _stream(stream)),
           "kvarn_decode_attention_noalloc")


def kvarn_decode_step(handle, layer, seq_ids, k, v, q, out, softmax_scale, stream=None):
    _check(load().kvarn_decode_step(handle, layer, len(seq_ids), _ints(seq_ids), _ptr(k), _ptr(v), _ptr(q),
                                    _ptr(out), float(softmax_scale), _stream(stream)), "kvarn_decode_step")


def kvarn_prefill_attention(handle, layer, seq_ids, q_lens, q, out, softmax_scale, stream=None):
    _check(load().kvarn_prefill_attention(handle, layer, len(seq_ids), _ints(seq_ids), _ints(q_lens), _ptr(q),
                                          _ptr(out), float(softmax_scale), _stream(stream)),
           "kvarn_prefill_attention")


def kvarn_prefill(handle, layer, seq_ids, n_tokens, k, v, q, out, softmax_scale, stream=None):
    _check(load().kvarn_prefill(handle, layer, len(seq_ids), _ints(seq_ids), _ints(n_tokens), _ptr(k), _ptr(v),
                                _ptr(q), _ptr(out), float(softmax_scale), _stream(stream)), "kvarn_prefill")


def kvarn_dequant_group(handle, layer, seq_id, group, kv_head, which, frame, out, out_fp32=True, stream=None):
    _check(load().kvarn_dequant_group(handle, layer, seq_id, group, kv_head, which, frame, int(bool(out_fp32)),
                                      _ptr(out), _stream(stream)), "kvarn_dequant_group")


def _host_ptr(buf) -> int:
    """Address of a host buffer: a numpy array, a (CPU, possibly pinned) torch tensor or an int."""
    if isinstance(buf, int):
        return buf
    if hasattr(buf, "data_ptr"):
        return buf.data_ptr()
    return buf.ctypes.data


def kvarn_snapshot_bytes(handle) -> int:
    n = ctypes.c_size_t()
    _check(load().kvarn_snapshot_bytes(handle, ctypes.byref(n)), "kvarn_snapshot_bytes")
    return n.value


def kvarn_snapshot_save(handle, dst, nbytes, stream=None):
    _check(load().kvarn_snapshot_save(handle, _host_ptr(dst), nbytes, _stream(stream)), "kvarn_snapshot_save")


def kvarn_snapshot_load(handle, src, nbytes, stream=None):
    _check(load().kvarn_snapshot_load(handle, _host_ptr(src), nbytes, _stream(stream)), "kvarn_snapshot_load")


def kvarn_seq_release(handle, seq_id):
    _check(load().kvarn_seq_release(handle, seq_id), "kvarn_seq_release")


def kvarn_seq_length(handle, layer, seq_id) -> int:
    n = ctypes.c_int64()
    _check(load().kvarn_seq_length(handle, layer, seq_id, ctypes.byref(n)), "kvarn_seq_length")
    return n.value


def kvarn_group_record(handle, layer, seq_id, group, kv_head, which):
    p = ctypes.c_void_p()
    n = ctypes.c_size_t()
    _check(load().kvarn_group_record(handle, layer, seq_id, group, kv_head, which, ctypes.byref(p),
                                     ctypes.byref(n)), "kvarn_group_record")
    return p.value, n.value


def kvarn_exact_regions(handle, layer, seq_id):
    ps = [ctypes.c_void_p() for _ in range(4)]
    _check(load().kvarn_exact_regions(handle, layer, seq_id, *[ctypes.byref(x) for x in ps]), "kvarn_exact_regions")
    return tuple(x.value for x in ps)


def kvarn_cache_stats(handle) -> kvarn_stats:
    s = kvarn_stats()
    _check(load().kvarn_cache_stats(handle, ctypes.byref(s)), "kvarn_cache_stats")
    return s


def kvarn_seal_groups(x, n, bits, which, sinkhorn_iters, records, scales=None, stream=None):
    _check(load().kvarn_seal_groups(_ptr(x), n, bits, which, sinkhorn_iters, _ptr(records), _ptr(scales),
                                    _stream(stream)), "kvarn_seal_groups")


def kvarn_check_device_error(handle, stream=None) -> int:
    return int(load().kvarn_check_device_error(handle, _stream(stream)))


def kvarn_partition_units(units, head, max_ctas: int, max_span: int, min_load: int, item_cost: int = 0):
    """Cut table of the decode scheduler's partition (host only): list of n + 1 cuts."""
    I32 = ctypes.c_int32
    nb = len(units)
    U = (I32 * max(nb, 1))(*units)
    H = (I32 * max(nb, 1))(*head)
    cuts = (I32 * (max_ctas + 1))()
    n = I32()
    _check(load().kvarn_partition_units(nb, U, H, max_ctas, max_span, min_load, item_cost, cuts, ctypes.byref(n)),
           "kvarn_partition_units")
    return [int(cuts[i]) for i in range(n.value + 1)]


def kvarn_device_accessible(ptr) -> bool:
    """Can kernels dereference this pointer as given (device memory, or pinned host
    memory mapped at the same address)?"""
    a = ctypes.c_int32()
    _check(load().kvarn_device_accessible(_ptr(ptr), ctypes.byref(a)), "kvarn_device_accessible")
    return bool(a.value)


def kvarn_status_string(status: int) -> str:
    return load().kvarn_status_string(status).decode()


def kvarn_last_error() -> str:
    return load().kvarn_last_error().decode()
