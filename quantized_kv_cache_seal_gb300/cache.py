"""A small owner object over the C ABI: allocates the cache's device block with torch
(PyTorch supplies device memory and streams only) and forwards every call to
libkvarn.so."""
from __future__ import annotations

import math
from typing import Optional, Sequence

import torch

from . import kvarn as K


class KVarNCache:
    def __init__(self, num_layers=1, max_seqs=1, num_q_heads=32, num_kv_heads=8, k_bits=2, v_bits=2,
                 sinkhorn_iters=16, max_seq_len=32768, pool_groups=None, device="cuda", flags=0, tail_floor=0):
        self.cfg = K.make_config(num_layers=num_layers, max_seqs=max_seqs, num_q_heads=num_q_heads,
                                 num_kv_heads=num_kv_heads, k_bits=k_bits, v_bits=v_bits,
                                 sinkhorn_iters=sinkhorn_iters, max_seq_len=max_seq_len, pool_groups=pool_groups,
                                 flags=flags, tail_floor=tail_floor)
        self.nbytes = K.kvarn_cache_required_bytes(self.cfg)
        self.mem = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device)
        base = self.mem.data_ptr()
        self.base = (base + 255) // 256 * 256
        self.handle = K.kvarn_cache_create(self.cfg, self.base, self.nbytes)
        self.scale = 1.0 / math.sqrt(128)

    def close(self):
        if self.handle:
            K.kvarn_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _stream(stream):
        return stream if stream is not None else torch.cuda.current_stream()

    def append(self, layer: int, seq_ids: Sequence[int], n_tokens: Sequence[int], k: torch.Tensor, v: torch.Tensor,
               stream=None):
        K.kvarn_append(self.handle, layer, list(seq_ids), list(n_tokens), k, v, self._stream(stream))

    def decode_attention(self, layer: int, seq_ids: Sequence[int], q: torch.Tensor, out: Optional[torch.Tensor] = None,
                         scale: Optional[float] = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(q)
        K.kvarn_decode_attention(self.handle, layer, list(seq_ids), q, out, self.scale if scale is None else scale,
                                 self._stream(stream))
        return out

    def decode_step(self, layer: int, seq_ids: Sequence[int], k: torch.Tensor, v: torch.Tensor, q: torch.Tensor,
                    out: Optional[torch.Tensor] = None, scale: Optional[float] = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(q)
        K.kvarn_decode_step(self.handle, layer, list(seq_ids), k, v, q, out, self.scale if scale is None else scale,
                            self._stream(stream))
        return out

    def prefill_attention(self, layer: int, seq_ids: Sequence[int], q_lens: Sequence[int], q: torch.Tensor,
                          out: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                          stream=None) -> torch.Tensor:
        """Causal attention of the last q_lens[i] tokens of each sequence over the cache as
        it stands; q, out: [sum(q_lens)][Hq][128] fp16."""
        if out is None:
            out = torch.empty_like(q)
        K.kvarn_prefill_attention(self.handle, layer, list(seq_ids), list(q_lens), q, out,
                                  self.scale if scale is None else scale, self._stream(stream))
        return out

    def prefill(self, layer: int, seq_ids: Sequence[int], n_tokens: Sequence[int], k: torch.Tensor, v: torch.Tensor,
                q: torch.Tensor, out: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                stream=None) -> torch.Tensor:
        """Append a prompt chunk (sealing the groups it completes) and attend its queries."""
        if out is None:
            out = torch.empty_like(q)
        K.kvarn_prefill(self.handle, layer, list(seq_ids), list(n_tokens), k, v, q, out,
                        self.scale if scale is None else scale, self._stream(stream))
        return out

    def dequant_group(self, layer, seq_id, group, kv_head, which, frame=0, stream=None) -> torch.Tensor:
        out = torch.empty((128, 128), dtype=torch.float32, device=self.mem.device)
        K.kvarn_dequant_group(self.handle, layer, seq_id, group, kv_head, which, frame, out, True,
                              self._stream(stream))
        return out

    def record(self, layer, seq_id, group, kv_head, which) -> torch.Tensor:
        """Copy of one record's bytes (uint8 tensor on the device)."""
        ptr, n = K.kvarn_group_record(self.handle, layer, seq_id, group, kv_head, which)
        off = ptr - self.mem.data_ptr()
        return self.mem[off:off + n].clone()

    def exact_regions(self, layer, seq_id):
        """(sink_k, sink_v, tail_k, tail_v) fp16 views: sink [Hkv][128][128], tail ring
        [Hkv][128 (tail_floor + 1)][128] (slot = (position - 128) mod ring rows)."""
        ptrs = K.kvarn_exact_regions(self.handle, layer, seq_id)
        ring = 128 * (self.cfg.tail_floor + 1)
        views = []
        for i, ptr in enumerate(ptrs):
            rows = 128 if i < 2 else ring
            off = ptr - self.mem.data_ptr()
            n = self.cfg.num_kv_heads * rows * 128 * 2
            views.append(self.mem[off:off + n].view(torch.float16).view(self.cfg.num_kv_heads, rows, 128))
        return tuple(views)

    def exact_tail(self, layer, seq_id):
        """The exact tail tokens in position order: (tail_k, tail_v) fp16 [Hkv][n_tail][128]."""
        n = self.length(layer, seq_id)
        F = self.cfg.tail_floor
        sealed = max(0, (n - 128) // 128 - F) if n > 128 else 0
        n_tail = n - 128 - 128 * sealed if n > 128 else 0
        ring = 128 * (F + 1)
        _, _, tk, tv = self.exact_regions(layer, seq_id)
        idx = (128 * sealed + torch.arange(n_tail, device=tk.device)) % ring
        return tk[:, idx], tv[:, idx]

    def length(self, layer, seq_id) -> int:
        return K.kvarn_seq_length(self.handle, layer, seq_id)

    def snapshot(self, pinned: bool = True, stream=None) -> torch.Tensor:
        """The cache's state as a host byte image (uint8 tensor, pinned by default)."""
        n = K.kvarn_snapshot_bytes(self.handle)
        buf = torch.empty(n, dtype=torch.uint8, pin_memory=pinned and self.mem.is_cuda)
        K.kvarn_snapshot_save(self.handle, buf, n, self._stream(stream))
        return buf

    def restore(self, image, stream=None):
        """Replace the cache's state by a host image from snapshot() (tensor or numpy array)."""
        n = image.numel() if hasattr(image, "numel") else image.nbytes
        K.kvarn_snapshot_load(self.handle, image, n, self._stream(stream))

    def save(self, path, stream=None):
        self.snapshot(pinned=False, stream=stream).numpy().tofile(path)

    def load(self, path, stream=None):
        import numpy as np
        self.restore(np.fromfile(path, dtype=np.uint8), stream=stream)

    def release(self, seq_id):
        K.kvarn_seq_release(self.handle, seq_id)

    def stats(self):
        return K.kvarn_cache_stats(self.handle)

    def check_device_error(self, stream=None) -> int:
        return K.kvarn_check_device_error(self.handle, self._stream(stream))


def seal_groups(x: torch.Tensor, bits: int, which: int, iters: int = 16, scales: bool = False, stream=None):
    """Seal fp16 matrices x[n][128][128]; returns (records uint8 [n][rec], scales f32 [n][256] or None)."""
    assert x.dtype == torch.float16 and x.is_cuda and x.is_contiguous() and x.shape[1:] == (128, 128)
    n = x.shape[0]
    rec = torch.empty((n, K.kvarn_record_bytes(bits)), dtype=torch.uint8, device=x.device)
    sc = torch.empty((n, 256), dtype=torch.float32, device=x.device) if scales else None
    K.kvarn_seal_groups(x, n, bits, which, iters, rec, sc,
                        stream if stream is not None else torch.cuda.current_stream())
    return rec, sc
