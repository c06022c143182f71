"""Decode calls with pinned host buffers for q, k, v and out.

Under unified addressing, pinned host memory from cudaHostAlloc (what torch's
pin_memory returns) is reachable by kernels at the same address; on Grace the GPU reads
and writes it over NVLink-C2C. The C ABI accepts such buffers wherever it takes device
buffers (kvarn_device_accessible says which pointers qualify). These tests run the same
calls on twin caches, one with device buffers and one with pinned host buffers, and
require bitwise-equal outputs and records. A pointer is passed to a kernel only after
kvarn_device_accessible has confirmed it.
"""
import numpy as np
import pytest

from quantized_kv_cache_seal_gb300 import kvarn as K
from quantized_kv_cache_seal_gb300 import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _cache():
    from quantized_kv_cache_seal_gb300.cache import KVarNCache
    return KVarNCache(num_layers=1, max_seqs=3, num_q_heads=8, num_kv_heads=2, k_bits=2, v_bits=2, max_seq_len=2048)


def _pinned(t):
    h = t.cpu().pin_memory()
    if not K.kvarn_device_accessible(h):
        pytest.skip("pinned host memory is not mapped for kernels on this system")
    return h


def test_device_accessible_classifies_pointers():
    d = torch.empty(64, dtype=torch.float16, device="cuda")
    assert K.kvarn_device_accessible(d)
    pageable = np.zeros(64, np.float16)
    assert not K.kvarn_device_accessible(pageable.ctypes.data)
    h = torch.empty(64, dtype=torch.float16).pin_memory()
    K.kvarn_device_accessible(h)  # answers either way without an error


def test_decode_step_with_pinned_host_buffers_matches_device_buffers():
    a, b = _cache(), _cache()
    lengths = [300, 1000, 255]  # the last one seals group 0 on its first step
    for c in (a, b):
        for s, n in enumerate(lengths):
            k, v = workloads.torch_tokens(7, s, 0, n, 2)
            c.append(0, [s], [n], k.contiguous(), v.contiguous())
    torch.cuda.synchronize()
    for step in range(3):
        ks, vs = [], []
        for s, n in enumerate(lengths):
            k, v = workloads.torch_tokens(7, s, n + step, 1, 2)
            ks.append(k)
            vs.append(v)
        k = torch.cat(ks).contiguous()
        v = torch.cat(vs).contiguous()
        q = workloads.torch_queries(7, 3, 3, 8)[step].contiguous()
        out_d = a.decode_step(0, [0, 1, 2], k, v, q)
        hk, hv, hq = _pinned(k), _pinned(v), _pinned(q)
        hout = _pinned(torch.empty_like(q))
        b.decode_step(0, [0, 1, 2], hk, hv, hq, out=hout)
        torch.cuda.synchronize()
        assert a.check_device_error() == 0 and b.check_device_error() == 0
        assert torch.equal(out_d.cpu(), hout), f"step {step}"
    # the group sealed from a host-resident token matches the one sealed from the device
    for which in (0, 1):
        assert torch.equal(a.record(0, 2, 0, 1, which), b.record(0, 2, 0, 1, which))


def test_decode_attention_with_pinned_host_query_and_output():
    a = _cache()
    k, v = workloads.torch_tokens(9, 0, 0, 700, 2)
    a.append(0, [0], [700], k.contiguous(), v.contiguous())
    q = workloads.torch_queries(9, 1, 1, 8)[0].contiguous()
    out_d = a.decode_attention(0, [0], q)
    hq = _pinned(q)
    hout = _pinned(torch.empty_like(q))
    a.decode_attention(0, [0], hq, out=hout)
    torch.cuda.synchronize()
    assert a.check_device_error() == 0
    assert torch.equal(out_d.cpu(), hout)
