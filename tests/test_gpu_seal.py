"""GPU parity of the group seal and of the dequantisation path (calls through the C ABI).

Seal: fig1.dev "KVarN ...", "What it is"; anbeeld.com "KVarN KV Cache: Implementation
and Benchmarks", sections 1 and 2.1. Protocol: tests/parity.py."""
import numpy as np
import pytest

import oracle
from quantized_kv_cache_seal_gb300 import workloads
from tests import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _seal_gpu(x_np, bits, which, iters=16):
    from quantized_kv_cache_seal_gb300.cache import seal_groups
    x = torch.from_numpy(np.ascontiguousarray(x_np)).cuda()
    rec, sc = seal_groups(x, bits, which, iters=iters, scales=True)
    torch.cuda.synchronize()
    return rec.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
@pytest.mark.parametrize("which", [0, 1])
def test_seal_parity(bits, which):
    xs = np.concatenate([workloads.group_matrices(100 + bits, 24),
                         workloads.group_matrices(200 + bits, 8, spike_frac=0.05)])
    rec, sc = _seal_gpu(xs, bits, which)
    mism = 0
    for i in range(xs.shape[0]):
        mism += parity.check_seal(xs[i], rec[i], bits, which, sc[i], label=f"b{bits} w{which} #{i}")
    assert mism <= 1e-3 * xs.size


def test_seal_is_deterministic():
    xs = workloads.group_matrices(7, 16)
    r1, _ = _seal_gpu(xs, 2, 0)
    r2, _ = _seal_gpu(xs, 2, 0)
    assert np.array_equal(r1, r2)


@pytest.mark.parametrize("iters", [0, 1, 3])
def test_seal_iteration_counts(iters):
    xs = workloads.group_matrices(11, 4)
    rec, sc = _seal_gpu(xs, 4, 0, iters=iters)
    if iters == 0:
        assert np.all(sc == 1.0)
    for i in range(xs.shape[0]):
        parity.check_seal(xs[i], rec[i], 4, 0, sc[i], iters=iters, label=f"iters {iters} #{i}")


def test_seal_degenerate_matrices():
    """All zero, one non-zero row, constant, a single huge spike, fp16 extremes."""
    xs = np.zeros((6, 128, 128), np.float16)
    xs[1, 5, :] = 1.5
    xs[2, :, :] = 0.25
    xs[3, 3, 7] = 60000.0
    xs[4] = workloads.tiny_matrix(3, 128, 128, 1000.0)
    xs[5] = (workloads.tiny_matrix(4, 128, 128, 1.0).astype(np.float32) * 1e-4).astype(np.float16)
    for bits in (2, 8):
        for which in (0, 1):
            rec, sc = _seal_gpu(xs, bits, which)
            for i in range(xs.shape[0]):
                parity.check_seal(xs[i], rec[i], bits, which, sc[i], label=f"degenerate {i} b{bits} w{which}")
            # all-zero matrix: unit scales, delta 1, all codes 0
            d, m, a, c = oracle.read_header(rec[0])
            assert d == 1.0 and m == 0.0 and np.all(a == 1.0) and np.all(c == 1.0)
            assert not rec[0][528:].any()


@pytest.mark.parametrize("bits,which,frame", [(2, 0, 0), (2, 1, 1), (4, 0, 1), (4, 1, 0), (8, 0, 0), (8, 1, 1),
                                                (3, 0, 0), (3, 1, 1), (5, 0, 1), (6, 1, 0)])
def test_dequant_group_parity(bits, which, frame):
    from quantized_kv_cache_seal_gb300.cache import KVarNCache
    if bits in (3, 5, 6):  # odd widths come in symmetric pairs
        kb = vb = bits
    else:
        kb, vb = (bits, 2) if which == 0 else (2, bits)
    cache = KVarNCache(num_layers=1, max_seqs=1, num_q_heads=4, num_kv_heads=2, k_bits=kb, v_bits=vb,
                       max_seq_len=1024)
    src = workloads.TokenSource(31, 0, 2)
    k, v = src.tokens(0, 128 + 256 + 10)
    cache.append(0, [0], [k.shape[0]], torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    for g in range(2):
        for h in range(2):
            out = cache.dequant_group(0, 0, g, h, which, frame).cpu().numpy()
            rec = cache.record(0, 0, g, h, which).cpu().numpy()
            ref = oracle.dequant(rec, bits, which, frame)
            scale = np.abs(ref).max()
            assert np.abs(out - ref).max() <= 2e-6 * scale
            x = (k if which == 0 else v)[128 + 128 * g:256 + 128 * g, h]
            parity.check_seal(x, rec, bits, which, label=f"cache group {g} head {h}")
