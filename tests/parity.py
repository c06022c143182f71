"""GPU-vs-oracle comparison helpers (test infrastructure).

Seal parity is checked in decoupled steps so that one fp16 rounding difference in a
scale cannot cascade into many code differences:
  1. layout: the GPU payload, unpacked and re-packed by the oracle, is byte-identical;
  2. scales: the GPU's fp32 Sinkhorn scales (before fp16 rounding) agree with the
     oracle's fp64 ones to 1e-4 relative; the stored fp16 scales equal the oracle's
     fp16 rounding except where the oracle value lies within 1e-4 relative of an fp16
     rounding midpoint (then one ulp either way);
  3. grid: m and delta agree with the oracle's grid recomputed from the GPU's stored
     scales to 1e-5 relative to the grid range;
  4. codes: the oracle recomputes every code from the GPU's own metadata; codes that
     differ must lie within 1e-3 of a rounding boundary and be at most 0.1 %.
Attention parity: max |o_gpu - o_ref| <= 2e-3 * ||o_ref||_2 per (sequence, head), with
o_ref the oracle's fp64 attention over the GPU's records and exact regions.
"""
import numpy as np

import oracle

SCALE_RTOL = 1e-4
GRID_RTOL = 1e-5
BOUNDARY = 1e-3
MAX_CODE_MISMATCH = 1e-3
ATTN_TOL = 2e-3


def _near_half_midpoint(x: np.ndarray, rtol: float) -> np.ndarray:
    """True where x lies within rtol (relative) of a midpoint between two fp16 values."""
    x = np.asarray(x, np.float64)
    lo = x.astype(np.float16)
    lo64 = lo.astype(np.float64)
    up = np.nextafter(lo, np.float16(np.inf)).astype(np.float64)
    dn = np.nextafter(lo, np.float16(-np.inf)).astype(np.float64)
    mid_up = (lo64 + up) / 2
    mid_dn = (lo64 + dn) / 2
    near = (np.abs(x - mid_up) <= rtol * np.abs(x)) | (np.abs(x - mid_dn) <= rtol * np.abs(x))
    return near


def check_seal(x_half: np.ndarray, rec_gpu: np.ndarray, bits: int, side: int, scales_gpu=None, iters: int = 16,
               label: str = ""):
    """Check one GPU record of the fp16 matrix x_half [128][128] against the oracle."""
    h = oracle.header_bytes()
    rec_gpu = np.asarray(rec_gpu, np.uint8)
    assert rec_gpu.size == oracle.record_bytes(bits), label
    # 1. layout
    codes_gpu = oracle.unpack(rec_gpu[h:], bits, side)
    assert np.array_equal(oracle.pack(codes_gpu, bits, side), rec_gpu[h:]), f"{label}: payload layout"
    assert rec_gpu[8:16].tolist() == [0] * 8, f"{label}: reserved bytes"
    # 2. scales
    rec_o, a_o, c_o = oracle.seal(x_half, bits, side, iters=iters, return_scales=True)
    delta_g, m_g, a16_g, c16_g = oracle.read_header(rec_gpu)
    if scales_gpu is not None:
        # Only values that fp16 can hold matter: beyond 65504 the stored scale saturates and
        # below 2^-24 it flushes to zero (degenerate inputs on which Sinkhorn diverges drive
        # the unrounded fp32 scales out of range). Those are checked through the stored fp16.
        a_g = np.asarray(scales_gpu[:128], np.float64)
        c_g = np.asarray(scales_gpu[128:], np.float64)
        for name, got, ref in (("token", a_g, a_o), ("channel", c_g, c_o)):
            inr = (ref >= 2.0 ** -24) & (ref <= 65504.0)
            assert np.all(np.abs(got[inr] - ref[inr]) <= SCALE_RTOL * np.abs(ref[inr])), f"{label}: {name} scales"
    for name, got, ref in (("a", a16_g, a_o), ("c", c16_g, c_o)):
        want = np.minimum(ref, 65504.0).astype(np.float16).astype(np.float64)
        bad = got != want
        if bad.any():
            near = _near_half_midpoint(ref, SCALE_RTOL)
            ulp_ok = np.abs(got - want) <= np.abs(np.spacing(want.astype(np.float16)).astype(np.float64)) * 1.01
            assert np.all(near[bad] & ulp_ok[bad]), f"{label}: stored {name} scales differ away from a midpoint"
    # 3. grid from the GPU's stored scales
    Y = oracle.rotate(np.asarray(x_half, np.float16).astype(np.float64))
    d_o, m_o, _, _ = oracle.quantize(Y, bits, a16_g, c16_g)
    rng = (2 ** bits - 1) * d_o
    assert abs(m_g - m_o) <= GRID_RTOL * rng + 1e-30, f"{label}: grid minimum {m_g} vs {m_o}"
    assert abs(delta_g - d_o) <= GRID_RTOL * d_o, f"{label}: grid step {delta_g} vs {d_o}"
    # 4. codes from the GPU's own metadata
    codes_o, t = oracle.codes_for_grid(Y, bits, a16_g, c16_g, m_g, delta_g)
    diff = codes_o != codes_gpu
    n_diff = int(diff.sum())
    if n_diff:
        frac = t[diff] - np.floor(t[diff])
        assert np.all(np.abs(frac - 0.5) < BOUNDARY), f"{label}: code differs away from a boundary"
        assert np.all(np.abs(codes_o[diff].astype(int) - codes_gpu[diff].astype(int)) == 1)
    assert n_diff <= MAX_CODE_MISMATCH * codes_gpu.size, f"{label}: {n_diff} code mismatches"
    return n_diff


def check_attention(out_gpu: np.ndarray, ref: np.ndarray, label: str = "", tol: float = ATTN_TOL):
    """Per row (head): max abs error <= tol * ||ref||_2. Returns the worst ratio."""
    out_gpu = np.asarray(out_gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(out_gpu)), f"{label}: non-finite output"
    worst = 0.0
    for h in range(ref.shape[0]):
        nrm = np.linalg.norm(ref[h])
        err = np.abs(out_gpu[h] - ref[h]).max()
        ratio = err / nrm if nrm > 0 else err
        worst = max(worst, ratio)
        assert err <= tol * nrm + 1e-7, f"{label}: head {h}: max err {err:.3e} vs ||o|| {nrm:.3e}"
    return worst
