"""Pins for the CPU oracle against facts that do not come from the oracle itself.

Each test names what fixes the expected value: a library routine (numpy, scipy),
a closed form, an invariant, brute force on a tiny input, or a number printed on
the KVarN pages (fig1.dev summary; anbeeld.com "KVarN KV Cache: Implementation
and Benchmarks").
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.linalg

import oracle
from quantized_kv_cache_seal_gb300 import workloads

RNG = np.random.default_rng(12345)


# --------------------------------------------------------------------------- fp16
def test_half_to_double_all_patterns_match_numpy():
    """Every binary16 bit pattern decodes to numpy's float16 value (library routine)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_double_to_half_rounds_like_numpy():
    """Round-to-nearest-even matches numpy's float64 -> float16 cast, including ties,
    subnormals and overflow (library routine)."""
    xs = np.concatenate([
        RNG.standard_normal(20000) * 10.0 ** RNG.uniform(-9, 5, 20000),
        # exact ties between neighbouring halves
        (np.arange(1, 2000) + 0.5) * 2.0 ** -10,
        (np.arange(1, 2000) + 0.5) * 2.0 ** -24,
        np.array([65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -25, 2.0 ** -26, 3 * 2.0 ** -26]),
    ])
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.double_to_half(float(x)) for x in xs], np.uint16)
    assert np.array_equal(got, ref)
    assert oracle.double_to_half(1e6, saturate=True) == 0x7BFF
    assert oracle.double_to_half(-1e6, saturate=True) == 0xFBFF


# --------------------------------------------------------------------------- rotation
@pytest.mark.parametrize("d", [2, 4, 8, 16, 32, 64, 128])
def test_hadamard_equals_scipy_sylvester(d):
    """H is scipy's Sylvester Hadamard matrix scaled by 1/sqrt(d) (library routine)."""
    H = oracle.hadamard(d)
    ref = scipy.linalg.hadamard(d).astype(np.float64) / math.sqrt(d)
    assert np.array_equal(H, ref)


def test_hadamard_orthonormal_symmetric():
    H = oracle.hadamard(128)
    assert np.allclose(H @ H.T, np.eye(128), atol=1e-14, rtol=0)
    assert np.array_equal(H, H.T)


def test_rotate_matches_library_matmul_and_round_trips():
    X = RNG.standard_normal((37, 128))
    Y = oracle.rotate(X)
    ref = X @ (scipy.linalg.hadamard(128) / math.sqrt(128))
    assert np.allclose(Y, ref, atol=1e-12, rtol=0)
    assert np.allclose(oracle.rotate(Y), X, atol=1e-12, rtol=0)


def test_query_key_product_invariant_under_joint_rotation():
    """anbeeld.com section 1: rotating q by the same matrix leaves QK unchanged."""
    q = RNG.standard_normal((4, 128))
    k = RNG.standard_normal((50, 128))
    assert np.allclose(oracle.rotate(q) @ oracle.rotate(k).T, q @ k.T, atol=1e-11, rtol=0)


# --------------------------------------------------------------------------- Sinkhorn
def test_sinkhorn_rank_one_closed_form():
    """|Y_ij| = u_i v_j: one token step then one channel step gives Z = sign(Y),
    a_i = u_i * rms(v) (token axis first) and c_j = v_j / rms(v), all row/column RMS 1."""
    T, d = 128, 128
    u = RNG.lognormal(0, 1, T)
    v = RNG.lognormal(0, 0.5, d)
    sgn = np.where(RNG.random((T, d)) < 0.5, -1.0, 1.0)
    Y = sgn * np.outer(u, v)
    a, c, Z = oracle.sinkhorn(Y, iters=1)
    rv = math.sqrt(np.mean(v ** 2))
    assert np.allclose(a, u * rv, rtol=1e-13, atol=0)
    assert np.allclose(c, v / rv, rtol=1e-13, atol=0)
    assert np.allclose(Z, sgn, atol=1e-13, rtol=0)
    # further iterations leave a balanced matrix unchanged
    a16, c16, Z16 = oracle.sinkhorn(Y, iters=16)
    assert np.allclose(a16, a, rtol=1e-12) and np.allclose(c16, c, rtol=1e-12)


def test_sinkhorn_factorisation_invariant():
    Y = oracle.rotate(workloads.group_matrices(1, 1)[0].astype(np.float64))
    for it in (1, 3, 16):
        a, c, Z = oracle.sinkhorn(Y, iters=it)
        assert np.allclose(a[:, None] * Z * c[None, :], Y, rtol=1e-12, atol=1e-12)


def test_sinkhorn_converges_to_unit_rms():
    """Column RMS is exactly 1 after every channel step; the row deviation shrinks and
    is small after the 16 iterations the method uses (anbeeld.com section 1)."""
    Y = oracle.rotate(workloads.group_matrices(2, 1)[0].astype(np.float64))
    a, c, Z, rd, cd = oracle.sinkhorn(Y, iters=16, trace=True)
    assert np.all(cd < 1e-12)
    assert np.all(np.diff(rd) <= 1e-15)
    assert rd[0] > 1e-2 and rd[-1] < 1e-3


def test_sinkhorn_matches_independent_matrix_balancing():
    """The scale vectors equal Sinkhorn-Knopp balancing of A = Y*Y written in the
    matrix-vector form (a^2 = A u / d with u = 1/c^2; c^2 = A^T v / T with v = 1/a^2),
    a different algorithm that never forms the rescaled matrix."""
    Y = oracle.rotate(workloads.group_matrices(3, 1, spike_frac=0.05)[0].astype(np.float64))
    A = Y * Y
    T, d = A.shape
    a2 = np.ones(T)
    c2 = np.ones(d)
    for _ in range(16):
        a2_new = (A @ (1.0 / c2)) / d
        a2 = np.where(a2_new > 0, a2_new, 1.0)
        c2_new = (A.T @ (1.0 / a2)) / T
        c2 = np.where(c2_new > 0, c2_new, 1.0)
    a, c, _ = oracle.sinkhorn(Y, iters=16)
    assert np.allclose(a, np.sqrt(a2), rtol=1e-10, atol=0)
    assert np.allclose(c, np.sqrt(c2), rtol=1e-10, atol=0)


def test_sinkhorn_zero_rows_and_columns_keep_unit_factor():
    Y = np.zeros((8, 8))
    Y[:4, :4] = RNG.standard_normal((4, 4))
    a, c, Z = oracle.sinkhorn(Y, iters=16)
    assert np.all(a[4:] == 1.0) and np.all(c[4:] == 1.0)
    assert np.all(np.isfinite(Z))


def test_seal_scale_equivariance_power_of_two():
    """x -> 2^k x multiplies the token scales by 2^k and leaves the channel scales,
    the grid and every code bit-identical."""
    x = workloads.group_matrices(4, 1)[0]
    r1 = oracle.seal(x, 2, 0)
    r2 = oracle.seal((x.astype(np.float32) * 4).astype(np.float16), 2, 0)
    d1, m1, a1, c1 = oracle.read_header(r1)
    d2, m2, a2, c2 = oracle.read_header(r2)
    assert np.array_equal(a2, 4 * a1) and np.array_equal(c1, c2)
    assert d1 == d2 and m1 == m2
    h = oracle.header_bytes()
    assert np.array_equal(r1[h:], r2[h:])


# --------------------------------------------------------------------------- quantisation
def test_rtn_ties_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "rtn_ties.json")))
    Y = np.array(g["Y"])
    delta, m, codes, t = oracle.quantize(Y, g["bits"], np.ones(Y.shape[0]), np.ones(Y.shape[1]))
    assert delta == g["delta"] and m == g["m"]
    assert codes.tolist() == g["codes"]


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_quantisation_half_step_bound_and_brute_force(bits):
    """Every normalised value lies within delta/2 of its grid point, the extreme
    codes 0 and L are used, and the code equals the nearest of all 2^b grid points
    found by exhaustive search."""
    x = workloads.group_matrices(10 + bits, 1)[0]
    rec = oracle.seal(x, bits, 0)
    delta, m, a16, c16 = oracle.read_header(rec)
    Y = oracle.rotate(x.astype(np.float64))
    Zp = Y / np.outer(a16, c16)
    codes = oracle.unpack(rec[oracle.header_bytes():], bits, 0)
    L = 2 ** bits - 1
    err = np.abs(Zp - (m + delta * codes))
    assert err.max() <= delta / 2 * (1 + 1e-9)
    assert codes.min() == 0 and codes.max() == L
    grid = m + delta * np.arange(L + 1)
    nearest = np.argmin(np.abs(Zp[..., None] - grid), axis=-1)
    dist_own = np.abs(Zp - grid[codes])
    dist_best = np.abs(Zp - grid[nearest])
    assert np.all(dist_own <= dist_best + 1e-12 * delta)


def test_codes_for_grid_hand_worked_golden(golden_dir):
    """Codes for a grid that is not the matrix's own: clamping at both ends, ties to
    even, a zero scale product, token scales per row and channel scales per column
    (hand-worked values in tests/golden/codes_for_grid.json)."""
    g = json.load(open(os.path.join(golden_dir, "codes_for_grid.json")))
    codes, t = oracle.codes_for_grid(np.array(g["Y"]), g["bits"], np.array(g["a16"]), np.array(g["c16"]),
                                     g["m"], g["delta"])
    assert t.tolist() == g["t"]
    assert codes.tolist() == g["codes"]


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 7, 8])
def test_codes_for_grid_reproduces_quantize_on_its_own_grid(bits):
    """Given the stored scales and the grid that kvo_quantize chose, the per-grid
    re-derivation returns exactly kvo_quantize's codes and t (several seeds, K- and
    V-like matrices, T != d so that a row/column swap of the scales cannot pass)."""
    for seed in range(3):
        x = workloads.group_matrices(40 + 7 * bits + seed, 1)[0]
        Y = oracle.rotate(x.astype(np.float64))[:96]  # 96 tokens x 128 channels
        rng = np.random.default_rng(seed)
        a16 = rng.lognormal(0.0, 0.7, Y.shape[0]).astype(np.float16).astype(np.float64)
        c16 = rng.lognormal(0.0, 0.5, Y.shape[1]).astype(np.float16).astype(np.float64)
        delta, m, codes_q, t_q = oracle.quantize(Y, bits, a16, c16)
        codes_g, t_g = oracle.codes_for_grid(Y, bits, a16, c16, m, delta)
        assert np.array_equal(t_g, t_q)
        assert np.array_equal(codes_g, codes_q)


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_codes_for_grid_is_the_nearest_clamped_grid_point(bits):
    """Brute force: on a grid narrower than the data (values below m and above
    m + L delta), each code is the nearest of the 2^b grid points m + q delta, found by
    exhaustive search over q; values off the grid take code 0 or L."""
    rng = np.random.default_rng(100 + bits)
    T, d = 24, 40
    a16 = rng.lognormal(0.0, 0.5, T).astype(np.float16).astype(np.float64)
    c16 = rng.lognormal(0.0, 0.5, d).astype(np.float16).astype(np.float64)
    Z = rng.uniform(-1.5, 1.5, (T, d))
    Y = Z * np.outer(a16, c16)
    L = 2 ** bits - 1
    m = float(np.float32(-1.0))
    delta = float(np.float32(2.0 / L))  # grid spans [-1, 1]; the data spans [-1.5, 1.5]
    codes, t = oracle.codes_for_grid(Y, bits, a16, c16, m, delta)
    z = Y / np.outer(a16, c16)
    grid = m + delta * np.arange(L + 1)
    nearest = np.argmin(np.abs(z[..., None] - grid), axis=-1)
    assert np.array_equal(codes, nearest)
    assert np.all(codes[z < m] == 0) and np.all(codes[z > m + L * delta] == L)
    assert (z < m).any() and (z > m + L * delta).any()


def test_tiny_seal_brute_force():
    """T=4, d=4: the seal equals a step-by-step restatement using numpy and scipy
    (library Hadamard, float16 casts, explicit loops), independent of the C code."""
    x = workloads.tiny_matrix(5, 4, 4)
    bits = 2
    X = x.astype(np.float64)
    Y = X @ (scipy.linalg.hadamard(4) / 2.0)
    a = np.ones(4)
    c = np.ones(4)
    Z = Y.copy()
    for _ in range(16):
        r = np.sqrt((Z ** 2).mean(axis=1))
        r[r == 0] = 1
        Z /= r[:, None]
        a *= r
        g = np.sqrt((Z ** 2).mean(axis=0))
        g[g == 0] = 1
        Z /= g[None, :]
        c *= g
    a16 = a.astype(np.float16).astype(np.float64)
    c16 = c.astype(np.float16).astype(np.float64)
    Zp = Y / np.outer(a16, c16)
    m32 = np.float32(Zp.min())
    d32 = np.float32((Zp.max() - Zp.min()) / 3)
    best = np.empty((4, 4), np.uint8)
    for i in range(4):
        for j in range(4):
            cand = [abs(Zp[i, j] - (float(m32) + float(d32) * q)) for q in range(4)]
            best[i, j] = int(np.argmin(cand))
    buf = oracle.seal(x, bits, 0)  # the oracle with general T and d
    delta, m, ga, gc = oracle.read_header(buf, 4, 4)
    assert np.array_equal(ga, a16) and np.array_equal(gc, c16)
    assert delta == float(d32) and m == float(m32)
    codes = oracle.unpack(buf[oracle.header_bytes(4, 4):], bits, 0, 4, 4)
    assert np.array_equal(codes, best)


# --------------------------------------------------------------------------- packing
def test_packing_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "pack_examples.json")))
    for case in g["cases"]:
        codes = np.array(case["codes"], np.uint8)
        payload = oracle.pack(codes, case["bits"], case["side"])
        assert payload.tobytes().hex() == case["payload_hex"], case["name"]
        back = oracle.unpack(payload, case["bits"], case["side"], case["T"], case["d"])
        assert np.array_equal(back, codes), case["name"]


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("side", [0, 1])
def test_packing_matches_numpy_packbits(bits, side):
    """The payload equals numpy.packbits (little bit order) of the code stream's bits,
    K in token-major and V in channel-major order (library routine)."""
    T, d = 128, 128
    codes = RNG.integers(0, 2 ** bits, size=(T, d)).astype(np.uint8)
    stream = codes.reshape(-1) if side == 0 else codes.T.reshape(-1)
    bitplanes = ((stream[:, None] >> np.arange(bits)[None, :]) & 1).astype(np.uint8).reshape(-1)
    ref = np.packbits(bitplanes, bitorder="little")
    pad = (-ref.size) % 4
    ref = np.concatenate([ref, np.zeros(pad, np.uint8)])
    got = oracle.pack(codes, bits, side)
    assert np.array_equal(got, ref)
    assert np.array_equal(oracle.unpack(got, bits, side), codes)


def test_record_layout_and_bits_per_element(golden_dir):
    """Record = 528 header bytes + 2048*b code bytes; body bits/element = b + 0.2578,
    which at two bits rounds to the 2.3 printed by the fig1.dev summary."""
    for b in (2, 3, 4, 8):
        assert oracle.record_bytes(b) == 528 + 2048 * b
        assert oracle.record_bytes(b) % 16 == 0
        assert abs(oracle.bits_per_element(b) - (b + 528 * 8 / 16384)) < 1e-12
    g = json.load(open(os.path.join(golden_dir, "page_numbers.json")))["bits_per_element_2bit"]
    assert abs(oracle.bits_per_element(2) - g["value"]) <= g["printed_precision"]
    x = workloads.group_matrices(6, 1)[0]
    rec, a, c = oracle.seal(x, 2, 1, return_scales=True)
    assert rec[8:16].tolist() == [0] * 8
    delta, m, a16, c16 = oracle.read_header(rec)
    assert np.array_equal(a16, a.astype(np.float16).astype(np.float64))
    assert np.array_equal(c16, c.astype(np.float16).astype(np.float64))
    assert np.float32(delta) == rec[0:4].view(np.float32)[0]


def test_memory_ladder_structure(golden_dir):
    """anbeeld.com sections 4 and 6: the cache total depends on k_bits + v_bits only and
    grows by a fixed amount per bit; the record sizes have the same structure."""
    rows = json.load(open(os.path.join(golden_dir, "page_numbers.json")))[
        "memory_ladder_qwen36_27b_64k_mib"]["rows"]
    per_bit = {(r["mib"] - rows[0]["mib"]) / ((r["k"] + r["v"]) - (rows[0]["k"] + rows[0]["v"]))
               for r in rows[1:] if r["k"] + r["v"] != rows[0]["k"] + rows[0]["v"]}
    assert per_bit == {128.0}
    ours = {(r["k"], r["v"]): oracle.record_bytes(r["k"]) + oracle.record_bytes(r["v"]) for r in rows}
    assert ours[(4, 2)] == ours[(3, 3)]
    steps = {ours[(r["k"], r["v"])] - ours[(3, 3)] - 2048 * (r["k"] + r["v"] - 6) for r in rows}
    assert steps == {0}


# --------------------------------------------------------------------------- dequant
@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("side", [0, 1])
def test_dequant_error_bound_and_frames(bits, side):
    """Rotated-frame dequantisation is within a_i c_j delta / 2 of Y (the half-step
    bound carried through the stored scales); the original frame is that times H."""
    x = workloads.group_matrices(20 + bits, 1)[0]
    rec = oracle.seal(x, bits, side)
    delta, m, a16, c16 = oracle.read_header(rec)
    Y = oracle.rotate(x.astype(np.float64))
    yh = oracle.dequant(rec, bits, side, frame=1)
    bound = np.outer(a16, c16) * delta / 2
    assert np.all(np.abs(yh - Y) <= bound * (1 + 1e-9) + 1e-12)
    xh = oracle.dequant(rec, bits, side, frame=0)
    assert np.allclose(xh, yh @ (scipy.linalg.hadamard(128) / math.sqrt(128)), atol=1e-10, rtol=0)


def test_eight_bit_reconstruction_is_close():
    x = workloads.group_matrices(30, 1)[0]
    xh = oracle.dequant(oracle.seal(x, 8, 0), 8, 0)
    rel = np.linalg.norm(xh - x.astype(np.float64)) / np.linalg.norm(x.astype(np.float64))
    assert rel < 2e-2


# --------------------------------------------------------------------------- attention
def _plain_attention(q, K, V, scale):
    s = scale * (q @ K.T)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    return (p @ V) / p.sum(axis=-1, keepdims=True)


def test_attention_exact_only_equals_softmax_attention():
    q = RNG.standard_normal((4, 128)).astype(np.float16)
    K = RNG.standard_normal((77, 128)).astype(np.float16)
    V = RNG.standard_normal((77, 128)).astype(np.float16)
    scale = 1 / math.sqrt(128)
    out = oracle.attention(q, scale, K[:50], V[:50], np.zeros(0, np.uint8), np.zeros(0, np.uint8),
                           K[50:], V[50:], 2, 2)
    ref = _plain_attention(q.astype(np.float64), K.astype(np.float64), V.astype(np.float64), scale)
    assert np.allclose(out, ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("kb,vb", [(2, 2), (4, 2), (8, 8)])
def test_attention_brute_force_over_dequantised_cache(kb, vb):
    """Rotated-frame attention with one rotation back equals plain softmax attention
    over the fully dequantised, unrotated K/V (anbeeld.com section 1)."""
    src = workloads.TokenSource(7, 0, 1)
    k, v = src.tokens(0, 128 + 256 + 19)
    k = k[:, 0]
    v = v[:, 0]
    q = RNG.standard_normal((4, 128)).astype(np.float16)
    kr = np.stack([oracle.seal(k[128 + 128 * g:256 + 128 * g], kb, 0) for g in range(2)])
    vr = np.stack([oracle.seal(v[128 + 128 * g:256 + 128 * g], vb, 1) for g in range(2)])
    scale = 1 / math.sqrt(128)
    out = oracle.attention(q, scale, k[:128], v[:128], kr, vr, k[384:], v[384:], kb, vb)
    Kd = np.concatenate([k[:128].astype(np.float64)] +
                        [oracle.dequant(kr[g], kb, 0) for g in range(2)] + [k[384:].astype(np.float64)])
    Vd = np.concatenate([v[:128].astype(np.float64)] +
                        [oracle.dequant(vr[g], vb, 1) for g in range(2)] + [v[384:].astype(np.float64)])
    ref = _plain_attention(q.astype(np.float64), Kd, Vd, scale)
    assert np.allclose(out, ref, atol=1e-11, rtol=1e-11)
    if kb == 8:
        exact = _plain_attention(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), scale)
        assert np.abs(out - exact).max() < 0.05 * np.abs(exact).max()


@pytest.mark.parametrize("kb,vb", [(2, 2), (4, 2), (3, 3)])
def test_prefill_attention_reduces_to_decode_attention(kb, vb):
    """Prefill (many-query) attention at the positions where the causal cut falls on a
    region boundary equals the decode-attention oracle (the C restatement) over the
    regions up to that cut: the last query over the whole cache; a query ending sealed
    group g over the sink and groups 0..g; a query inside the sink over the sink up to
    it; a query inside the tail over the sink, every group and the tail up to it."""
    src = workloads.TokenSource(11, 0, 1)
    n = 128 + 128 * 3 + 41
    k, v = src.tokens(0, n)
    k = k[:, 0]
    v = v[:, 0]
    kr = np.stack([oracle.seal(k[128 + 128 * g:256 + 128 * g], kb, 0) for g in range(3)])
    vr = np.stack([oracle.seal(v[128 + 128 * g:256 + 128 * g], vb, 1) for g in range(3)])
    positions = [0, 5, 127, 255, 383, 511, 512, 530, n - 1]
    q = RNG.standard_normal((len(positions), 2, 128)).astype(np.float16)
    scale = 1 / math.sqrt(128)
    out = oracle.prefill_attention(q, positions, scale, k[:128], v[:128], kr, vr, k[512:], v[512:], kb, vb)
    empty = np.zeros(0, np.uint8)
    none = np.zeros((0, 128), np.float16)
    for i, P in enumerate(positions):
        if P < 128:
            ref = oracle.attention(q[i], scale, k[:P + 1], v[:P + 1], empty, empty, none, none, kb, vb)
        elif P < 512:
            assert (P - 127) % 128 == 0
            g = (P - 255) // 128
            ref = oracle.attention(q[i], scale, k[:128], v[:128], kr[:g + 1], vr[:g + 1], none, none, kb, vb)
        else:
            ref = oracle.attention(q[i], scale, k[:128], v[:128], kr, vr, k[512:P + 1], v[512:P + 1], kb, vb)
        assert np.allclose(out[i], ref, atol=1e-11, rtol=1e-11), P


def test_prefill_attention_is_causal_and_matches_cache_helper():
    """Keys after a query's position do not move its output: changing every token from
    the next group boundary on leaves it bit-identical (a sealed record depends on all
    128 tokens of its group, so the boundary, not the position, is the cut). The
    cache-level helper over the last n_q tokens equals the per-head function."""
    src = workloads.TokenSource(12, 0, 2)
    n = 128 + 128 * 2 + 9
    k, v = src.tokens(0, n)
    cache = oracle.OracleCache(2, 2, 2)
    cache.append(0, k, v)
    q = RNG.standard_normal((20, 4, 128)).astype(np.float16)
    scale = 1 / math.sqrt(128)
    out = cache.prefill_attend(0, q, scale)
    k2, v2 = k.copy(), v.copy()
    k2[384:] = -k2[384:]
    v2[384:] = v2[384:] * np.float16(2)
    other = oracle.OracleCache(2, 2, 2)
    other.append(0, k2, v2)
    pos = np.arange(n - 20, n)
    out2 = other.prefill_attend(0, q, scale)
    seen = pos >= 384  # queries at or after the first changed token see it
    assert seen.any() and (~seen).any()
    assert np.array_equal(out[~seen], out2[~seen])
    assert all(not np.array_equal(out[i], out2[i]) for i in np.nonzero(seen)[0])
    q_early = RNG.standard_normal((2, 4, 128)).astype(np.float16)
    for c in (cache, other):
        st = c.seqs[0]
        kr = np.stack([g[1] for g in st["krec"]])
        vr = np.stack([g[1] for g in st["vrec"]])
        tk, tv = c.tail(0)
        c.early = oracle.prefill_attention(q_early[:, 2:], [299, 383], scale, st["sink_k"][:, 1], st["sink_v"][:, 1],
                                           kr, vr, tk[:, 1], tv[:, 1], 2, 2)
    assert np.array_equal(cache.early, other.early)
    # the helper equals the per-head call (KV head 1 holds query heads 2, 3)
    st = cache.seqs[0]
    kr = np.stack([g[1] for g in st["krec"]])
    vr = np.stack([g[1] for g in st["vrec"]])
    tk, tv = cache.tail(0)
    ref = oracle.prefill_attention(q[:, 2:], list(pos), scale, st["sink_k"][:, 1], st["sink_v"][:, 1], kr, vr,
                                   tk[:, 1], tv[:, 1], 2, 2)
    assert np.array_equal(out[:, 2:], ref)


@pytest.mark.parametrize("floor", [0, 1])
def test_prefill_last_query_equals_cache_attend(floor):
    """At the cache level, with and without a tail floor: the newest token's prefill
    query equals the decode-attention oracle over the same cache (the floor only moves
    groups from the records to the exact tail, which both read)."""
    src = workloads.TokenSource(13, 0, 2)
    n = 128 + 128 * 3 + 17
    k, v = src.tokens(0, n)
    cache = oracle.OracleCache(2, 2, 2, tail_floor=floor)
    cache.append(0, k, v)
    q = RNG.standard_normal((3, 4, 128)).astype(np.float16)
    scale = 1 / math.sqrt(128)
    out = cache.prefill_attend(0, q, scale)
    ref = cache.attend(0, q[-1], scale)
    assert np.allclose(out[-1], ref, atol=1e-11, rtol=1e-11)
    assert cache.regions(0)[1] == 3 - floor


# --------------------------------------------------------------------------- regions
def test_cache_regions_and_seal_timing():
    """anbeeld.com 2.1: sink = first 128 tokens; a group seals exactly when its 128th
    token arrives; the tail is the partial newest group and grows 0..127."""
    cache = oracle.OracleCache(1, 2, 2)
    src = workloads.TokenSource(8, 0, 1)
    k, v = src.tokens(0, 128 + 128 * 2 + 5)
    for n in range(1, k.shape[0] + 1):
        cache.append(0, k[n - 1:n], v[n - 1:n])
        ns, ng, nt = cache.regions(0)
        assert ns == min(n, 128)
        assert ng == max(n - 128, 0) // 128
        assert nt == max(n - 128, 0) % 128
    # sink and tail hold the input bits unchanged
    st = cache.seqs[0]
    assert np.array_equal(st["sink_k"][:, 0].view(np.uint16), k[:128, 0].view(np.uint16))
    assert np.array_equal(cache.tail(0)[1][:5, 0].view(np.uint16), v[384:389, 0].view(np.uint16))


@pytest.mark.parametrize("floor", [1, 2])
def test_tail_floor_seal_timing_and_records(floor):
    """anbeeld.com 2.1 (BeeLlama): the exact tail never drops below `floor` full groups,
    i.e. group g seals when group g + floor fills. The tail then holds exactly the input
    tokens of the unsealed positions, and every sealed record equals the one the
    published design (no floor) makes for the same group: a seal depends only on the
    group's own tokens."""
    src = workloads.TokenSource(10, 0, 1)
    n_all = 128 + 128 * (floor + 3) + 7
    k, v = src.tokens(0, n_all)
    fl = oracle.OracleCache(1, 2, 2, tail_floor=floor)
    pub = oracle.OracleCache(1, 2, 2)
    for n in range(1, n_all + 1):
        fl.append(0, k[n - 1:n], v[n - 1:n])
        ns, ng, nt = fl.regions(0)
        body = max(n - 128, 0)
        assert ng == max(body // 128 - floor, 0)
        assert nt == body - 128 * ng
        if body >= 128 * floor:
            assert nt >= 128 * floor
        tk, tv = fl.tail(0)
        assert np.array_equal(tk.view(np.uint16), k[128 + 128 * ng:n].view(np.uint16))
        assert np.array_equal(tv.view(np.uint16), v[128 + 128 * ng:n].view(np.uint16))
    pub.append(0, k, v)
    ng = fl.regions(0)[1]
    assert ng == (n_all - 128) // 128 - floor and ng >= 3
    for g in range(ng):
        assert np.array_equal(fl.seqs[0]["krec"][g], pub.seqs[0]["krec"][g])
        assert np.array_equal(fl.seqs[0]["vrec"][g], pub.seqs[0]["vrec"][g])


def test_streaming_append_equals_bulk_append():
    """Pseudo-decode (fig1.dev 'Practical takeaway'): sealing groups as tokens stream in
    one at a time gives the same records as appending the whole prompt at once."""
    src = workloads.TokenSource(9, 0, 2)
    k, v = src.tokens(0, 128 + 256 + 3)
    a = oracle.OracleCache(2, 4, 2)
    b = oracle.OracleCache(2, 4, 2)
    a.append(0, k, v)
    for t in range(k.shape[0]):
        b.append(0, k[t:t + 1], v[t:t + 1])
    for g in range(2):
        assert np.array_equal(a.seqs[0]["krec"][g], b.seqs[0]["krec"][g])
        assert np.array_equal(a.seqs[0]["vrec"][g], b.seqs[0]["vrec"][g])


def test_rotation_of_fp16_rows_is_exact_before_the_scaling():
    """fp16 inputs are integers times 2^-24, so X * (+-1 Sylvester matrix) is an exact
    integer sum (Python ints here); the oracle's Y must equal that sum divided by
    sqrt(128) with a single rounding, and exact zeros (a constant row) stay zero."""
    x = workloads.tiny_matrix(21, 3, 128, 300.0)
    x[2] = np.float16(1.5)
    ints = (x.astype(np.float64) * 2.0 ** 24).astype(np.int64)
    S = scipy.linalg.hadamard(128).astype(np.int64)
    exact = [[int(sum(int(ints[i, k]) * int(S[k, j]) for k in range(128))) for j in range(128)] for i in range(3)]
    Y = oracle.rotate(x.astype(np.float64))
    for i in range(3):
        for j in range(128):
            ref = exact[i][j] * 2.0 ** -24 / math.sqrt(128)
            assert abs(Y[i, j] - ref) <= abs(ref) * 2.0 ** -52
    assert np.count_nonzero(Y[2]) == 1
