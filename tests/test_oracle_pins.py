"""Pins of the CPU oracle to things other than itself.

Each ``check_*`` function asserts one property that the pages or the
mathematics fix: element-format tables, brute-force rounding by table search,
closed forms, invariants and exact brute-force GEMMs.  The planted-mistake
tests at the bottom run some of these checks against deliberately broken
copies of oracle functions and expect them to fail, so a plausible slip in
the oracle (a dropped term, a wrong sign or index, a transposed operand)
would not go unnoticed.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import iq_oracle as O
from fp4_fp8_quant_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "element_formats.txt")


# ----------------------------------------------------------------- formats

def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                fmt, code, val = line.split()
                rows.append((fmt, int(code, 16), float(val)))
    return rows


def test_element_format_tables_match_spec_values():
    e4 = O.e4m3_value_table()
    e2 = O.e2m1_value_table()
    for fmt, code, val in _golden_rows():
        got = {"e4m3": lambda c: e4[c], "e2m1": lambda c: e2[c],
               "ue8m0": lambda c: float(O.decode_ue8m0(np.array([c]))[0])}[fmt](code)
        if math.isnan(val):
            assert math.isnan(got), (fmt, hex(code))
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), (fmt, hex(code), got, val)
    # exactly two NaN codes, no infinities, and the finite positive codes increase
    assert np.isnan(e4).sum() == 2 and not np.isinf(e4).any()
    assert np.all(np.diff(e4[:0x7F]) > 0)


def _nearest_even_code(v, table, n_pos, sign_bit):
    """Round by table search: the nearest positive grid value to |v|, ties to
    the even code (even mantissa bit), saturated at the largest value."""
    a = np.minimum(np.abs(v), table[n_pos - 1])
    pos = table[:n_pos]
    d = np.abs(a[:, None] - pos[None, :])
    dmin = d.min(axis=1, keepdims=True)
    cand = d == dmin
    codes = np.arange(n_pos)
    # among tied candidates take the even code
    even_pick = np.where(cand & (codes[None, :] % 2 == 0), codes[None, :], 10 ** 6).min(axis=1)
    any_pick = np.where(cand, codes[None, :], 10 ** 6).min(axis=1)
    pick = np.where(cand.sum(axis=1) > 1, even_pick, any_pick)
    return pick | (np.signbit(v).astype(np.int64) * sign_bit)


def check_e4m3_rounding_exhaustive():
    # every finite BF16 pattern, shifted across the E4M3 range (subnormals,
    # normals, the top binade) and clipped to the saturation bound
    bits = np.arange(65536, dtype=np.uint32)
    v0 = O.bf16_bits_to_f64(bits.astype(np.uint16))
    v0 = v0[np.isfinite(v0)]
    table = O.e4m3_value_table()
    for shift in (-130, -12, -6, 0, 4, 8):
        v = np.ldexp(v0, 0) * 2.0 ** shift
        v = v[np.abs(v) <= 448.0]
        for chunk in np.array_split(v, 16):
            want = _nearest_even_code(chunk, table, 127, 0x80)
            got = O.round_to_e4m3_codes(chunk).astype(np.int64)
            assert np.array_equal(got, want), (shift, chunk[got != want][:5])


def test_e4m3_rounding_matches_table_search():
    check_e4m3_rounding_exhaustive()


def check_e2m1_rounding_dense():
    table = O.e2m1_value_table()
    grid = table[:8]
    mids = (grid[1:] + grid[:-1]) / 2
    pts = np.concatenate([np.linspace(-6, 6, 200001), mids, -mids,
                          np.nextafter(mids, 0), np.nextafter(mids, 10), grid, -grid, [-0.0]])
    want = _nearest_even_code(pts, table, 8, 0x8)
    got = O.round_to_e2m1_codes(pts).astype(np.int64)
    assert np.array_equal(got, want), pts[got != want][:8]
    # the ties spelled out: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    assert np.array_equal(O.decode_e2m1(O.round_to_e2m1_codes(ties)), [0, 1, 1, 2, 2, 4, 4])


def test_e2m1_rounding_matches_table_search():
    check_e2m1_rounding_dense()


def test_signed_zero_is_kept():
    assert O.round_to_e4m3_codes(np.array([-0.0, -1e-6]))[0] == 0x80
    assert O.round_to_e4m3_codes(np.array([-1e-6]))[0] == 0x80
    assert O.round_to_e2m1_codes(np.array([-0.0, -0.2])).tolist() == [0x8, 0x8]


def check_ue8m0_exponent_bruteforce():
    rng = np.random.default_rng(7)
    for qmax in (448.0, 6.0):
        a = np.concatenate([
            np.exp(rng.uniform(np.log(1e-8), np.log(1e8), 4000)),
            qmax * np.ldexp(1.0, np.arange(-30, 30)),            # exact boundaries
            np.nextafter(qmax * np.ldexp(1.0, np.arange(-30, 30)), np.inf),
            [0.0, 1e-7, 0.99e-4, 1e-4, 1.01e-4]])
        e = O.ue8m0_exponent(a, qmax)
        for ai, ei in zip(a, e):
            af = max(ai, O.AMAX_FLOOR)
            k = -200
            while qmax * 2.0 ** k < af:
                k += 1
            assert ei == k, (qmax, ai, ei, k)


def test_ue8m0_exponent_is_smallest_power_covering_amax():
    check_ue8m0_exponent_bruteforce()


# ------------------------------------------------------- FP8 1x128 quantizer

def check_fp8_quantizer_invariants(M=64, K=1536, seed=11):
    bits = W.quant_blocks_input(M, K, seed=seed, p_large=0.05, p_zero=0.05, p_tiny=0.05)
    x = O.bf16_bits_to_f64(bits)
    codes, sb = O.quantize_fp8_1x128(x)
    e = sb.astype(np.int64) - 127
    xb = x.reshape(M, K // 128, 128)
    amax = np.abs(xb).max(axis=2)
    floored = amax < O.AMAX_FLOOR
    r = amax / np.ldexp(1.0, e)
    assert np.all((r[~floored] > 224) & (r[~floored] <= 448)), "amax/2^e must lie in (224, 448]"
    assert np.all(sb[floored] == 105)
    assert np.all(sb[amax == 0] == 105) and np.all(sb[amax < 1e-6] == 105)
    dec = O.decode_e4m3(codes).reshape(M, K // 128, 128) * np.ldexp(1.0, e)[..., None]
    # decoded within half an E4M3 step of the scaled value
    a = np.abs(xb) / np.ldexp(1.0, e)[..., None]
    _, ex = np.frexp(a)
    step = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3) * np.ldexp(1.0, e)[..., None]
    assert np.all(np.abs(dec - xb) <= step / 2)
    zero_blocks = amax == 0
    assert np.all(codes.reshape(M, K // 128, 128)[zero_blocks] == 0)
    return floored.sum(), zero_blocks.sum()


def test_fp8_quantizer_invariants():
    nf, nz = check_fp8_quantizer_invariants()
    assert nf > 0 and nz > 0   # the sample exercises the floor


def test_packed_scale_layout_by_hand():
    sb = np.arange(1, 31, dtype=np.uint8).reshape(5, 6)   # M=5 rows, 6 blocks
    w = O.pack_scales_m_major(sb).view(np.uint32)
    assert w.shape == (2, 8)
    for m in range(5):
        b = [int(v) for v in sb[m]]
        assert w[0, m] == b[0] | b[1] << 8 | b[2] << 16 | b[3] << 24
        assert w[1, m] == b[4] | b[5] << 8
    assert np.all(w[:, 5:] == 0)


# ---------------------------------------------------------------------- GEMM

def check_gemm_bruteforce(M=2, N=128, K=256, seed=5):
    rng = np.random.default_rng(seed)
    xq = rng.integers(0, 256, (M, K)).astype(np.uint8)
    wq = rng.integers(0, 256, (N, K)).astype(np.uint8)
    xq[(xq & 0x7F) == 0x7F] = 0x01        # no NaN codes
    wq[(wq & 0x7F) == 0x7F] = 0x02
    xs = rng.integers(100, 150, (M, K // 128)).astype(np.uint8)
    ws = rng.integers(100, 150, (N // 128, K // 128)).astype(np.uint8)
    Y = O.block_scaled_gemm(xq, xs, wq, ws)
    e4 = O.e4m3_value_table()
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                sx = Fraction(2) ** (int(xs[m, k // 128]) - 127)
                sw = Fraction(2) ** (int(ws[n // 128, k // 128]) - 127)
                acc += Fraction(e4[xq[m, k]]) * sx * Fraction(e4[wq[n, k]]) * sw
            assert abs(Fraction(Y[m, n]) - acc) <= abs(acc) * Fraction(1, 2 ** 50), (m, n)


def test_gemm_matches_exact_bruteforce():
    check_gemm_bruteforce()


# ---------------------------------------------------------------------- RoPE

def check_rope_closed_form():
    pos = np.array([0, 1, 100, 163839])
    y = np.zeros((4, 2 * 128))
    # unit vector in dim i of head 1: out[i] = cos(p f_i), out[i+32] = sin(p f_i)
    for i in (0, 16, 31):
        yi = y.copy()
        yi[:, 128 + i] = 1.0
        r = O.rope_neox(yi, pos)
        f = 10000.0 ** (-2 * i / 64)
        assert np.allclose(r[:, 128 + i], np.cos(pos * f), atol=1e-14)
        assert np.allclose(r[:, 128 + i + 32], np.sin(pos * f), atol=1e-14)
        mask = np.ones(256, bool)
        mask[[128 + i, 128 + i + 32]] = False
        assert np.all(r[:, mask] == 0)
    # unit vector in dim i+32: out[i] = -sin, out[i+32] = cos
    yj = y.copy()
    yj[:, 128 + 32 + 5] = 1.0
    r = O.rope_neox(yj, pos)
    f = 10000.0 ** (-2 * 5 / 64)
    assert np.allclose(r[:, 128 + 5], -np.sin(pos * f), atol=1e-14)
    assert np.allclose(r[:, 128 + 37], np.cos(pos * f), atol=1e-14)
    # i = 16 has frequency 10000^-0.5 = 0.01: position 100 rotates by one radian
    assert abs(10000.0 ** (-2 * 16 / 64) - 0.01) < 1e-18


def test_rope_closed_form_and_invariants():
    check_rope_closed_form()
    rng = np.random.default_rng(3)
    y = rng.standard_normal((8, 8192))
    assert np.array_equal(O.rope_neox(y, np.zeros(8, np.int64)), y)     # pos 0 = identity
    p1 = rng.integers(0, 80000, 8)
    p2 = rng.integers(0, 80000, 8)
    r = O.rope_neox(y, p1)
    yh, rh = y.reshape(8, 64, 128), r.reshape(8, 64, 128)
    n0 = yh[..., :32] ** 2 + yh[..., 32:64] ** 2
    n1 = rh[..., :32] ** 2 + rh[..., 32:64] ** 2
    assert np.allclose(n0, n1, rtol=1e-14, atol=0)                     # pair norms
    assert np.array_equal(rh[..., 64:], yh[..., 64:])                  # no-rope half
    assert np.allclose(O.rope_neox(r, p2), O.rope_neox(y, p1 + p2), atol=1e-9)   # R(a)R(b)=R(a+b)


# ------------------------------------------------------------------ Hadamard

def check_hadamard():
    import scipy.linalg
    H = O.hadamard_matrix(128)
    assert np.array_equal(H, scipy.linalg.hadamard(128))       # Sylvester construction
    assert np.array_equal(H @ H.T, 128 * np.eye(128))
    e0 = np.zeros((1, 128))
    e0[0, 0] = 1
    assert np.allclose(O.hadamard_heads(e0), 1 / np.sqrt(128), atol=1e-16)
    e5 = np.zeros((1, 128))
    e5[0, 5] = 1
    z5 = O.hadamard_heads(e5)[0]
    assert np.allclose(z5 * np.sqrt(128), [(-1) ** bin(j & 5).count("1") for j in range(128)])


def test_hadamard_properties():
    check_hadamard()
    rng = np.random.default_rng(9)
    r = rng.standard_normal((4, 8192))
    z = O.hadamard_heads(r)
    assert np.allclose(O.hadamard_heads(z), r, atol=1e-13)            # involution after scaling
    assert np.allclose(np.linalg.norm(z.reshape(4, 64, 128), axis=2),
                       np.linalg.norm(r.reshape(4, 64, 128), axis=2), rtol=1e-14)


# ----------------------------------------------------------------------- FP4

def check_fp4_invariants(seed=4):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((16, 8192)) * np.exp(rng.uniform(-12, 12, (16, 1)))
    z[3, :32] = 0.0
    z[4, 32:64] = 1e-6 * rng.standard_normal(32)
    codes, sb = O.quantize_fp4_1x32(z)
    assert codes.max() <= 0xF
    e = sb.astype(np.int64) - 127
    amax = np.abs(z.reshape(16, 256, 32)).max(axis=2)
    floored = amax < O.AMAX_FLOOR
    r = amax / np.ldexp(1.0, e)
    assert np.all((r[~floored] > 3) & (r[~floored] <= 6)), "amax/2^e must lie in (3, 6]"
    assert np.all(sb[floored] == 112) and floored[3, 0] and floored[4, 1]
    assert np.all(codes[3, :32] == 0)
    # decoded within half an E2M1 step (step 0.5 below 2, 1 in [2,4), 2 in [4,6])
    dec = O.decode_e2m1(codes).reshape(16, 256, 32)
    a = np.abs(z.reshape(16, 256, 32)) / np.ldexp(1.0, e)[..., None]
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    assert np.all(np.abs(dec - z.reshape(16, 256, 32) / np.ldexp(1.0, e)[..., None]) <= step / 2)


def test_fp4_invariants_and_packing():
    check_fp4_invariants()
    codes = np.array([[0x1, 0x2, 0xF, 0x8]], np.uint8)
    assert O.pack_fp4(codes).tolist() == [[0x21, 0x8F]]


def _nearest_even_by_search(values: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the grid value nearest to each |value| (ties to the even index),
    by exhaustive comparison; values above the grid saturate to its top."""
    a = np.abs(np.asarray(values, np.float64))[..., None]
    d = np.abs(grid[None, :] - a.reshape(-1, 1))
    best = d.min(axis=1, keepdims=True)
    ties = d == best
    idx = np.where(ties.sum(axis=1) > 1, np.argmax(ties & (np.arange(len(grid)) % 2 == 0), axis=1),
                   np.argmin(d, axis=1))
    return idx.reshape(np.shape(values))


def check_fp4_ocp_rule(seed=5):
    """[OCP] MX v1.0: the shared exponent puts the block's largest magnitude in
    [4, 8) (emax(E2M1) = 2, floor of log2), elements round to nearest-even on
    the E2M1 grid and saturate at 6; floored blocks take floor(log2 1e-4) - 2 =
    -16 (byte 111)."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((8, 1024)) * np.exp(rng.uniform(-10, 10, (8, 1)))
    z[1, :32] = 0.0
    z[2, 32:64] = 31.999                               # amax just below the binade edge 2^5
    z[2, 64:96] = np.ldexp(1.0, 5)                    # amax exactly a power of two
    codes, sb = O.quantize_fp4_1x32_ocp(z)
    e = sb.astype(np.int64) - 127
    amax = np.abs(z.reshape(8, 32, 32)).max(axis=2)
    floored = amax < O.AMAX_FLOOR
    lo, hi = np.ldexp(4.0, e), np.ldexp(8.0, e)
    assert np.all((amax[~floored] >= lo[~floored]) & (amax[~floored] < hi[~floored]))
    assert np.all(sb[floored] == 111) and floored[1, 0]
    assert e[2, 2] == 3 and e[2, 1] == 2
    u = z.reshape(8, 32, 32) / np.ldexp(1.0, e)[..., None]
    grid = O.e2m1_value_table()[:8]
    want = _nearest_even_by_search(u, grid) | (np.signbit(u) << 3)
    assert np.array_equal(codes.reshape(8, 32, 32), want.astype(np.uint8))
    assert np.any((np.abs(u) > 6) & ((codes.reshape(8, 32, 32) & 7) == 7)), "saturation must occur"


def check_nvfp4_rule(seed=6):
    """A14: 1x16 blocks; the scale is the E4M3 value nearest float32(amax / 6)
    (ties to even), 2^-9 when that is zero; codes are the E2M1 values nearest
    float32(z * float32(1 / s)), saturating at 6."""
    rng = np.random.default_rng(seed)
    z = (rng.standard_normal((8, 512)) * np.exp(rng.uniform(-6, 6, (8, 1)))).astype(np.float32)
    z[1, :16] = 0.0
    z[2, 16:32] = np.float32(1e-5)
    codes, sc = O.quantize_nvfp4_1x16(z)
    e4 = O.e4m3_value_table()[:0x7F]
    amax = np.maximum(np.abs(z.reshape(8, 32, 16)).max(axis=2), np.float32(O.AMAX_FLOOR))
    target = (amax / np.float32(6.0)).astype(np.float64)
    want_sc = _nearest_even_by_search(target, e4)
    want_sc = np.where(want_sc == 0, 1, want_sc)
    assert np.array_equal(sc, want_sc.astype(np.uint8))
    assert sc[1, 0] == 1 and sc[2, 1] == 1
    s = e4[sc]
    r = np.float32(1.0) / s.astype(np.float32)
    u = (z.reshape(8, 32, 16) * r[..., None]).astype(np.float32).astype(np.float64)
    want = _nearest_even_by_search(u, O.e2m1_value_table()[:8]) | (np.signbit(u) << 3)
    assert np.array_equal(codes.reshape(8, 32, 16), want.astype(np.uint8))


def test_fp4_output_variants():
    check_fp4_ocp_rule()
    check_nvfp4_rule()
    x, wq, wsf, pos = W.tiny_chain(3)
    shapes = {f: tuple(a.shape for a in O.prepare_q(x, wq, wsf, pos, f)[:2]) for f in O.FP4_FORMATS}
    assert shapes == {"mx": ((3, 4096), (3, 256)), "mx_ocp": ((3, 4096), (3, 256)), "nv": ((3, 4096), (3, 512))}


def test_pins_catch_ocp_ceil_instead_of_floor(monkeypatch):
    good = O.ue8m0_exponent_ocp

    def bad(amax, floor=O.AMAX_FLOOR):   # the ceil rule in the floor rule's place
        return O.ue8m0_exponent(amax, O.E2M1_MAX, floor)
    _expect_fail(check_fp4_ocp_rule, monkeypatch, "ue8m0_exponent_ocp", bad)
    assert good is O.ue8m0_exponent_ocp


def test_pins_catch_nvfp4_scale_error(monkeypatch):
    good = O.nvfp4_block_scale

    def bad(amax_f32):   # amax / 4 instead of amax / 6
        return good(np.asarray(amax_f32, np.float32) * np.float32(1.5))
    _expect_fail(check_nvfp4_rule, monkeypatch, "nvfp4_block_scale", bad)


# ---------------------------------------------------------------- end to end

def test_zero_latent_gives_zero_codes_and_floor_scales():
    x, wq, wsf, pos = W.tiny_chain(M=4)
    x = np.zeros_like(x)
    q, sf, z = O.prepare_q(x, wq, wsf, pos)
    assert np.all(q == 0) and np.all(sf == 112) and np.all(z == 0)
    codes, packed = O.fp8_quant_1x128_ue8m0(x)
    assert np.all(codes == 0)
    assert np.all(packed.view(np.uint32)[:, :4] == 0x69696969)


def check_one_hot_chain(seed=0):
    """A latent row that is one-hot with value 1.0 at column k0 and position 0
    makes Y[n] = W[n, k0] (RoPE is the identity at position 0), so each head
    of the pre-quant Q is the Hadamard transform of one weight column slice."""
    import scipy.linalg
    wq, wsf = W.weights(seed)
    k0 = 300
    x = np.zeros((1, 1536), np.uint16)
    x[0, k0] = 0x3F80                       # BF16 1.0
    q, sf, z = O.prepare_q(x, wq, wsf, np.zeros(1, np.int32))
    wcol = O.e4m3_value_table()[wq[:, k0]] * np.ldexp(1.0, wsf[:, k0 // 128].astype(np.int64) - 127).repeat(128)
    Hs = scipy.linalg.hadamard(128) / np.sqrt(128)
    want = (wcol.reshape(64, 128) @ Hs.T).reshape(-1)
    assert np.allclose(z[0], want, rtol=0, atol=1e-14 * np.abs(want).max())


def test_one_hot_chain_closed_form():
    check_one_hot_chain()


def _rotation_matrix(p):
    """The 128x128 matrix of the NeoX rotation at position p, built entry by
    entry: for i < 32 the plane of dims (i, i + 32) turns by p * 10000^(-i/32);
    dims 64..127 are fixed."""
    R = np.eye(128)
    for i in range(32):
        a = p * 10000.0 ** (-i / 32.0)
        c, s = math.cos(a), math.sin(a)
        R[i, i], R[i, i + 32] = c, -s
        R[i + 32, i], R[i + 32, i + 32] = s, c
    return R


def check_one_hot_chain_at_positions(seed=0):
    """One-hot latent rows at nonzero positions: Y[n] = W[n, k] again, and each
    head of the pre-quant Q must be z = H R(p) w / sqrt(128) -- the rotation
    first, then the transform.  The two do not commute, so a chain that
    applied the Hadamard transform before RoPE would give H-then-R instead."""
    import scipy.linalg
    wq, wsf = W.weights(seed)
    cols = [5, 300, 1535]
    pos = np.array([1, 4631, 163839], np.int32)
    x = np.zeros((3, 1536), np.uint16)
    for r, k in enumerate(cols):
        x[r, k] = 0x3F80                    # BF16 1.0
    _, _, z = O.prepare_q(x, wq, wsf, pos)
    Hs = scipy.linalg.hadamard(128) / np.sqrt(128)
    e4 = O.e4m3_value_table()
    for r, (k, p) in enumerate(zip(cols, pos)):
        wcol = e4[wq[:, k]] * np.ldexp(1.0, wsf[:, k // 128].astype(np.int64) - 127).repeat(128)
        R = _rotation_matrix(float(p))
        want = (Hs @ R @ wcol.reshape(64, 128).T).T.reshape(-1)
        swapped = (R @ Hs @ wcol.reshape(64, 128).T).T.reshape(-1)
        assert np.abs(want - swapped).max() > 1e-3 * np.abs(want).max()   # the orders differ here
        # the angle p * f carries a few float64 ulps of p * f (two routes to
        # f = 10000^(-i/32) may differ by an ulp): allow that, nothing more
        tol = (1e-13 + 8.0 * float(p) * 2.0 ** -53) * np.abs(want).max()
        assert np.allclose(z[r], want, rtol=0, atol=tol), (k, p)


def test_one_hot_chain_closed_form_at_nonzero_positions():
    check_one_hot_chain_at_positions()


# ------------------------------------------------- planted mistakes are caught

def _expect_fail(check, monkeypatch, name, bad):
    monkeypatch.setattr(O, name, bad)
    with pytest.raises(AssertionError):
        check()
    monkeypatch.undo()
    check()   # and the real oracle passes again


def test_pins_catch_rope_sign_flip(monkeypatch):
    good = O.rope_neox

    def bad(Y, pos):
        return good(Y, -np.asarray(pos))
    _expect_fail(check_rope_closed_form, monkeypatch, "rope_neox", bad)


def test_pins_catch_rope_pairing_error(monkeypatch):
    good_inv = O.rope_inv_freq

    def bad_inv():
        return good_inv()[::-1].copy()
    _expect_fail(check_rope_closed_form, monkeypatch, "rope_inv_freq", bad_inv)


def test_pins_catch_weight_scale_index_error(monkeypatch):
    good = O.block_scaled_gemm

    def bad(xq, xs, wq, ws):   # weight block scales taken in reversed K-block order
        return good(xq, xs, wq, ws[:, ::-1].copy())
    _expect_fail(check_one_hot_chain, monkeypatch, "block_scaled_gemm", bad)


def test_pins_catch_transposed_weight(monkeypatch):
    good = O.block_scaled_gemm

    def bad(xq, xs, wq, ws):   # W read as [K, N] column blocks: rows of each 128x128 tile transposed
        N, K = wq.shape
        blk = wq.reshape(N // 128, 128, K // 128, 128).transpose(0, 3, 2, 1).reshape(N, K)
        return good(xq, xs, np.ascontiguousarray(blk), ws)
    _expect_fail(check_one_hot_chain, monkeypatch, "block_scaled_gemm", bad)


def test_pins_catch_interleaved_rope_pairs(monkeypatch):
    def bad(Y, pos):   # GPT-J pairing (2i, 2i+1) instead of NeoX (i, i+32)
        M = Y.shape[0]
        Yh = Y.reshape(M, -1, 128).copy()
        ang = np.asarray(pos, np.float64)[:, None] * O.rope_inv_freq()[None, :]
        c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
        x1, x2 = Yh[:, :, 0:64:2].copy(), Yh[:, :, 1:64:2].copy()
        Yh[:, :, 0:64:2] = x1 * c - x2 * s
        Yh[:, :, 1:64:2] = x2 * c + x1 * s
        return Yh.reshape(M, -1)
    _expect_fail(check_rope_closed_form, monkeypatch, "rope_neox", bad)


def test_pins_catch_dropped_block_scale(monkeypatch):
    def bad(xq, xs, wq, ws):
        X = O.decode_e4m3(xq)
        Wd = O.decode_e4m3(wq)
        return (X @ Wd.T) * O.decode_ue8m0(xs)[:, :1]      # drops the weight scale
    _expect_fail(check_gemm_bruteforce, monkeypatch, "block_scaled_gemm", bad)


def test_pins_catch_floor_rule_error(monkeypatch):
    good = O.ue8m0_exponent

    def bad(amax, qmax, floor=O.AMAX_FLOOR):   # floor(log2) instead of the ceil rule
        return good(amax, qmax, floor) - 1
    _expect_fail(check_ue8m0_exponent_bruteforce, monkeypatch, "ue8m0_exponent", bad)


def test_pins_catch_hadamard_order_error(monkeypatch):
    good = O.hadamard_matrix

    def bad(n=128):   # a row permutation of a Hadamard matrix is still orthogonal
        return good(n)[::-1].copy()
    _expect_fail(check_hadamard, monkeypatch, "hadamard_matrix", bad)


def test_pins_catch_hadamard_before_rope(monkeypatch):
    """A chain that transforms first and rotates second: rope_neox is made to
    apply the Hadamard transform and remember the positions, hadamard_heads
    to apply RoPE with them."""
    good_rope, good_had = O.rope_neox, O.hadamard_heads
    seen = {}

    def bad_rope(Y, pos):
        seen["pos"] = pos
        return good_had(Y)

    def bad_had(R):
        return good_rope(R, seen["pos"])
    monkeypatch.setattr(O, "hadamard_heads", bad_had)
    _expect_fail(check_one_hot_chain_at_positions, monkeypatch, "rope_neox", bad_rope)


def test_pins_catch_rounding_ties_away(monkeypatch):
    def bad(v):
        v = np.asarray(v, np.float64)
        a = np.abs(v)
        step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
        q = np.minimum(np.floor(a / step + 0.5) * step, 6.0)      # ties away from zero
        idx = np.searchsorted(O.e2m1_value_table()[:8], q)
        return (idx | (np.signbit(v) << 3)).astype(np.uint8)
    _expect_fail(check_e2m1_rounding_dense, monkeypatch, "round_to_e2m1_codes", bad)
