"""Comparison rules between the CUDA path and the CPU oracle.

* FP8 quantizer: codes and packed scale words bit-exact (pad words included).
* Pre-quant Q (float32 debug output): |gpu - oracle| <= 1e-4 * RMS of the
  oracle's row (over all 8192 values) for every element.
* FP4 output: the FP4 decisions of both sides are taken on float32 values that
  differ by the GPU's float32 rounding, so they may differ only where the
  oracle's value sits next to a decision boundary:
    - a block's scale byte may differ only where the oracle's floored amax / 6
      is within 1e-4 relative of a power of two; such blocks are compared by
      decoded value (within one step of the finer of the two scales) and all
      their elements count as mismatches;
    - in blocks with equal scales, a code may differ only by one step on the
      E2M1 grid, at an oracle value u = z * 2^-e within 1e-4 relative of the
      rounding midpoint between the two codes; a sign difference of a value
      that rounds to zero counts as a step across the zero boundary and needs
      |u| <= 6e-4 (1e-4 of the FP4 range);
    - at least 99.99% of all elements are equal, where +0 and -0 (codes 0x0
      and 0x8, the same value) count as equal: the sign of an exact zero
      depends on the order of the additions that produced it.
"""

from __future__ import annotations

import numpy as np

from oracle import iq_oracle as O

E2M1_GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)


def unpack_fp4(q: np.ndarray) -> np.ndarray:
    """[M, D/2] packed bytes -> [M, D] codes (low nibble = even element)."""
    out = np.empty((q.shape[0], q.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = q & 0xF
    out[:, 1::2] = q >> 4
    return out


def check_fp8(gpu_codes, gpu_words, ora_codes, ora_words):
    gpu_codes = np.asarray(gpu_codes)
    assert gpu_codes.shape == ora_codes.shape
    bad = np.argwhere(gpu_codes != ora_codes)
    assert bad.size == 0, f"{len(bad)} FP8 code mismatches, first {bad[:5].tolist()}"
    gw = np.asarray(gpu_words).view(np.uint32)
    ow = np.asarray(ora_words).view(np.uint32)
    assert gw.shape == ow.shape, (gw.shape, ow.shape)
    badw = np.argwhere(gw != ow)
    assert badw.size == 0, f"{len(badw)} scale-word mismatches, first {badw[:5].tolist()}"


def check_prequant(gpu_z, ora_z, tol=1e-4):
    gpu_z = np.asarray(gpu_z, dtype=np.float64)
    rms = np.sqrt(np.mean(ora_z ** 2, axis=1, keepdims=True))
    err = np.abs(gpu_z - ora_z)
    worst = float((err / np.maximum(rms, 1e-300)).max()) if err.size else 0.0
    assert np.all(err <= tol * rms), f"pre-quant Q error {worst:.3g} x row RMS exceeds {tol}"
    return worst


def _code_index(c):
    return (c & 0x7).astype(np.int64)


def check_fp4(gpu_q, gpu_sf, ora_q, ora_sf, ora_z, min_equal=0.9999):
    """Returns a dict of mismatch statistics; raises AssertionError on a
    violation of the rules in the module docstring."""
    gpu_q = np.asarray(gpu_q)
    gpu_sf = np.asarray(gpu_sf)
    M = ora_z.shape[0]
    assert gpu_q.shape == ora_q.shape and gpu_sf.shape == ora_sf.shape
    gc = unpack_fp4(gpu_q).reshape(M, -1, 32)
    oc = unpack_fp4(ora_q).reshape(M, -1, 32)
    z32 = ora_z.astype(np.float32).astype(np.float64).reshape(M, -1, 32)
    amax = np.maximum(np.abs(z32).max(axis=2), O.AMAX_FLOOR)

    # scale bytes
    sf_diff = gpu_sf != ora_sf
    e_o = ora_sf.astype(np.int64) - 127
    e_g = gpu_sf.astype(np.int64) - 127
    near_pow2 = np.zeros_like(sf_diff)
    r = amax / 6.0
    pw = np.ldexp(1.0, np.round(np.log2(r)).astype(np.int64))
    near_pow2 = np.abs(r - pw) <= 1e-4 * pw
    bad_sf = sf_diff & ~near_pow2
    assert not bad_sf.any(), f"{int(bad_sf.sum())} FP4 scale bytes differ away from a power-of-two boundary, " \
                             f"first {np.argwhere(bad_sf)[:5].tolist()}"
    n_mis = 0
    if sf_diff.any():
        idx = np.argwhere(sf_diff)
        for m, b in idx:
            dg = O.decode_e2m1(gc[m, b]) * np.ldexp(1.0, e_g[m, b])
            do = O.decode_e2m1(oc[m, b]) * np.ldexp(1.0, e_o[m, b])
            ef = min(e_g[m, b], e_o[m, b])
            u = np.abs(z32[m, b]) * np.ldexp(1.0, -ef)
            step = np.where(u < 2, 0.5, np.where(u < 4, 1.0, 2.0)) * np.ldexp(1.0, ef)
            assert np.all(np.abs(dg - do) <= step + 1e-300), f"block ({m},{b}) decoded values too far apart"
        n_mis += int(sf_diff.sum()) * 32

    # codes in blocks whose scales agree
    same = ~sf_diff
    diff = (gc != oc) & same[..., None]
    n_code = int(diff.sum())
    n_zero_flip = 0
    worst_rel = 0.0
    if n_code:
        mi, bi, ji = np.nonzero(diff)
        g = gc[mi, bi, ji]
        o = oc[mi, bi, ji]
        u = z32[mi, bi, ji] * np.ldexp(1.0, -e_o[mi, bi])
        gi, oi = _code_index(g), _code_index(o)
        gs, os_ = g >> 3, o >> 3
        same_sign = gs == os_
        step_ok = same_sign & (np.abs(gi - oi) == 1)
        zero_flip = (~same_sign) & (gi == 0) & (oi == 0)
        assert np.all(step_ok | zero_flip), "FP4 code differs by more than one step"
        lo = np.minimum(gi, oi)
        mid = np.where(step_ok, (E2M1_GRID[lo] + E2M1_GRID[np.minimum(lo + 1, 7)]) / 2, 0.0)
        dist = np.where(step_ok, np.abs(np.abs(u) - mid) / np.maximum(mid, 1e-300), np.abs(u) / 6.0)
        worst_rel = float(dist.max())
        assert np.all(dist <= 1e-4), f"FP4 code mismatch {worst_rel:.3g} away from a rounding boundary"
        n_zero_flip = int(zero_flip.sum())
        n_code -= int(zero_flip.sum())
    n_mis += n_code
    total = gc.size
    frac_equal = 1.0 - n_mis / max(total, 1)
    assert frac_equal >= min_equal, f"only {frac_equal:.6f} of FP4 codes equal"
    return {"scale_mismatch_blocks": int(sf_diff.sum()), "code_mismatches": n_code,
            "signed_zero_flips": n_zero_flip,
            "equal_fraction": frac_equal, "worst_boundary_rel": worst_rel}
