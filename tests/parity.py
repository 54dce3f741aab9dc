"""Comparison rules between the CUDA path and the CPU oracle.

* FP8 quantizer: codes and packed scale words bit-exact (pad words included).
* Pre-quant Q (float32 debug output): |gpu - oracle| <= 1e-4 * RMS of the
  oracle's row (over all 8192 values) for every element.
* FP4 output: the FP4 decisions of both sides are taken on float32 values that
  differ by the GPU's float32 rounding, so they may differ only where the
  oracle's value sits next to a decision boundary:
    - a block's scale byte may differ only next to the scale rule's decision
      boundary, within 1e-4 relative of it: the oracle's floored amax / 6 at a
      power of two (MXFP4, ceil rule), amax at a power of two (MXFP4, OCP
      floor rule), amax / 6 at a rounding midpoint between two E4M3 values
      (NVFP4-style); in such blocks the GPU's codes must be a correct rounding
      of the values under the GPU's own scale (same one-step rule as below)
      and all their elements count as mismatches;
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


_E4M3_POS = O.e4m3_value_table()[:0x7F]
_E4M3_MID = (_E4M3_POS[:-1] + _E4M3_POS[1:]) / 2


def _units(z32, sf, fmt):
    """The value each code encodes in units of its block's scale, computed the
    way the format's rule does (float32 for the NVFP4 product)."""
    if fmt == "nv":
        s = O.decode_e4m3(sf)
        r = (1.0 / s).astype(np.float32)
        return (z32.astype(np.float32) * r[..., None]).astype(np.float32).astype(np.float64), s
    e = sf.astype(np.int64) - 127
    return z32 * np.ldexp(1.0, -e)[..., None], np.ldexp(1.0, e)


def _near_scale_boundary(amax, fmt):
    if fmt == "mx":          # ceil rule: amax / 6 at a power of two
        r = amax / 6.0
        pw = np.ldexp(1.0, np.round(np.log2(np.maximum(r, 1e-300))).astype(np.int64))
        return np.abs(r - pw) <= 1e-4 * pw
    if fmt == "mx_ocp":      # floor rule: amax at a power of two
        pw = np.ldexp(1.0, np.round(np.log2(np.maximum(amax, 1e-300))).astype(np.int64))
        return np.abs(amax - pw) <= 1e-4 * pw
    r = amax / 6.0           # nv: amax / 6 at an E4M3 rounding midpoint
    i = np.clip(np.searchsorted(_E4M3_MID, r), 1, len(_E4M3_MID) - 1)
    d = np.minimum(np.abs(r - _E4M3_MID[i - 1]), np.abs(r - _E4M3_MID[i]))
    return d <= 1e-4 * np.maximum(r, 1e-300)


def _check_codes(gc, oc, u, mask):
    """Codes that differ (where mask) must be one E2M1 step apart at a value
    within 1e-4 relative of the rounding midpoint, or a sign flip of a value
    that rounds to zero (|u| <= 6e-4).  Returns (mismatches, zero flips, worst)."""
    diff = (gc != oc) & mask
    if not diff.any():
        return 0, 0, 0.0
    idx = np.nonzero(diff)
    g, o, uu = gc[idx], oc[idx], u[idx]
    gi, oi = _code_index(g), _code_index(o)
    same_sign = (g >> 3) == (o >> 3)
    step_ok = same_sign & (np.abs(gi - oi) == 1)
    zero_flip = (~same_sign) & (gi == 0) & (oi == 0)
    assert np.all(step_ok | zero_flip), "FP4 code differs by more than one step"
    lo = np.minimum(gi, oi)
    mid = np.where(step_ok, (E2M1_GRID[lo] + E2M1_GRID[np.minimum(lo + 1, 7)]) / 2, 0.0)
    dist = np.where(step_ok, np.abs(np.abs(uu) - mid) / np.maximum(mid, 1e-300), np.abs(uu) / 6.0)
    worst = float(dist.max())
    assert np.all(dist <= 1e-4), f"FP4 code mismatch {worst:.3g} away from a rounding boundary"
    nz = int(zero_flip.sum())
    return int(diff.sum()) - nz, nz, worst


def check_fp4(gpu_q, gpu_sf, ora_q, ora_sf, ora_z, min_equal=0.9999, fmt="mx"):
    """Returns a dict of mismatch statistics; raises AssertionError on a
    violation of the rules in the module docstring.  fmt: the FP4 output
    variant ("mx", "mx_ocp" or "nv"); the scale-decision boundary is the one
    of that variant's rule."""
    gpu_q = np.asarray(gpu_q)
    gpu_sf = np.asarray(gpu_sf)
    M = ora_z.shape[0]
    assert gpu_q.shape == ora_q.shape and gpu_sf.shape == ora_sf.shape
    blk = O.NVFP4_BLOCK if fmt == "nv" else O.FP4_BLOCK
    gc = unpack_fp4(gpu_q).reshape(M, -1, blk)
    oc = unpack_fp4(ora_q).reshape(M, -1, blk)
    z32 = ora_z.astype(np.float32).astype(np.float64).reshape(M, -1, blk)
    amax = np.maximum(np.abs(z32).max(axis=2), O.AMAX_FLOOR)

    # scale bytes: may differ only next to the variant's decision boundary;
    # there the GPU's codes must be a correct rounding under its own scale
    sf_diff = gpu_sf != ora_sf
    bad_sf = sf_diff & ~_near_scale_boundary(amax, fmt)
    assert not bad_sf.any(), f"{int(bad_sf.sum())} FP4 scale bytes differ away from a decision boundary, " \
                             f"first {np.argwhere(bad_sf)[:5].tolist()}"
    n_mis = int(sf_diff.sum()) * blk
    if sf_diff.any():
        u_g, _ = _units(z32, gpu_sf, fmt)
        _check_codes(gc, O.round_to_e2m1_codes(u_g), u_g, np.broadcast_to(sf_diff[..., None], gc.shape))

    # codes in blocks whose scales agree
    u, _ = _units(z32, ora_sf, fmt)
    n_code, n_zero_flip, worst_rel = _check_codes(gc, oc, u, np.broadcast_to(~sf_diff[..., None], gc.shape))
    n_mis += n_code
    total = gc.size
    frac_equal = 1.0 - n_mis / max(total, 1)
    assert frac_equal >= min_equal, f"only {frac_equal:.6f} of FP4 codes equal"
    return {"scale_mismatch_blocks": int(sf_diff.sum()), "code_mismatches": n_code,
            "signed_zero_flips": n_zero_flip,
            "equal_fraction": frac_equal, "worst_boundary_rel": worst_rel}


# ---------------------------------------------------- downstream indexer rules
#
# Logits: |gpu - oracle| <= 2^-16 * S[t, s] for every visible pair, where S is
# the sum of the magnitudes of every term of the score (the oracle's
# indexer_logit_magnitude): the float32 accumulation of the 128-term head dot
# products, the ReLU and the 64-term weighted sum stays within ~200 float32
# roundings of S.
# Top-k: bit-exact against the oracle's selection applied to the GPU's own
# scores (the selection itself is exact); against the oracle's float64 scores
# the chosen sets may differ only at keys whose score is within the logits
# tolerance of the oracle's k-th largest score.

LOGIT_TOL = 2.0 ** -16


def check_logits(gpu, ora, mag, lengths):
    gpu = np.asarray(gpu, np.float64)
    worst = 0.0
    for t in range(ora.shape[0]):
        L = int(min(max(lengths[t], 0), ora.shape[1]))
        if L == 0:
            continue
        err = np.abs(gpu[t, :L] - ora[t, :L])
        bound = LOGIT_TOL * mag[t, :L] + 1e-30
        assert np.all(err <= bound), f"row {t}: logit error {float((err / bound).max()):.3g} x the bound"
        worst = max(worst, float((err / (mag[t, :L] + 1e-30)).max()))
    return worst


def check_topk_vs_oracle_scores(gpu_idx, ora_scores, mag, lengths, k):
    """Chosen sets equal except at keys within the logits tolerance of the
    oracle's k-th largest score.  Returns the number of rows whose sets differ."""
    rows_differing = 0
    for t in range(ora_scores.shape[0]):
        L = int(min(max(lengths[t], 0), ora_scores.shape[1]))
        g = set(int(i) for i in gpu_idx[t] if i >= 0)
        assert len(g) == min(L, k) and all(i < L for i in g), f"row {t}: bad selection size or index"
        if L <= k:
            assert g == set(range(L))
            continue
        s = ora_scores[t, :L]
        kth = np.sort(s)[::-1][k - 1]
        near = np.abs(s - kth) <= 2 * LOGIT_TOL * mag[t, :L] + 1e-30
        must = set(np.nonzero((s > kth) & ~near)[0].tolist())
        must_not = set(np.nonzero((s < kth) & ~near)[0].tolist())
        assert must <= g, f"row {t}: {len(must - g)} keys clearly above the threshold not chosen"
        assert not (must_not & g), f"row {t}: {len(must_not & g)} keys clearly below the threshold chosen"
        ora_set = set(np.sort(np.lexsort((np.arange(L), -s))[:k]).tolist())
        rows_differing += int(g != ora_set)
    return rows_differing
