"""Pins of the oracle's downstream consumer (indexer logits and top-k) to
things other than itself: an exact brute force over explicit loops that
decodes every nibble from the element-format table in tests/golden, closed
forms for ReLU and the per-head weights, and top-k against a brute-force sort.
The planted-mistake tests break the oracle on purpose (swapped nibbles, no
ReLU, ties to the larger index, keys visible one position too far) and expect
a pin to fail."""

import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import iq_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "element_formats.txt")


def _e2m1_from_golden():
    """The 16 E2M1 values: the golden file lists codes 0..7 and some negative
    codes; bit 3 is the sign (checked against the listed negatives)."""
    listed = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                fmt, code, val = line.split()
                if fmt == "e2m1":
                    listed[int(code, 16)] = Fraction(float(val))
    vals = {c: (-1 if c & 8 else 1) * listed[c & 7] for c in range(16)}
    assert all(vals[c] == v for c, v in listed.items()) and len(listed) >= 8
    return vals


def _inputs(M, N, seed):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 256, (M, 4096)).astype(np.uint8)
    qs = rng.integers(118, 132, (M, 256)).astype(np.uint8)
    k = rng.integers(0, 256, (N, 64)).astype(np.uint8)
    ks = rng.integers(118, 132, (N, 4)).astype(np.uint8)
    w = (rng.standard_normal((M, 64)) / 8).astype(np.float32)
    return q, qs, k, ks, w


def check_logits_bruteforce(seed=3):
    """Two queries, three keys, every head: explicit loops, exact fractions."""
    e2 = _e2m1_from_golden()
    M, N = 2, 3
    q, qs, k, ks, w = _inputs(M, N, seed)
    L = np.array([3, 2])
    got = O.indexer_logits(q, qs, k, ks, w, L)

    def elem(packed_row, sf_row, d):
        byte = int(packed_row[d // 2])
        code = byte & 0xF if d % 2 == 0 else byte >> 4
        return e2[code] * Fraction(2) ** (int(sf_row[d // 32]) - 127)

    for t in range(M):
        for s in range(N):
            if s >= L[t]:
                assert got[t, s] == -np.inf
                continue
            total = Fraction(0)
            for h in range(64):
                dot = Fraction(0)
                for d in range(128):
                    dot += elem(q[t, 64 * h:64 * h + 64], qs[t, 4 * h:4 * h + 4], d) * elem(k[s], ks[s], d)
                total += Fraction(float(w[t, h])) * max(dot, Fraction(0))
            assert abs(Fraction(got[t, s]) - total) <= abs(total) * Fraction(1, 2 ** 48) + Fraction(1, 2 ** 200), (t, s)


def test_logits_match_exact_bruteforce():
    check_logits_bruteforce()


def check_relu_and_weights(seed=4):
    """Closed forms: a key equal to one head's query (same codes and scales)
    scores w * |q|^2 on that head when the other weights are 0; the negated
    key (every sign bit flipped) scores 0; the score is linear in w."""
    q, qs, k, ks, w = _inputs(1, 2, seed)
    h = 7
    k[0] = q[0, 64 * h:64 * h + 64]
    ks[0] = qs[0, 4 * h:4 * h + 4]
    k[1] = k[0] ^ 0x88
    ks[1] = ks[0]
    w1 = np.zeros((1, 64), np.float32)
    w1[0, h] = 0.5
    got = O.indexer_logits(q, qs, k, ks, w1, np.array([2]))
    qh = O.decode_mxfp4(q[:, 64 * h:64 * h + 64], qs[:, 4 * h:4 * h + 4])[0]
    assert got[0, 0] == 0.5 * float(np.dot(qh, qh)) and got[0, 0] > 0
    assert got[0, 1] == 0.0
    wa, wb = w.copy(), (np.arange(64, dtype=np.float32) / 64)[None, :]
    sa = O.indexer_logits(q, qs, k, ks, wa, np.array([2]))
    sb = O.indexer_logits(q, qs, k, ks, wb, np.array([2]))
    sab = O.indexer_logits(q, qs, k, ks, wa.astype(np.float64) + wb.astype(np.float64), np.array([2]))
    assert np.allclose(sab, sa + sb, rtol=1e-12, atol=1e-9)


def test_relu_and_weights_closed_forms():
    check_relu_and_weights()


def check_topk_against_sort(seed=5):
    """Integer scores with many ties: the selection equals a brute-force sort
    by (score descending, index ascending), taken k at a time, then sorted by
    index; rows with fewer visible keys than k are padded with -1."""
    rng = np.random.default_rng(seed)
    M, N, k = 6, 40, 9
    scores = rng.integers(-3, 4, (M, N)).astype(np.float64)
    L = np.array([40, 9, 3, 0, 17, 40])
    got = O.indexer_topk(scores, L, k)
    for t in range(M):
        vis = list(range(L[t]))
        best = sorted(vis, key=lambda s: (-scores[t, s], s))[:k]
        want = sorted(best) + [-1] * (k - len(best))
        assert got[t].tolist() == want, t


def test_topk_matches_sort():
    check_topk_against_sort()


def _expect_fail(check, monkeypatch, name, bad):
    monkeypatch.setattr(O, name, bad)
    with pytest.raises(AssertionError):
        check()
    monkeypatch.undo()
    check()


def check_mxfp4_layout():
    """The decoder reads the layout iq_prepare_q writes (A10/A18): element
    2i in the low nibble of byte i, scale byte b for elements 32b..32b+31.  A
    permutation applied to both Q and K would leave every dot product as it
    is, so the layout is pinned against hand-written bytes and against the
    (separately pinned) packer."""
    packed = np.zeros((1, 64), np.uint8)
    packed[0, 0] = 0x21          # elements 0, 1 = codes 1, 2 = 0.5, 1.0
    packed[0, 17] = 0x9F         # elements 34, 35 = codes 0xF, 0x9 = -6, -0.5
    sf = np.array([[127, 129, 120, 127]], np.uint8)
    v = O.decode_mxfp4(packed, sf)
    want = np.zeros(128)
    want[0], want[1] = 0.5, 1.0
    want[34], want[35] = -6.0 * 4, -0.5 * 4
    assert np.array_equal(v[0], want)
    codes = np.random.default_rng(9).integers(0, 16, (3, 128)).astype(np.uint8)
    scales = np.array([[120, 125, 130, 127]] * 3, np.uint8)
    got = O.decode_mxfp4(O.pack_fp4(codes), scales)
    assert np.array_equal(got, O.decode_e2m1(codes) * np.repeat(O.decode_ue8m0(scales), 32, axis=1))


def test_mxfp4_decode_layout():
    check_mxfp4_layout()


def test_pins_catch_swapped_nibbles(monkeypatch):
    good = O.decode_mxfp4

    def bad(codes_packed, scale_bytes, block=O.FP4_BLOCK):   # high nibble taken as the even element
        c = np.asarray(codes_packed, np.uint8)
        return good(((c & 0xF) << 4) | (c >> 4), scale_bytes, block)
    _expect_fail(check_mxfp4_layout, monkeypatch, "decode_mxfp4", bad)


def test_pins_catch_missing_relu(monkeypatch):
    def bad(q_fp4, q_sf, k_fp4, k_sf, weights, lengths):
        M, N = q_fp4.shape[0], k_fp4.shape[0]
        Q = O.decode_mxfp4(q_fp4.reshape(M * 64, 64), q_sf.reshape(M * 64, 4)).reshape(M, 64, 128)
        K = O.decode_mxfp4(k_fp4, k_sf)
        s = np.einsum("mh,mhn->mn", np.asarray(weights, np.float64), np.einsum("mhd,nd->mhn", Q, K))
        return np.where(np.arange(N)[None, :] < np.asarray(lengths)[:, None], s, -np.inf)
    _expect_fail(check_relu_and_weights, monkeypatch, "indexer_logits", bad)


def test_pins_catch_off_by_one_visibility(monkeypatch):
    good = O.indexer_logits

    def bad(q_fp4, q_sf, k_fp4, k_sf, weights, lengths):   # keys s <= L visible
        return good(q_fp4, q_sf, k_fp4, k_sf, weights, np.asarray(lengths) + 1)
    _expect_fail(check_logits_bruteforce, monkeypatch, "indexer_logits", bad)


def test_pins_catch_ties_to_larger_index(monkeypatch):
    def bad(scores, lengths, k):
        M = scores.shape[0]
        out = np.full((M, k), -1, np.int32)
        for t in range(M):
            L = int(lengths[t])
            idx = np.arange(L)
            order = np.lexsort((-idx, -scores[t, :L]))
            ch = np.sort(order[:k])
            out[t, :len(ch)] = ch
        return out
    _expect_fail(check_topk_against_sort, monkeypatch, "indexer_topk", bad)
