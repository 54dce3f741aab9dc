"""The FP4 comparison rules of tests/parity.py, on the CPU: they accept the
oracle's own output, accept a code flipped at a rounding midpoint, and reject
a code or a scale byte that is wrong away from a decision boundary."""

import numpy as np
import pytest

from oracle import iq_oracle as O
from fp4_fp8_quant_gb300 import workloads as W
from tests.parity import check_fp4, unpack_fp4


def _repack(codes):
    return O.pack_fp4(codes)


@pytest.mark.parametrize("fmt", O.FP4_FORMATS)
def test_rules_accept_the_oracle_and_reject_planted_errors(fmt):
    x, wq, wsf, pos = W.tiny_chain(8)
    q, sf, z = O.prepare_q(x, wq, wsf, pos, fmt)
    check_fp4(q, sf, q, sf, z, fmt=fmt)
    codes = unpack_fp4(q)
    # a code two steps away from the oracle's: rejected
    bad = codes.copy()
    j = int(np.argmax((bad[0] & 7) <= 4))
    bad[0, j] = (bad[0, j] & 8) | ((bad[0, j] & 7) + 2)
    with pytest.raises(AssertionError):
        check_fp4(_repack(bad), sf, q, sf, z, fmt=fmt, min_equal=0.0)
    # a scale byte changed in a block whose amax is far from the rule's boundary: rejected
    bad_sf = sf.copy()
    bad_sf[1, 3] = bad_sf[1, 3] + 1
    with pytest.raises(AssertionError):
        check_fp4(q, bad_sf, q, sf, z, fmt=fmt, min_equal=0.0)


def test_rules_accept_a_flip_at_a_rounding_midpoint():
    # a value exactly at the E2M1 midpoint 2.5 (between codes 4 and 5) in a
    # block whose scale is 1: either neighbouring code is acceptable
    z = np.zeros((1, 8192))
    z[0, 0] = 6.0          # block amax 6 -> ceil-rule scale 2^0
    z[0, 1] = 2.5
    codes, sb = O.quantize_fp4_1x32(z.astype(np.float32).astype(np.float64))
    assert sb[0, 0] == 127 and codes[0, 1] == 4       # ties to even: 2.5 -> 2
    flipped = codes.copy()
    flipped[0, 1] = 5                                  # 3
    stats = check_fp4(O.pack_fp4(flipped), sb, O.pack_fp4(codes), sb, z, min_equal=0.0)
    assert stats["code_mismatches"] == 1
