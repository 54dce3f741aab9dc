"""The literal constants of the FP4 stage's device code, read from its header
and checked against values computed here: float32(1/6), float32(1/sqrt(128)),
and the reciprocal tables that give 1/s from an E4M3 scale code.  The
reciprocal is replayed for every finite positive E4M3 code and compared with
the correctly rounded float32 quotient (numpy's float32 division is IEEE
round-to-nearest-even), with the code values taken from the oracle's E4M3
table."""

from __future__ import annotations

import re
from decimal import Decimal, getcontext
from pathlib import Path

import numpy as np
import pytest

from oracle import iq_oracle as O

HEADER = Path(__file__).resolve().parents[1] / "fp4_fp8_quant_gb300" / "csrc" / "iq_fp4.cuh"


def _f32(x: float) -> np.float32:
    return np.float32(x)


def _body(name: str) -> str:
    src = HEADER.read_text()
    start = src.index(f"float {name}(")
    return src[start:src.index("\n}\n", start)]


def _constexpr(name: str) -> str:
    m = re.search(rf"constexpr float {name} = ([^;]+);", HEADER.read_text())
    assert m, name
    return m.group(1).rstrip("f")


def _select_tables() -> list[list[int]]:
    body = _body("e4m3_reciprocal")
    calls = re.findall(r"select8\(m,([^)]*)\)", body.replace("\n", " "))
    tables = [[int(t.strip().rstrip("u"), 16) if t.strip() != "0u" else 0 for t in c.split(",")] for c in calls]
    assert len(tables) == 2 and all(len(t) == 8 for t in tables)
    return tables


def _replay(code: int, sub: list[int], norm: list[int]) -> np.float32:
    """The device routine's steps: pick the constant by the mantissa, add the
    power-of-two factor to the exponent field."""
    m, E = code & 7, (code >> 3) & 15
    bits = sub[m] + (9 << 23) if E == 0 else norm[m] + ((7 - E) << 23)
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


def test_sixth_is_float32_one_sixth():
    assert _f32(float.fromhex(_constexpr("kSixth"))) == np.float32(1) / np.float32(6)


def test_inv_sqrt128_is_correctly_rounded():
    getcontext().prec = 60
    exact = Decimal(2).sqrt() / 16          # 1 / sqrt(128)
    got = _f32(float(Decimal(_constexpr("kInvSqrt128"))))
    lo, hi = np.nextafter(got, np.float32(0)), np.nextafter(got, np.float32(1))
    d = abs(Decimal(float(got)) - exact)
    assert d <= abs(Decimal(float(lo)) - exact) and d <= abs(Decimal(float(hi)) - exact)


def test_e4m3_reciprocal_every_positive_code():
    sub, norm = _select_tables()
    vals = O.e4m3_value_table()
    checked = 0
    for code in range(1, 0x7F):              # 0x7F is NaN; 0 is never a scale
        v = np.float32(vals[code])
        assert np.float64(v) == vals[code]   # every E4M3 value is a float32
        want = np.float32(1) / v
        got = _replay(code, sub, norm)
        assert got == want, (hex(code), got, want)
        checked += 1
    assert checked == 126


def test_replay_catches_a_wrong_constant():
    """A planted one-ulp error in a table entry fails the comparison."""
    sub, norm = _select_tables()
    bad = list(norm)
    bad[3] += 1
    vals = O.e4m3_value_table()
    assert any(_replay(c, sub, bad) != np.float32(1) / np.float32(vals[c]) for c in range(1, 0x7F))


@pytest.mark.gpu
def test_gpu_e2m1_conversion_dense_sweep(cuda_device):
    """The GPU's float -> E2M1 conversion (the one both fused GEMM kernels
    use) on a dense float32 sweep of [-7, 7] with every rounding midpoint, the
    float32 neighbours of each midpoint and grid value, signed zeros and
    values past the saturation bound, against the oracle's round-to-nearest-
    even rule."""
    import torch
    from fp4_fp8_quant_gb300 import iq
    from oracle import iq_oracle as O
    grid = O.e2m1_value_table()[:8].astype(np.float32)
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    special = np.concatenate([mids, grid, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(10)),
                              np.nextafter(grid, np.float32(0)), np.nextafter(grid, np.float32(10)),
                              [6.5, 7.0, 1e30, 0.0, 1e-30, 1e-45]]).astype(np.float32)
    dense = np.linspace(-7, 7, 1 << 21, dtype=np.float32)
    x = np.concatenate([dense, special, -special]).astype(np.float32)
    x = np.concatenate([x, np.zeros((-len(x)) % 8, np.float32)])
    x[-1] = np.float32(-0.0)
    xd = torch.from_numpy(x).cuda()
    codes = torch.empty(len(x), dtype=torch.uint8, device="cuda")
    rc = iq.lib().iq_debug_e2m1_codes(xd.data_ptr(), len(x), codes.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    got = codes.cpu().numpy()
    want = O.round_to_e2m1_codes(x.astype(np.float64))      # saturates at 6, keeps the sign
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first x={x[bad[:5]]} got={got[bad[:5]]} want={want[bad[:5]]}"
