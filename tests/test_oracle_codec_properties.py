"""Property tests of the oracle's 4-bit quantisers (CPU only; needs hypothesis).

Arbitrary float32 blocks -- subnormals, signed zeros, values at and around every rounding
boundary the strategies happen to hit -- quantised by the C oracle must match the
Fraction brute force of oracle/tiny.py bit for bit: MXFP4 (OCP MX rule; report §2.4.4,
indexer queries and keys) and E2M1 + E4M3 per 16 (report §2.4.4, main KV)."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import tiny

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

f32 = st.floats(width=32, allow_nan=False, allow_infinity=False)
# values near the E2M1 grid at a common scale, so ties and near-ties occur often
grid = st.sampled_from([0.0, 0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0, 6.0])
scaled_grid = st.builds(lambda v, e, neg: np.float32((-v if neg else v) * 2.0 ** e), grid,
                        st.integers(-20, 20), st.booleans())
elem = st.one_of(f32, scaled_grid)


def _signs(xs):
    return [bool(np.signbit(np.float32(v))) for v in xs]


@settings(max_examples=300, deadline=None)
@given(st.lists(elem, min_size=32, max_size=32))
def test_mxfp4_matches_bruteforce(xs):
    x = np.array(xs, np.float32).astype(np.float64)[None]
    codes, scales = oracle.quant_mxfp4(x)
    sb, cs = tiny.quant_block([Fraction(float(v)) for v in xs], _signs(xs))
    assert scales[0, 0] == sb
    assert tiny.unpack_codes(codes[0]) == cs


@settings(max_examples=300, deadline=None)
@given(st.lists(elem, min_size=16, max_size=16))
def test_e2m1_e4m3_16_matches_bruteforce(xs):
    x = np.array(xs, np.float32).astype(np.float64)[None]
    codes, scales = oracle.quant_nvfp4(x)
    sb, cs = tiny.quant_block_nvfp4([Fraction(float(v)) for v in xs], _signs(xs))
    assert scales[0, 0] == sb
    assert tiny.unpack_codes(codes[0]) == cs
