"""The hi + lo E4M3 split the FP8 kernels feed to E4M3 MMAs (Q, and P in the decode kernel):
hi = e4m3(x), lo = e4m3(x - hi), after scaling x by a power of two into [128, 256).  In that
range hi is within half a step (8) of x and lo carries the remainder with 3 mantissa bits, so
hi + lo keeps x to within 2^-8 relative -- the precision of a bf16 operand -- which is why the
FP8 paths meet the same bar as bf16.  Checked with the oracle's E4M3 encoder (RNE, saturating)."""
import numpy as np

import oracle


def _split(x):
    hi = oracle.e4m3_decode(oracle.e4m3_encode(x.astype(np.float32)))
    lo = oracle.e4m3_decode(oracle.e4m3_encode((x - hi).astype(np.float32)))
    return hi, lo


def test_split_keeps_eight_bits_in_the_scaled_range():
    rng = np.random.default_rng(7)
    x = rng.uniform(128.0, 256.0, 200000) * rng.choice([-1.0, 1.0], 200000)
    hi, lo = _split(x)
    rel = np.abs(x - (hi + lo)) / np.abs(x)
    assert rel.max() <= 2.0 ** -8
    # one E4M3 code alone is far coarser (up to half a step of 16 at 128..256)
    assert (np.abs(x - hi) / np.abs(x)).max() > 2.0 ** -5


def test_split_of_scaled_rows_matches_a_bf16_operand():
    # a Q row scaled by 2^(8 - e), e the exponent of its largest |q|: the largest element lands
    # in [128, 256); smaller ones keep at least bf16's precision relative to the row maximum
    rng = np.random.default_rng(11)
    q = rng.standard_normal((64, 128))
    amax = np.abs(q).max(axis=1, keepdims=True)
    e = np.frexp(amax)[1]
    up = np.ldexp(1.0, 8 - e)
    x = q * up
    hi, lo = _split(x)
    err = np.abs(x - (hi + lo)).max(axis=1) / np.abs(x).max(axis=1)
    assert err.max() <= 2.0 ** -8
