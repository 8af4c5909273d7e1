"""Comparison helpers for GPU-vs-oracle parity (test infrastructure)."""
import numpy as np

# bits of mantissa (excluding the implicit bit) and smallest normal exponent
_FMT = {"f16": (10, -14), "bf16": (7, -126)}


def ulp(ref: np.ndarray, fmt: str) -> np.ndarray:
    """One unit in the last place of `fmt` at |ref| (subnormal spacing below
    the smallest normal)."""
    mant, emin = _FMT[fmt]
    mag = np.maximum(np.abs(ref), 2.0 ** emin)
    return np.exp2(np.floor(np.log2(mag)) - mant)


def within_bound(got, ref, absref, fmt: str, rel: float = 4e-3):
    """|got - ref| <= rel * sum_k |a_k w_k| + 1 ulp(fmt at ref): the float
    acceptance bound for every W4A16 output element."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bound = rel * absref + ulp(ref, fmt)
    bad = ~(err <= bound)
    return bad, err, bound


def assert_within(got, ref, absref, fmt: str, what: str = ""):
    bad, err, bound = within_bound(got, ref, absref, fmt)
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} elements outside the bound; first at flat "
            f"{list(i)}: got {np.asarray(got).ravel()[i]}, ref {ref.ravel()[i]}, "
            f"err {err.ravel()[i]}, bound {bound.ravel()[i]}")


def assert_fp16_within_ulp(got, ref, what: str = ""):
    """W4A8 fp16 output: within one fp16 ulp of the fp64 reference."""
    got = np.asarray(got, dtype=np.float64)
    bad = ~(np.abs(got - ref) <= ulp(ref, "f16"))
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} fp16 outputs off by > 1 ulp: got "
                             f"{got.ravel()[i]}, ref {ref.ravel()[i]}")


def assert_fp16_near(got, ref, scale, what: str = ""):
    """W4A8 fp16 output with a bias: within one fp16 ulp of the fp64
    reference, plus the fp32 rounding of the epilogue (2^-21 of the
    magnitudes it adds: |acc * s_tok * s_ch| + |bias|), which a bias close to
    minus the product can expose."""
    got = np.asarray(got, dtype=np.float64)
    bound = ulp(ref, "f16") + 2.0 ** -21 * np.asarray(scale, dtype=np.float64)
    bad = ~(np.abs(got - ref) <= bound)
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} fp16 outputs outside 1 ulp + epilogue "
                             f"rounding: got {got.ravel()[i]}, ref {ref.ravel()[i]}")
