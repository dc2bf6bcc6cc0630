"""Helpers shared by the tests (comparison rules, device setup)."""
import numpy as np
import torch


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").double().numpy()


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits); floor at the smallest normal."""
    a = np.maximum(np.abs(x), 2.0 ** -126)
    e = np.floor(np.log2(a))
    return np.ldexp(1.0, (e - 7).astype(int))


def assert_within_ulps(got: np.ndarray, ref: np.ndarray, ulps: float = 1.0, min_exact: float = 0.0, what="",
                       atol=0.0):
    """|got - ref| <= ulps * ulp_bf16(ref) + atol elementwise; at least `min_exact` of the elements identical."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    tol = ulps * bf16_ulp(ref) + atol
    bad = np.abs(got - ref) > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements beyond {ulps} ulp; first at {tuple(i)}: "
                             f"got {got[tuple(i)]!r} ref {ref[tuple(i)]!r}")
    if min_exact > 0:
        frac = float(np.mean(got == ref))
        assert frac >= min_exact, f"{what}: only {frac:.4f} of elements bit-identical (need {min_exact})"


def normwise_rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))
