"""Acceptance checks shared by the GPU parity tests.

  * indices, counts, offsets, row_src, inv: bit-exact;
  * FP32 routing weights: relative error <= 1e-6;
  * dtype routing weights: the GPU's value is its own FP32 weight rounded to
    nearest-even, and differs from the oracle's dtype weight by at most one
    dtype ulp (only where the two FP32 weights straddle a rounding boundary);
  * outputs: F32 max-abs <= 1e-4; F16/BF16 per element
    |gpu - ref| <= 2e-2 * (|ref| + rms(ref)) and max|gpu - ref| / max|ref| <= 2e-2;
  * NaN positions identical everywhere.
"""
import numpy as np
import torch

from oracle import moe_oracle

WEIGHT_RTOL_FP32 = 1e-6
OUT_ATOL_F32 = 1e-4
OUT_RTOL_16 = 2e-2
_ULP_REL = {torch.bfloat16: 2.0 ** -7, torch.float16: 2.0 ** -10, torch.float32: 2.0 ** -23}


def u32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def assert_nan_positions_equal(got: np.ndarray, ref: np.ndarray, what: str):
    bad = np.isnan(got) != np.isnan(ref)
    assert not bad.any(), f"{what}: NaN positions differ at {np.argwhere(bad)[:5].tolist()}"


def assert_route_matches(indices, weights, weights32, ref: "moe_oracle.RouteResult", dtype):
    gi = u32(indices)
    mism = np.argwhere(gi != ref.indices)
    assert mism.size == 0, f"indices differ at {mism[:5].tolist()}: {gi[tuple(mism[0])]} vs {ref.indices[tuple(mism[0])]}"

    g32 = f64(weights32)
    assert_nan_positions_equal(g32, ref.weights32.astype(np.float64), "FP32 weights")
    fin = ~np.isnan(ref.weights32)
    r32 = ref.weights32.astype(np.float64)[fin]
    rel = np.abs(g32[fin] - r32) / np.maximum(np.abs(r32), np.finfo(np.float32).tiny)
    assert rel.size == 0 or rel.max() <= WEIGHT_RTOL_FP32, f"FP32 weight rel error {rel.max():.3e}"

    gd = f64(weights)
    assert_nan_positions_equal(gd, ref.weights, "dtype weights")
    if dtype == torch.float32:  # the dtype weights are the FP32 weights checked above
        assert np.array_equal(gd[fin], g32[fin])
        return
    own = moe_oracle.round_to_dtype(f64(weights32).astype(np.float32), dtype)
    assert np.array_equal(gd[fin], own[fin]), "GPU dtype weights are not its FP32 weights rounded to nearest-even"
    diff = np.abs(gd[fin] - ref.weights[fin])
    assert (diff <= _ULP_REL[dtype] * np.abs(ref.weights[fin]) * 1.0000001).all(), "dtype weights differ by more than 1 ulp"
    assert np.count_nonzero(diff) <= max(2, int(0.01 * diff.size)), "too many dtype-weight rounding flips"


def assert_output_close(got: np.ndarray, ref: np.ndarray, dtype, what: str = "out"):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert_nan_positions_equal(got, ref, what)
    fin = ~np.isnan(ref)
    g, r = got[fin], ref[fin]
    if g.size == 0:
        return
    if dtype == torch.float32:
        err = np.abs(g - r).max()
        assert err <= OUT_ATOL_F32, f"{what}: max-abs error {err:.3e} > {OUT_ATOL_F32}"
    else:
        rms = float(np.sqrt(np.mean(r * r)))
        per = np.abs(g - r) / (np.abs(r) + rms)
        assert per.max() <= OUT_RTOL_16, f"{what}: per-element relative error {per.max():.3e}"
        tens = np.abs(g - r).max() / max(np.abs(r).max(), 1e-30)
        assert tens <= OUT_RTOL_16, f"{what}: tensor relative error {tens:.3e}"
