"""Shared helpers of the parity tests: tolerances and the comparison report."""
import numpy as np

# Bars: bf16 inputs with fp32 accumulation -> max |dO| <= 2e-2 and mean |dO| <= 2e-3;
# fp32 inputs -> |dO| <= 1e-4; LSE within 1e-3 in both cases.
BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
FP32_MAX_ABS = 1e-4
LSE_MAX_ABS = 1e-3


def compare(o_gpu, lse_gpu, o_ref, lse_ref, dtype: str, what: str = ""):
    """Assert the GPU result (float arrays) is within the bars of the fp64 oracle."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    err = np.abs(o_gpu - o_ref)
    mx, mean = float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0
    if dtype == "fp32":
        assert mx <= FP32_MAX_ABS, f"{what}: max |dO| {mx:.3e} > {FP32_MAX_ABS}"
    else:
        assert mx <= BF16_MAX_ABS, f"{what}: max |dO| {mx:.3e} > {BF16_MAX_ABS}"
        assert mean <= BF16_MEAN_ABS, f"{what}: mean |dO| {mean:.3e} > {BF16_MEAN_ABS}"
    if lse_gpu is not None:
        lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
        lse_ref = np.asarray(lse_ref, dtype=np.float64)
        inf_g, inf_r = np.isneginf(lse_gpu), np.isneginf(lse_ref)
        assert np.array_equal(inf_g, inf_r), f"{what}: -inf LSE pattern differs"
        fin = ~inf_r
        lerr = float(np.abs(lse_gpu[fin] - lse_ref[fin]).max(initial=0.0))
        assert lerr <= LSE_MAX_ABS, f"{what}: max |dLSE| {lerr:.3e} > {LSE_MAX_ABS}"
    return mx, mean
