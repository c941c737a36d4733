"""Shared helpers of the GPU parity tests: tolerances and comparison with the oracle."""
import numpy as np
import torch

# Output tolerance |gpu - oracle| <= atol + rtol * |oracle| per storage dtype, and the
# absolute tolerance on the natural-log LSE.
TOL = {torch.bfloat16: (2e-2, 2e-2), torch.float16: (5e-3, 5e-3), torch.float32: (1e-5, 1e-5)}
LSE_TOL = 1e-3


def assert_matches_oracle(o, lse, ref_o, ref_lse, dtype, what=""):
    atol, rtol = TOL[dtype]
    o = o.float().cpu().numpy().astype(np.float64)
    ref_o = np.asarray(ref_o, dtype=np.float64)
    assert o.shape == ref_o.shape, (o.shape, ref_o.shape)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    excess = np.abs(o - ref_o) - (atol + rtol * np.abs(ref_o))
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, (f"{what}: output off by {np.abs(o - ref_o)[worst]:.3e} at {worst} "
                               f"(gpu {o[worst]:.5f}, oracle {ref_o[worst]:.5f})")
    if lse is not None:
        lse = lse.float().cpu().numpy().astype(np.float64)
        ref_lse = np.asarray(ref_lse, dtype=np.float64)
        both_inf = np.isneginf(lse) & np.isneginf(ref_lse)
        with np.errstate(invalid="ignore"):
            d = np.where(both_inf, 0.0, np.abs(lse - ref_lse))
        assert np.isfinite(d).all() and d.max() <= LSE_TOL, f"{what}: lse off by {np.nanmax(d):.3e}"
