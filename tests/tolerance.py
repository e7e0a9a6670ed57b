"""The attention tolerance: |gpu - ref| <= 2e-3 + 1e-2 * |ref| elementwise,
the bf16 GPU output upcast to fp64 against the fp64 oracle."""

import numpy as np

ATOL = 2e-3
RTOL = 1e-2


def check_close(gpu_bf16, ref_f64, what=""):
    g = gpu_bf16.detach().to("cpu").double().numpy()
    r = np.asarray(ref_f64, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    err = np.abs(g - r)
    bound = ATOL + RTOL * np.abs(r)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"max abs err {err.max():.3e}; first bad {idx.tolist()} "
                             f"gpu {g[tuple(idx[0])]:.6f} ref {r[tuple(idx[0])]:.6f}")
    return float(err.max()), float((err / (np.abs(r) + 1e-30)).max())
