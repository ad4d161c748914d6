"""Helpers shared by the GPU parity tests (not a test module)."""
import numpy as np
import pytest
import torch

import oracle

FP32_TOL = 1e-5    # max relative L2 error, float32 activations
BF16_TOL = 1e-2    # max relative L2 error, bf16 activations


def lib():
    """Builds (if stale) and loads the CUDA library; skips when no GPU is visible."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_w4a16_group_gb300.build import build
    build()
    import int4_w4a16_group_gb300 as w4
    torch.cuda.set_device(0)
    return w4


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_close_rows(got, ref, tol, what=""):
    """rel-L2 over the whole tensor and over every row must be <= tol."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    e = oracle.rel_l2(got, ref)
    assert e <= tol, f"{what}: rel-L2 {e:.3e} > {tol:.0e}"
    for r in range(ref.shape[0]):
        if np.linalg.norm(ref[r]) > 0:
            er = oracle.rel_l2(got[r], ref[r])
            assert er <= tol, f"{what}: row {r} rel-L2 {er:.3e} > {tol:.0e}"
    return e
