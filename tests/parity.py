"""Comparison helpers shared by the GPU parity tests.

Tolerances (floating point, fixed for the hot path): output max-abs <= 2e-2
and relative L2 <= 5e-3; LSE max-abs <= 1e-3 on finite entries with the -inf
entries in the same places; dQ/dK/dV relative L2 <= 1e-2; rows with no
visible key exactly 0.  Integer and index work is compared bit for bit.
"""
import numpy as np
import torch

OUT_MAX_ABS = 2e-2
OUT_REL_L2 = 5e-3
LSE_MAX_ABS = 1e-3
GRAD_REL_L2 = 1e-2


def to64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def rel_l2(got, ref):
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def check_out(got, ref, what="out"):
    got, ref = to64(got), to64(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    rel = rel_l2(got, ref)
    assert err <= OUT_MAX_ABS, f"{what}: max-abs {err:.3e} > {OUT_MAX_ABS}"
    assert rel <= OUT_REL_L2, f"{what}: rel-L2 {rel:.3e} > {OUT_REL_L2}"
    return err, rel


def check_lse(got, ref, what="lse"):
    got, ref = to64(got), to64(ref)
    assert got.shape == ref.shape
    ninf_g, ninf_r = np.isneginf(got), np.isneginf(ref)
    assert np.array_equal(ninf_g, ninf_r), \
        f"{what}: -inf mismatch at {np.argwhere(ninf_g != ninf_r)[:5].tolist()}"
    fin = ~ninf_r
    assert np.all(np.isfinite(got[fin])), f"{what}: non-finite values"
    err = float(np.abs(got[fin] - ref[fin]).max()) if fin.any() else 0.0
    assert err <= LSE_MAX_ABS, f"{what}: max-abs {err:.3e} > {LSE_MAX_ABS}"
    return err


def check_grad(got, ref, what):
    got, ref = to64(got), to64(ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    rel = rel_l2(got, ref)
    assert rel <= GRAD_REL_L2, f"{what}: rel-L2 {rel:.3e} > {GRAD_REL_L2}"
    return rel
