"""Shared helpers for the GPU parity tests (comparison metrics and tolerances)."""
import numpy as np
import torch

# fp32 inputs: relative L2 error over the whole output
TOL_F32_REL = 1e-5
# bf16 inputs with fp32 accumulation: relative L2 AND absolute max error
TOL_BF16_REL = 1e-2
TOL_BF16_ABS = 2e-2


def to_np(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def errors(got, ref):
    g, r = to_np(got), to_np(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.isfinite(g).all(), "non-finite output"
    diff = g - r
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(r), 1e-300))
    return rel, float(np.abs(diff).max()) if diff.size else 0.0


def report(what, rel, mx, ref=None):
    """One line per comparison, for the parity record a `pytest -s` run prints."""
    top = f" max|ref| {float(np.abs(to_np(ref)).max()):.3g}" if ref is not None else ""
    print(f"PARITY {what}: rel-L2 {rel:.3e} max-abs {mx:.3e}{top}")


def assert_f32(got, ref, what=""):
    rel, mx = errors(got, ref)
    report(what, rel, mx, ref)
    assert rel <= TOL_F32_REL, f"{what}: rel-L2 {rel:.3e} > {TOL_F32_REL} (max-abs {mx:.3e})"
    return rel, mx


def assert_bf16(got, ref, what=""):
    rel, mx = errors(got, ref)
    report(what, rel, mx, ref)
    assert rel <= TOL_BF16_REL and mx <= TOL_BF16_ABS, \
        f"{what}: rel-L2 {rel:.3e} (<= {TOL_BF16_REL}), max-abs {mx:.3e} (<= {TOL_BF16_ABS})"
    return rel, mx
