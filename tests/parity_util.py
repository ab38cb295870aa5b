"""Shared helpers of the GPU parity tests: seeded inputs, tolerances, oracle runs.

Tolerances (stated by the benchmark spec for this path):
* fp32 momentum, RowNorm and apply: 1e-5, read here elementwise relative to
  |ref| + RMS(ref) (so that entries near zero are judged on the matrix's scale);
* bf16 W after an fp32-exact update: within 1 bf16 ulp of the oracle's rounding;
* Newton-Schulz output: relative Frobenius error 3e-2 (bf16 GEMMs) or 1e-4
  (fp32 mode).
"""
import math

import numpy as np
import torch

from oracle import muon_ref
from synth import gradient_np, quantize_np, weight_init_np

TOL_F32 = 1e-5
TOL_NS5_BF16 = 3e-2
TOL_NS5_F32 = 1e-4
SCALES8 = tuple(1e-2 * 0.5 ** i for i in range(8))
TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def dev():
    return torch.device("cuda:0")


def to_dev(x: np.ndarray, dt: str):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev(), TORCH_DT[dt])


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def inputs(shapes, dt_w, dt_g, steps, seed=0, scales=SCALES8):
    """W0 and the per-step gradients as the storage dtypes hold them (float32 arrays)."""
    W0 = [quantize_np(weight_init_np(a, b, seed, i), dt_w) for i, (a, b) in enumerate(shapes)]
    Gs = [[quantize_np(gradient_np(a, b, scales, seed, i, t), dt_g) for i, (a, b) in enumerate(shapes)]
          for t in range(steps)]
    return W0, Gs


def assert_f32_close(got, ref, tol=TOL_F32, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    scale = np.abs(ref) + (muon_ref.rms(ref) if ref.size else 0.0)
    bad = np.abs(got - ref) > tol * scale + 1e-30
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} beyond {tol}; max rel " \
                          f"{float(np.max(np.abs(got - ref) / (scale + 1e-30)))}"


def bf16_ulp(x):
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(x > 0, x, 1.0)))
    return np.where(x > 0, 2.0 ** (e - 7), 2.0 ** -133)


def assert_bf16_within_ulp(got, ref_exact, ulps=1.0, what=""):
    """got (bf16 values) within `ulps` bf16 ulps of the exact fp64 result."""
    got = np.asarray(got, dtype=np.float64)
    diff = np.abs(got - ref_exact)
    lim = ulps * bf16_ulp(ref_exact) + 1e-30
    bad = diff > lim
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} beyond {ulps} ulp; worst {float(np.max(diff / lim))}"


def apply_terms(W_old, U, s, eta, lam):
    """Magnitudes of the summands of W - eta*(s*U + lambda*W), elementwise."""
    W_old = np.abs(np.asarray(W_old, dtype=np.float64))
    return W_old * (1.0 + eta * lam) + eta * s * np.abs(np.asarray(U, dtype=np.float64))


def assert_bf16_close(got, ref_exact, terms, what=""):
    """bf16 result of an fp32 update: within 1 bf16 ulp of the exact result plus the
    fp32 tolerance (1e-5) on the magnitudes of the summed terms.  The second part
    matters only where the terms cancel and the result is much smaller than them."""
    got = np.asarray(got, dtype=np.float64)
    lim = bf16_ulp(ref_exact) + TOL_F32 * np.asarray(terms, dtype=np.float64) + 1e-30
    diff = np.abs(got - ref_exact)
    bad = diff > lim
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} beyond 1 ulp + 1e-5*terms; worst {float(np.max(diff / lim))}"


def rel_fro(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / d) if d > 0 else float(np.linalg.norm(got))


def check_implied_direction(got, prevW, refW_exact, eta, lam, s, tol, what=""):
    """Newton-Schulz direction implied by a refresh step's stored W:
        O = (W_prev*(1 - eta*lam) - W_new) / (eta*s),
    for the GPU's W_new and for the oracle's unrounded W_new.  The GPU's implied O must
    be within `tol` (relative Frobenius) of the oracle's, plus the storage rounding of
    W_new: at most half an ulp per element (of bf16 or fp32), divided by eta*s."""
    got = np.asarray(got, dtype=np.float64)
    prevW = np.asarray(prevW, dtype=np.float64)
    refW_exact = np.asarray(refW_exact, dtype=np.float64)
    keep = prevW * (1.0 - eta * lam)
    O_got = (keep - got) / (eta * s)
    O_ref = (keep - refW_exact) / (eta * s)
    half_ulp = 0.5 * bf16_ulp(np.maximum(np.abs(got), np.abs(refW_exact)))
    err = np.linalg.norm(O_got - O_ref)
    lim = tol * np.linalg.norm(O_ref) + np.linalg.norm(half_ulp) / (eta * s)
    assert err <= lim, f"{what}: implied direction error {err:.3e} > {lim:.3e} " \
                       f"(relative {err / max(np.linalg.norm(O_ref), 1e-30):.3e})"
    return err / max(np.linalg.norm(O_ref), 1e-30)
