"""fp64 CPU oracle for the Muon optimizer step and Periodic Row-wise Muon.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this module.  The product path (the
CUDA library and its Python binding) never calls it and shares no code with it.

Everything is plain numpy in float64.  Each function follows one passage of
the pages, in the pages' order and notation:

* "Muon is Scalable for LLM Training" (paper notes), section 2.1, Eq. (1):
  M_t = mu*M_{t-1} + grad, with M_0 = 0;  O_t = Newton-Schulz(M_t).
* same page, section 2.1, Eq. (2): X_0 = M_t/||M_t||_F, then
  X_k = a X + b (X X^T) X + c (X X^T)^2 X with (a, b, c) = (3.4445, -4.7750, 2.0315);
  section 2.2 "Other hyper-parameters": N = 5 iterations, mu = 0.95.
* same page, section 2.2, Eq. (3)/(4) and section 3.1 Eq. (7):
  W_t = W_{t-1} - eta*(0.2*sqrt(max(A, B))*O_t + lambda*W_{t-1}).
* "Scaling Muon for Diffusion Transformers" (summary page), the Periodic
  Row-wise paragraphs, and the same paper's abstract: a full NS5 refresh once
  every K steps (K = 3) and, on the other steps, a row-wise constrained update
  built from the current momentum, with step size gamma (= 0.15) relative to
  the NS5 branch; wide matrices normalise rows, tall matrices normalise columns
  (the distributed-implementation paragraph: "tall matrices only all-reduce the
  per-column norm scalars").

Readings where the pages are silent:
* the RowNorm lines are the min(A, B) lines along the long dimension: rows when
  A <= B (square counts as wide), columns when A > B;
* RowNorm steps use the scale gamma*0.2*sqrt(max(A, B)); weight decay applies on
  both branches;
* refresh iff step % K == 0 with step counted from 0;
* a zero matrix (for NS5) or a zero line (for RowNorm) gives a zero direction,
  with no epsilon; any other norm, NaN or Inf included, divides as written, so
  non-finite values in M propagate as IEEE arithmetic carries them;
* the NS5 iteration runs on the short side: a tall matrix is transposed, iterated,
  and transposed back;
* bf16 storage of W is round-to-nearest-even of the exact fp64 result;
* the Eq. (6) "Update Norm" variant on RowNorm steps takes the RMS over the lines
  that carry the update, i.e. it equals the Eq. (7) scale unless a line is zero.

Every function here is pinned by the tests in tests/test_oracle_pins.py against
closed forms, invariants, values the pages print, or brute force.  No function
is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

# Muon is Scalable for LLM Training, section 2.1 (text after Eq. (2)).
NS_A = 3.4445
NS_B = -4.7750
NS_C = 2.0315
# Same page, section 2.2 "Other hyper-parameters".
NS_STEPS = 5
MU_DEFAULT = 0.95
# Same page, Eq. (4): match AdamW's update RMS of about 0.2.
RMS_MATCH = 0.2
# Scaling Muon for Diffusion Transformers, the Periodic Row-wise paragraph
# (final choice after the K/gamma sweep).
K_DEFAULT = 3
GAMMA_DEFAULT = 0.15


def is_refresh(step: int, K: int) -> bool:
    """Periodic schedule: a full NS5 refresh once every K steps.

    Scaling Muon for Diffusion Transformers, the Periodic Row-wise paragraph and
    the abstract ("a full NS5 spectral update once every K steps").  Reading: the
    refresh falls on steps with step % K == 0, counting from 0.
    """
    if K < 1:
        raise ValueError("K must be >= 1")
    if step < 0:
        raise ValueError("step must be >= 0")
    return step % K == 0


def momentum(M_prev: np.ndarray, G: np.ndarray, mu: float) -> np.ndarray:
    """Muon is Scalable for LLM Training, section 2.1, Eq. (1), first line: M_t = mu*M_{t-1} + G_t."""
    return mu * np.asarray(M_prev, dtype=np.float64) + np.asarray(G, dtype=np.float64)


def frobenius_norm(M: np.ndarray) -> float:
    """||M||_F = sqrt(sum of squares), used for X_0 = M/||M||_F (section 2.1)."""
    M = np.asarray(M, dtype=np.float64)
    return float(np.sqrt(np.sum(M * M)))


def newton_schulz(M: np.ndarray, steps: int = NS_STEPS,
                  coeffs: tuple = (NS_A, NS_B, NS_C)) -> np.ndarray:
    """Newton-Schulz orthogonalisation of M.

    Muon is Scalable for LLM Training, section 2.1, Eq. (2):
    X_0 = M/||M||_F;  X_k = a X_{k-1} + b (X_{k-1} X_{k-1}^T) X_{k-1}
                           + c (X_{k-1} X_{k-1}^T)^2 X_{k-1};  returns X_N.
    The iteration runs on the short side (a tall matrix is transposed first and
    the result transposed back).  A zero matrix returns zeros.
    """
    a, b, c = coeffs
    M = np.asarray(M, dtype=np.float64)
    tall = M.shape[0] > M.shape[1]
    X = M.T if tall else M
    nrm = frobenius_norm(X)
    if nrm == 0.0:
        return np.zeros_like(M)
    X = X / nrm
    for _ in range(steps):
        XXt = X @ X.T
        X = a * X + b * (XXt @ X) + c * ((XXt @ XXt) @ X)
    return X.T.copy() if tall else X


def rownorm(M: np.ndarray) -> np.ndarray:
    """Row-wise constrained direction of the current momentum (RowNorm branch).

    Scaling Muon for Diffusion Transformers, the abstract and the distributed-
    implementation paragraph: each of the min(A, B) lines along the long dimension
    is scaled to unit L2 norm -- the rows of a wide (or square) matrix, the columns
    of a tall one.  A zero line stays zero.  Every other line is divided by its norm
    as written, so a NaN or Inf in a line gives what IEEE division gives (a NaN norm
    makes the whole line NaN; an Inf norm sends the finite entries to 0).
    """
    M = np.asarray(M, dtype=np.float64)
    A, B = M.shape
    axis = 1 if A <= B else 0          # norm over the long dimension
    norms = np.sqrt(np.sum(M * M, axis=axis, keepdims=True))
    zero = norms == 0.0
    safe = np.where(zero, 1.0, norms)
    with np.errstate(invalid="ignore"):
        return np.where(zero, 0.0, M / safe)


def update_scale(A: int, B: int, refresh: bool, gamma: float) -> float:
    """0.2*sqrt(max(A, B)) (Muon is Scalable, Eq. (4)/(7)); times gamma on RowNorm steps."""
    s = RMS_MATCH * math.sqrt(max(A, B))
    return s if refresh else gamma * s


def apply_update(W: np.ndarray, U: np.ndarray, scale: float, eta: float, lam: float) -> np.ndarray:
    """Muon is Scalable for LLM Training, Eq. (4): W_t = W_{t-1} - eta*(scale*U + lambda*W_{t-1})."""
    W = np.asarray(W, dtype=np.float64)
    return W - eta * (scale * np.asarray(U, dtype=np.float64) + lam * W)


def round_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Value held by a W of the given storage dtype, as float64.

    "f32": IEEE binary32 round-to-nearest-even.  "bf16": round to 8 significant bits,
    ties to even (bfloat16 keeps fp32's exponent range and 7 stored mantissa bits).
    """
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f64":
        return x.copy()
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        frac, exp = np.frexp(x)                 # x = frac * 2**exp, 0.5 <= |frac| < 1
        q = np.rint(np.ldexp(frac, 8))          # 8 significant bits, ties to even
        return np.ldexp(q, exp - 8)
    raise ValueError(dtype)


SCALE_ADJUSTED_LR = "adjusted_lr"   # Eq. (4)/(7): 0.2*sqrt(max(A, B))
SCALE_UPDATE_NORM = "update_norm"   # Eq. (6): 0.2/RMS(U)


def update_norm_scale(U: np.ndarray, refresh: bool, gamma: float) -> float:
    """Muon is Scalable for LLM Training, section 3.1, Eq. (6): the update is normalised
    to RMS 0.2 exactly, s = 0.2/RMS(U) (times gamma on RowNorm steps).

    Reading for the RowNorm branch: the RMS is taken over the lines that carry the
    update (a zero line carries none), so each unit line of length m gives RMS
    1/sqrt(m).  A zero direction gives s = 0.
    """
    U = np.asarray(U, dtype=np.float64)
    A, B = U.shape
    if refresh:
        r = rms(U)
    else:
        line_axis = 1 if B >= A else 0
        nz = int(np.count_nonzero(np.sqrt(np.sum(U * U, axis=line_axis)) > 0.0))
        r = math.sqrt(float(np.sum(U * U)) / (nz * max(A, B))) if nz else 0.0
    if r == 0.0:
        return 0.0
    s = RMS_MATCH / r
    return s * gamma if not refresh else s


def update_rms(U: np.ndarray) -> float:
    """Update-RMS telemetry (Muon is Scalable, section 2.2, the monitoring after Lemma 1):
    RMS of the direction before scaling, over all A*B elements."""
    return rms(U)


def muon_direction(M: np.ndarray, refresh: bool) -> np.ndarray:
    """U_t: Newton-Schulz on refresh steps, RowNorm otherwise."""
    return newton_schulz(M) if refresh else rownorm(M)


def periodic_step(W: np.ndarray, M_prev: np.ndarray, G: np.ndarray, step: int, K: int = K_DEFAULT,
                  gamma: float = GAMMA_DEFAULT, mu: float = MU_DEFAULT, eta: float = 0.02,
                  lam: float = 0.01, w_dtype: str = "f64", scale_mode: str = SCALE_ADJUSTED_LR,
                  telemetry: bool = False):
    """One Periodic Row-wise Muon step on one matrix; returns (W_new, M_new, refresh).

    Order: momentum (Eq. (1)), branch choice (step % K), direction (Eq. (2) or RowNorm),
    scale (Eq. (4)/(7), times gamma on RowNorm steps), apply with weight decay (Eq. (4)),
    then W is stored in w_dtype.  K = 1 is vanilla Muon.
    """
    A, B = np.shape(W)
    M = momentum(M_prev, G, mu)
    refresh = is_refresh(step, K)
    U = muon_direction(M, refresh)
    if scale_mode == SCALE_ADJUSTED_LR:
        scale = update_scale(A, B, refresh, gamma)
    elif scale_mode == SCALE_UPDATE_NORM:
        scale = update_norm_scale(U, refresh, gamma)
    else:
        raise ValueError(scale_mode)
    W_new = apply_update(W, U, scale, eta, lam)
    if telemetry:
        return round_to_storage(W_new, w_dtype), M, refresh, update_rms(U)
    return round_to_storage(W_new, w_dtype), M, refresh


# ---------------------------------------------------------------------------
# Reference quantities used by the pins.
# ---------------------------------------------------------------------------

def quintic(x, coeffs: tuple = (NS_A, NS_B, NS_C)):
    """Scalar map f(x) = a x + b x^3 + c x^5 (Muon is Scalable, section 2.1)."""
    a, b, c = coeffs
    x = np.asarray(x, dtype=np.float64)
    return a * x + b * x ** 3 + c * x ** 5


def quintic_iterated(x, n: int = NS_STEPS, coeffs: tuple = (NS_A, NS_B, NS_C)):
    for _ in range(n):
        x = quintic(x, coeffs)
    return x


def polar_factor(M: np.ndarray) -> np.ndarray:
    """Exact orthogonal factor U V^T of M = U S V^T (Muon is Scalable, section 2.1)."""
    U, _, Vt = np.linalg.svd(np.asarray(M, dtype=np.float64), full_matrices=False)
    return U @ Vt


def rms(X: np.ndarray) -> float:
    X = np.asarray(X, dtype=np.float64)
    return float(np.sqrt(np.mean(X * X))) if X.size else 0.0


# ---------------------------------------------------------------------------
# AdamW for the parameters Muon does not take
# ---------------------------------------------------------------------------
ADAMW_BETA1 = 0.9
ADAMW_BETA2 = 0.999
ADAMW_EPS = 1e-8
ADAMW_AUX_LR = 1e-4   # Scaling Muon for Diffusion Transformers (summary page): auxiliary AdamW group


def adamw_step(p: np.ndarray, g: np.ndarray, m: np.ndarray, v: np.ndarray, t: int, lr: float,
               beta1: float = ADAMW_BETA1, beta2: float = ADAMW_BETA2, eps: float = ADAMW_EPS,
               weight_decay: float = 0.0):
    """One AdamW step (Adam moments with bias correction, decoupled weight decay) on a
    parameter that Muon does not update.

    Scaling Muon for Diffusion Transformers (summary page, experimental setup): bias,
    normalisation and out-of-block parameters keep AdamW; an auxiliary AdamW group uses
    LR 1e-4.  Muon is Scalable for LLM Training (notes, section 2.2, "Matching update RMS
    of AdamW"): Muon and AdamW share the learning rate and weight decay.  The pages give
    no betas or epsilon; the reading here is the usual (0.9, 0.999, 1e-8).  t counts
    steps from 1.  Returns (p, m, v).
    """
    if t < 1:
        raise ValueError("t counts from 1")
    p = np.asarray(p, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    p = p - lr * (m_hat / (np.sqrt(v_hat) + eps) + weight_decay * p)
    return p, m, v
