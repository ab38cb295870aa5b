"""Pins for the fp64 oracle: each check ties it to something other than itself.

Sources of truth used here:
* values printed on the pages (tests/golden/pages_values.json, each cited);
* closed forms: Newton-Schulz acts on every singular value separately, so
  NS5(U diag(s) V^T) = U diag(g(s/||s||_2)) V^T with g the scalar quintic applied
  five times (the scalar map is written here from the printed coefficients);
* invariants: polar factor preserved, scale and transpose equivariance, unit
  lines after RowNorm, Lemma 1's update RMS;
* brute force with Python scalar loops on tiny inputs.

Each check takes the oracle module as an argument so that the mutation test at the
bottom can run the same checks against copies of the oracle with planted mistakes.
"""
import json
import math
import os
import types

import numpy as np
import pytest

from oracle import muon_ref

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_values.json")))
A_ = GOLDEN["ns_coefficients"]["a"]
B_ = GOLDEN["ns_coefficients"]["b"]
C_ = GOLDEN["ns_coefficients"]["c"]
N_ = GOLDEN["ns_steps"]["value"]


def g5(x):
    """The scalar quintic x -> a x + b x^3 + c x^5, applied N times (printed coefficients)."""
    x = np.asarray(x, dtype=np.float64)
    for _ in range(N_):
        x2 = x * x
        x = x * (A_ + x2 * (B_ + x2 * C_))
    return x


def rand_orth(rng, n, k):
    """n x k matrix with orthonormal columns (k <= n)."""
    q, r = np.linalg.qr(rng.standard_normal((n, k)))
    return q * np.sign(np.diag(r))[None, :]


def svd_built(rng, A, B, sigmas):
    k = min(A, B)
    U = rand_orth(rng, A, k)
    V = rand_orth(rng, B, k)
    return U, np.asarray(sigmas, dtype=np.float64), V


SHAPES = [(2, 3), (3, 2), (4, 4), (16, 64), (64, 16), (33, 17), (24, 40)]


# ---------------------------------------------------------------------------
# checks (take the oracle module)
# ---------------------------------------------------------------------------

def check_constants(o):
    assert o.NS_A == A_ and o.NS_B == B_ and o.NS_C == C_
    assert o.NS_STEPS == N_
    assert o.MU_DEFAULT == GOLDEN["momentum_mu"]["value"]
    assert o.RMS_MATCH == GOLDEN["rms_match"]["value"]
    assert o.K_DEFAULT == GOLDEN["periodic_K"]["value"]
    assert o.GAMMA_DEFAULT == GOLDEN["periodic_gamma"]["value"]


def check_ns5_closed_form(o):
    rng = np.random.default_rng(1)
    for (A, B) in SHAPES:
        k = min(A, B)
        sig = np.exp(rng.uniform(-3, 0, size=k))
        U, s, V = svd_built(rng, A, B, sig)
        M = (U * s[None, :]) @ V.T
        got = o.newton_schulz(M)
        want = (U * g5(s / np.linalg.norm(s))[None, :]) @ V.T
        err = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert err < 1e-11, (A, B, err)


def check_ns5_diagonal(o):
    for (A, B) in [(5, 9), (9, 5), (6, 6)]:
        d = np.linspace(0.1, 2.0, min(A, B))
        M = np.zeros((A, B))
        M[np.arange(len(d)), np.arange(len(d))] = d
        got = o.newton_schulz(M)
        want = np.zeros((A, B))
        want[np.arange(len(d)), np.arange(len(d))] = g5(d / np.sqrt(np.sum(d * d)))
        assert np.max(np.abs(got - want)) < 1e-12


def check_ns5_orthogonal_input(o):
    rng = np.random.default_rng(2)
    for (n, m) in [(8, 8), (8, 32), (32, 8), (16, 48)]:
        Q = rand_orth(rng, max(n, m), min(n, m))
        Q = Q.T if n < m else Q          # orthonormal along the short side
        got = o.newton_schulz(Q)
        want = g5(1.0 / math.sqrt(min(n, m))) * Q
        assert np.max(np.abs(got - want)) < 1e-12


def check_ns5_polar_and_band(o):
    rng = np.random.default_rng(3)
    for (A, B) in [(12, 20), (20, 12), (16, 16)]:
        k = min(A, B)
        sig = np.exp(rng.uniform(-2, 0, size=k))
        U, s, V = svd_built(rng, A, B, sig)
        M = (U * s[None, :]) @ V.T
        O = o.newton_schulz(M)
        P = U @ V.T
        Uo, so, Vto = np.linalg.svd(O, full_matrices=False)
        # polar factor preserved exactly (f > 0 for x > 0)
        assert np.max(np.abs(Uo @ Vto - P)) < 1e-9
        s0 = s / np.linalg.norm(s)
        assert np.all(s0 >= 3e-3)
        assert so.min() >= 0.68 and so.max() <= 1.21
        bound = np.max(np.abs(g5(s0) - 1.0))
        assert np.linalg.norm(O - P) / math.sqrt(k) <= bound + 1e-12


def check_ns5_short_side(o):
    """Tall input: short-side iteration equals Eq. (2) run literally on the long side."""
    rng = np.random.default_rng(4)
    M = rng.standard_normal((24, 7))
    X = M / math.sqrt(float(np.sum(M * M)))
    for _ in range(N_):
        P = [[sum(X[i][t] * X[j][t] for t in range(X.shape[1])) for j in range(X.shape[0])]
             for i in range(X.shape[0])]
        P = np.array(P)
        X = A_ * X + B_ * (P @ X) + C_ * (P @ (P @ X))
    assert np.max(np.abs(o.newton_schulz(M) - X)) < 1e-12
    assert np.max(np.abs(o.newton_schulz(M.T) - o.newton_schulz(M).T)) < 1e-13


def check_ns5_scale_and_zero(o):
    rng = np.random.default_rng(5)
    M = rng.standard_normal((6, 10))
    assert np.max(np.abs(o.newton_schulz(M) - o.newton_schulz(37.5 * M))) < 1e-12
    assert np.max(np.abs(o.newton_schulz(M) - o.newton_schulz(1e-9 * M))) < 1e-12
    Z = np.zeros((4, 7))
    assert np.array_equal(o.newton_schulz(Z), Z)


def check_rownorm_bruteforce(o):
    rng = np.random.default_rng(6)
    for (A, B) in [(3, 5), (5, 3), (4, 4), (1, 7), (7, 1)]:
        M = rng.standard_normal((A, B))
        M[0, :] = 0.0 if A <= B else M[0, :]
        if A > B:
            M[:, 0] = 0.0
        R = o.rownorm(M)
        want = [[0.0] * B for _ in range(A)]
        if A <= B:   # wide or square: rows
            for i in range(A):
                nrm = math.sqrt(sum(M[i][j] ** 2 for j in range(B)))
                for j in range(B):
                    want[i][j] = M[i][j] / nrm if nrm > 0 else 0.0
        else:        # tall: columns
            for j in range(B):
                nrm = math.sqrt(sum(M[i][j] ** 2 for i in range(A)))
                for i in range(A):
                    want[i][j] = M[i][j] / nrm if nrm > 0 else 0.0
        assert np.max(np.abs(R - np.array(want))) < 1e-15


def check_nonfinite_propagation(o):
    """NaN and Inf in the momentum: RowNorm divides every line by its norm as written
    (brute force with Python floats, whose division is IEEE's: x/inf = 0, inf/inf =
    nan, x/nan = nan); only an exactly zero line maps to zero.  NS5 of a matrix with
    one non-finite entry is NaN everywhere: X_0 has a non-finite entry, so X X^T has a
    non-finite row, and (X X^T)^2 carries it into every entry of B and of B X."""
    nan, inf = float("nan"), float("inf")
    for (A, B) in [(3, 6), (6, 3)]:
        rng = np.random.default_rng(11)
        M = rng.standard_normal((A, B))
        if A <= B:
            M[0, 2] = nan
            M[1, 4] = inf
            M[2, :] = 0.0
        else:
            M[2, 0] = nan
            M[4, 1] = -inf
            M[:, 2] = 0.0
        R = o.rownorm(M)
        want = [[0.0] * B for _ in range(A)]
        lines = range(A) if A <= B else range(B)
        for l in lines:
            cells = [(l, j) for j in range(B)] if A <= B else [(i, l) for i in range(A)]
            nrm = math.sqrt(sum(float(M[i][j]) ** 2 for i, j in cells))
            for i, j in cells:
                want[i][j] = float(M[i][j]) / nrm if nrm != 0.0 else 0.0
        want = np.array(want)
        assert np.array_equal(np.isnan(R), np.isnan(want))
        fin = ~np.isnan(want)
        assert np.max(np.abs(R[fin] - want[fin])) < 1e-15
        assert np.isnan(R).sum() == (B if A <= B else A) + 1   # the NaN line, and inf/inf
    for bad in (nan, inf, -inf):
        M = np.random.default_rng(12).standard_normal((5, 9))
        M[3, 7] = bad
        assert np.isnan(o.newton_schulz(M)).all()
        assert np.isnan(o.newton_schulz(M.T)).all()


def check_rownorm_invariants(o):
    rng = np.random.default_rng(7)
    for (A, B) in [(16, 64), (64, 16), (32, 32)]:
        M = rng.standard_normal((A, B))
        R = o.rownorm(M)
        axis = 1 if A <= B else 0
        assert np.max(np.abs(np.sqrt(np.sum(R * R, axis=axis)) - 1.0)) < 1e-12
        # Lemma-1-style RMS: n unit lines of length m -> RMS = 1/sqrt(m)
        assert abs(o.rms(R) - 1.0 / math.sqrt(max(A, B))) < 1e-12
        # scaled RowNorm update RMS is exactly 0.2*gamma
        s = o.update_scale(A, B, False, 0.15)
        assert abs(s * o.rms(R) - 0.2 * 0.15) < 1e-12


def check_lemma1(o):
    rng = np.random.default_rng(8)
    for (A, B) in [(16, 64), (64, 16), (32, 32), (10, 50)]:
        P = o.polar_factor(rng.standard_normal((A, B)))
        assert abs(o.rms(P) - math.sqrt(1.0 / max(A, B))) < 1e-12
        assert abs(o.update_scale(A, B, True, 0.15) * o.rms(P) - 0.2) < 1e-12


def check_momentum(o):
    rng = np.random.default_rng(9)
    G = rng.standard_normal((3, 4))
    M = np.zeros((3, 4))
    mu = 0.95
    for t in range(1, 8):
        M = o.momentum(M, G, mu)
        assert np.max(np.abs(M - G * (1 - mu ** t) / (1 - mu))) < 1e-13
    M0 = rng.standard_normal((2, 3))
    G1 = rng.standard_normal((2, 3))
    got = o.momentum(M0, G1, 0.9)
    for i in range(2):
        for j in range(3):
            assert got[i][j] == 0.9 * M0[i][j] + G1[i][j]


def check_apply(o):
    rng = np.random.default_rng(10)
    W = rng.standard_normal((3, 5))
    U = rng.standard_normal((3, 5))
    eta, lam, s = 0.02, 0.01, 1.7
    got = o.apply_update(W, U, s, eta, lam)
    for i in range(3):
        for j in range(5):
            assert abs(got[i][j] - (W[i][j] - eta * s * U[i][j] - eta * lam * W[i][j])) < 1e-15
    Wt = W.copy()
    for _ in range(10):
        Wt = o.apply_update(Wt, np.zeros_like(W), s, eta, lam)
    assert np.max(np.abs(Wt - W * (1 - eta * lam) ** 10)) < 1e-14


def check_scale(o):
    H = 1536
    ratio = o.update_scale(H, 4 * H, True, 0.15) / o.update_scale(H, H, True, 0.15)
    assert abs(ratio - GOLDEN["mlp_to_square_update_ratio"]["value"]) < 1e-12
    assert abs(o.update_scale(4 * H, H, True, 0.15) - 0.2 * math.sqrt(4 * H)) < 1e-12
    assert abs(o.update_scale(7, 3, False, 0.15) - 0.15 * 0.2 * math.sqrt(7)) < 1e-12


def check_schedule(o):
    def count(T, K):
        return sum(1 for s in range(T) if o.is_refresh(s, K))
    for K in (1, 2, 3, 4, 7):
        for T in range(0, 40):
            assert count(T, K) == -(-T // K)
    assert o.is_refresh(0, 3) and not o.is_refresh(1, 3) and not o.is_refresh(2, 3) and o.is_refresh(3, 3)
    T = 1200
    cut23 = 1 - count(T, 3) / count(T, 2)
    cut34 = 1 - count(T, 4) / count(T, 3)
    assert round(cut23, 2) == GOLDEN["ns5_count_cut_K2_to_K3"]["value"]
    assert round(cut34, 2) == GOLDEN["ns5_count_cut_K3_to_K4"]["value"]
    # refresh-only traffic at K=3 is one third of vanilla: cut of 66.7% (printed)
    assert round(1 - count(T, 3) / count(T, 1), 3) == GOLDEN["logical_comm_cut_K3"]["value"]
    v = GOLDEN["comm_volume_gib"]
    assert abs(v["periodic"] / v["naive"] - count(T, 3) / count(T, 1)) < 1e-3


def check_step(o):
    """Whole step against an independent assembly: SVD closed form or brute-force RowNorm."""
    rng = np.random.default_rng(11)
    for (A, B) in [(6, 10), (10, 6)]:
        W = 0.02 * rng.standard_normal((A, B))
        M = np.zeros((A, B))
        for step in range(4):
            G = rng.standard_normal((A, B)) * 1e-3
            Mn = 0.95 * M + G
            if step % 3 == 0:
                U_, s_, Vt_ = np.linalg.svd(Mn, full_matrices=False)
                D = (U_ * g5(s_ / np.linalg.norm(s_))[None, :]) @ Vt_
                sc = 0.2 * math.sqrt(max(A, B))
            else:
                ax = 1 if A <= B else 0
                D = Mn / np.sqrt(np.sum(Mn * Mn, axis=ax, keepdims=True))
                sc = 0.15 * 0.2 * math.sqrt(max(A, B))
            Wn = W - 0.02 * (sc * D + 0.01 * W)
            gW, gM, refresh = o.periodic_step(W, M, G, step, 3, 0.15, 0.95, 0.02, 0.01)
            assert refresh == (step % 3 == 0)
            assert np.max(np.abs(gM - Mn)) < 1e-15
            assert np.max(np.abs(gW - Wn)) < 1e-12
            W, M = Wn, Mn


def check_bf16_rounding(o):
    r = lambda v: float(o.round_to_storage(np.array([v]), "bf16")[0])
    assert r(1.0) == 1.0
    assert r(1.0 + 2.0 ** -8) == 1.0                       # tie -> even
    assert r(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6       # tie -> even (up)
    assert r(1.0 + 2.0 ** -8 + 2.0 ** -20) == 1.0 + 2.0 ** -7
    assert r(-3.0) == -3.0 and r(0.0) == 0.0
    assert r(255.5) == 256.0 and r(254.5) == 254.0
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(12)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(o.round_to_storage(x.astype(np.float64), "bf16"), want)


def check_update_norm(o):
    """Eq. (6): the applied direction has RMS exactly 0.2 (0.2*gamma on RowNorm steps),
    is a positive multiple of U, and on RowNorm steps without zero lines it equals Eq. (7)."""
    rng = np.random.default_rng(13)
    for (A, B) in [(12, 30), (30, 12), (16, 16)]:
        M = rng.standard_normal((A, B))
        O = o.newton_schulz(M)
        s = o.update_norm_scale(O, True, 0.15)
        assert abs(math.sqrt(float(np.mean((s * O) ** 2))) - 0.2) < 1e-12
        assert s > 0
        R = o.rownorm(M)
        s_r = o.update_norm_scale(R, False, 0.15)
        assert abs(s_r - 0.15 * 0.2 * math.sqrt(max(A, B))) < 1e-12
        W = rng.standard_normal((A, B))
        a = o.periodic_step(W, np.zeros((A, B)), M, 1, 3, scale_mode="update_norm")
        b = o.periodic_step(W, np.zeros((A, B)), M, 1, 3, scale_mode="adjusted_lr")
        assert np.max(np.abs(a[0] - b[0])) < 1e-12
        # refresh step: brute force W - eta*(0.2*O/RMS(O) + lam*W)
        c = o.periodic_step(W, np.zeros((A, B)), M, 0, 3, scale_mode="update_norm")
        r = math.sqrt(sum(O[i][j] ** 2 for i in range(A) for j in range(B)) / (A * B))
        for i in range(A):
            for j in range(B):
                assert abs(c[0][i][j] - (W[i][j] - 0.02 * (0.2 * O[i][j] / r + 0.01 * W[i][j]))) < 1e-12
    # a zero line carries no update; the RMS is over the remaining lines
    M = rng.standard_normal((5, 9))
    M[2, :] = 0.0
    R = o.rownorm(M)
    assert abs(o.update_norm_scale(R, False, 1.0) - 0.2 * 3.0) < 1e-12
    assert o.update_norm_scale(np.zeros((3, 4)), True, 0.15) == 0.0


def check_update_rms(o):
    rng = np.random.default_rng(14)
    for (A, B) in [(6, 11), (11, 6)]:
        M = rng.standard_normal((A, B))
        if A <= B:
            M[0, :] = 0.0
        else:
            M[:, 0] = 0.0
        R = o.rownorm(M)
        n_nz = min(A, B) - 1
        assert abs(o.update_rms(R) - math.sqrt(n_nz / (A * B))) < 1e-12
        W = rng.standard_normal((A, B))
        out = o.periodic_step(W, np.zeros((A, B)), M, 1, 3, telemetry=True)
        assert abs(out[3] - math.sqrt(n_nz / (A * B))) < 1e-12
        out = o.periodic_step(W, np.zeros((A, B)), M, 0, 3, telemetry=True)
        Uo = o.newton_schulz(M)
        assert abs(out[3] - math.sqrt(sum(Uo[i][j] ** 2 for i in range(A) for j in range(B)) / (A * B))) < 1e-12


def check_adamw(o):
    """AdamW against torch.optim.AdamW (a library routine, float64), a closed form of
    the first step, and a scalar brute-force loop."""
    rng = np.random.default_rng(15)
    p0 = rng.standard_normal(37)
    gs = [rng.standard_normal(37) * 10.0 ** rng.uniform(-4, 0) for _ in range(6)]
    lr, wd = 3e-3, 0.01
    torch = pytest.importorskip("torch")
    tp = torch.tensor(p0.copy(), dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([tp], lr=lr, betas=(0.9, 0.999), eps=1e-8, weight_decay=wd)
    p, m, v = p0.copy(), np.zeros(37), np.zeros(37)
    for t, g in enumerate(gs, start=1):
        tp.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        p, m, v = o.adamw_step(p, g, m, v, t, lr, weight_decay=wd)
        assert np.max(np.abs(p - tp.detach().numpy())) < 1e-12, t
    # first step: m_hat = g, v_hat = g^2, so the step is lr*(g/(|g|+eps) + wd*p)
    g = rng.standard_normal(9)
    q = rng.standard_normal(9)
    p1, m1, v1 = o.adamw_step(q, g, np.zeros(9), np.zeros(9), 1, 0.5, weight_decay=0.1)
    assert np.max(np.abs(p1 - (q - 0.5 * (g / (np.abs(g) + 1e-8) + 0.1 * q)))) < 1e-12
    assert np.max(np.abs(m1 - 0.1 * g)) < 1e-15 and np.max(np.abs(v1 - 0.001 * g * g)) < 1e-15
    # scalar brute force, third step with nonzero state
    pp, mm_, vv = 0.3, 0.02, 1e-4
    gg = -0.7
    b1, b2 = 0.9, 0.999
    m2 = b1 * mm_ + (1 - b1) * gg
    v2 = b2 * vv + (1 - b2) * gg * gg
    want = pp - 0.01 * ((m2 / (1 - b1 ** 3)) / (math.sqrt(v2 / (1 - b2 ** 3)) + 1e-8) + 0.05 * pp)
    got = o.adamw_step(np.array([pp]), np.array([gg]), np.array([mm_]), np.array([vv]), 3, 0.01,
                       weight_decay=0.05)[0][0]
    assert abs(got - want) < 1e-15
    assert o.ADAMW_AUX_LR == GOLDEN["adamw_aux_lr"]["value"]


ALL_CHECKS = [check_constants, check_ns5_closed_form, check_ns5_diagonal, check_ns5_orthogonal_input,
              check_ns5_polar_and_band, check_ns5_short_side, check_ns5_scale_and_zero,
              check_rownorm_bruteforce, check_nonfinite_propagation, check_rownorm_invariants, check_lemma1,
              check_momentum,
              check_apply, check_scale, check_schedule, check_step, check_bf16_rounding, check_update_norm,
              check_update_rms, check_adamw]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(muon_ref)


def test_quintic_fixed_points():
    """f(x) = x at x^2 = roots of c y^2 + b y + (a - 1) = 0; f(1) = a + b + c."""
    disc = B_ * B_ - 4 * C_ * (A_ - 1)
    ys = [(-B_ - math.sqrt(disc)) / (2 * C_), (-B_ + math.sqrt(disc)) / (2 * C_)]
    for y in ys:
        x = math.sqrt(y)
        assert abs(float(muon_ref.quintic(x)) - x) < 1e-12
    assert abs(float(muon_ref.quintic(1.0)) - (A_ + B_ + C_)) < 1e-15
    # no positive root of a + b y + c y^2: f(x) > 0 for every x > 0
    assert B_ * B_ - 4 * A_ * C_ < 0
    assert abs(float(muon_ref.quintic_iterated(0.3)) - float(g5(0.3))) < 1e-13


# ---------------------------------------------------------------------------
# mutation test: plant mistakes in a copy of the oracle; some pin must fail
# ---------------------------------------------------------------------------

MUTATIONS = [
    ("X = a * X + b * (XXt @ X) + c * ((XXt @ XXt) @ X)", "X = a * X + b * (XXt @ X)"),
    ("X = a * X + b * (XXt @ X) + c * ((XXt @ XXt) @ X)", "X = a * X - b * (XXt @ X) + c * ((XXt @ XXt) @ X)"),
    ("XXt = X @ X.T", "XXt = X.T @ X if X.shape[0] == X.shape[1] else X @ X.T"),
    ("for _ in range(steps):", "for _ in range(steps - 1):"),
    ("X = X / nrm", "X = X / np.linalg.norm(X, 2)"),
    ("return X.T.copy() if tall else X", "return X"),
    ("NS_B = -4.7750", "NS_B = -4.7705"),
    ("axis = 1 if A <= B else 0", "axis = 1"),
    ("    zero = norms == 0.0\n", "    zero = ~(norms > 0.0)\n"),
    ("axis = 1 if A <= B else 0", "axis = 1 if A < B else 0"),
    ("return mu * np.asarray(M_prev, dtype=np.float64) + np.asarray(G, dtype=np.float64)",
     "return np.asarray(M_prev, dtype=np.float64) + mu * np.asarray(G, dtype=np.float64)"),
    ("return W - eta * (scale * np.asarray(U, dtype=np.float64) + lam * W)",
     "return W - eta * (scale * np.asarray(U, dtype=np.float64) - lam * W)"),
    ("s = RMS_MATCH * math.sqrt(max(A, B))", "s = RMS_MATCH * math.sqrt(min(A, B))"),
    ("return s if refresh else gamma * s", "return s"),
    ("return step % K == 0", "return step % K == K - 1"),
    ("q = np.rint(np.ldexp(frac, 8))", "q = np.floor(np.ldexp(frac, 8) + 0.5)"),
    ("U = muon_direction(M, refresh)", "U = muon_direction(M_prev, refresh)"),
    ("    s = RMS_MATCH / r\n", "    s = RMS_MATCH * r\n"),
    ("    v = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g * g",
     "    v = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g"),
    ("    m_hat = m / (1.0 - beta1 ** t)", "    m_hat = m"),
    ("    p = p - lr * (m_hat / (np.sqrt(v_hat) + eps) + weight_decay * p)",
     "    p = p - lr * (m_hat / (np.sqrt(v_hat) + eps)) - weight_decay * p"),
    ("nz = int(np.count_nonzero(np.sqrt(np.sum(U * U, axis=line_axis)) > 0.0))", "nz = min(A, B)"),
    ("        r = rms(U)\n", "        r = math.sqrt(float(np.mean(np.abs(U))))\n"),
]


def _mutant(src, old, new):
    assert src.count(old) == 1, old
    mod = types.ModuleType("muon_ref_mutant")
    exec(compile(src.replace(old, new), "muon_ref_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("old,new", MUTATIONS)
def test_planted_mistake_is_caught(old, new):
    src = open(muon_ref.__file__).read()
    mod = _mutant(src, old, new)
    failed = []
    for chk in ALL_CHECKS:
        try:
            chk(mod)
        except (AssertionError, ValueError, IndexError):
            failed.append(chk.__name__)
    assert failed, f"no pin caught mutation {new!r}"
