"""GPU parity: every entry point of the C ABI against the fp64 oracle, element by
element on the same seeded inputs, at sizes spanning several tiles with ragged
tails, plus edge cases (empty, 1 x n, n x 1, zero lines, zero matrices)."""
import math

import numpy as np
import pytest
import torch

from oracle import muon_ref
from parity_util import (SCALES8, TOL_F32, TOL_NS5_BF16, TOL_NS5_F32, apply_terms, assert_bf16_close,
                         assert_bf16_within_ulp, assert_f32_close, check_implied_direction, dev, inputs, rel_fro,
                         to_dev, to_np)
from synth import gradient_np, quantize_np

pytestmark = pytest.mark.gpu

mm = pytest.importorskip("matrix_aware_optimizer_muon_gb300")

SHAPES_EW = [(256, 1024), (300, 1000), (1000, 300), (64, 128), (7, 13), (13, 7), (1, 1), (1, 517), (517, 1),
             (129, 129), (65, 130)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mm.load_library()
    torch.cuda.set_device(0)
    yield
    mm.muon_debug_set(0, 0)


def rand_M(shapes, seed=3, zero_line=False):
    rng = np.random.default_rng(seed)
    out = []
    for (a, b) in shapes:
        M = (rng.standard_normal((a, b)) * 1e-2).astype(np.float32)
        if zero_line and a > 2 and b > 2:
            if a <= b:
                M[1, :] = 0.0
            else:
                M[:, 1] = 0.0
        out.append(M)
    return out


# ---------------------------------------------------------------------------
# momentum and Frobenius norm
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("gdt", ["bf16", "f32"])
def test_momentum_parity(gdt):
    shapes = SHAPES_EW
    M0 = rand_M(shapes)
    _, Gs = inputs(shapes, "bf16", gdt, 1)
    G = [to_dev(g, gdt) for g in Gs[0]]
    M = [to_dev(m, "f32") for m in M0]
    ws = mm.alloc_workspace(shapes)
    fro = torch.full((len(shapes),), -1.0, device=dev())
    mm.muon_momentum(G, M, 0.95, fro, ws)
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        ref = muon_ref.momentum(M0[i], Gs[0][i], 0.95)
        assert_f32_close(to_np(M[i]), ref, what=f"M {shapes[i]}")
        want = float(np.sum(ref * ref))
        assert abs(float(fro[i]) - want) <= TOL_F32 * want, (shapes[i], float(fro[i]), want)
    # without the norm output (no workspace needed)
    M2 = [to_dev(m, "f32") for m in M0]
    mm.muon_momentum(G, M2, 0.9)
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        assert_f32_close(to_np(M2[i]), muon_ref.momentum(M0[i], Gs[0][i], 0.9), what="M mu=0.9")


def test_fro_norm_parity():
    shapes = SHAPES_EW + [(3, 40000)]
    M0 = rand_M(shapes, seed=4)
    M0[2][:] = 0.0
    M = [to_dev(m, "f32") for m in M0]
    ws = mm.alloc_workspace(shapes)
    out = torch.full((len(shapes),), -1.0, device=dev())
    mm.muon_fro_norm(M, out, ws)
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        want = muon_ref.frobenius_norm(M0[i])
        assert abs(float(out[i]) - want) <= TOL_F32 * max(want, 1e-30), shapes[i]


# ---------------------------------------------------------------------------
# RowNorm and apply
# ---------------------------------------------------------------------------
def test_rownorm_parity():
    shapes = SHAPES_EW + [(4, 20000), (20000, 4)]
    M0 = rand_M(shapes, seed=5, zero_line=True)
    M = [to_dev(m, "f32") for m in M0]
    R = [torch.full(s, 7.0, device=dev()) for s in shapes]
    ws = mm.alloc_workspace(shapes)
    mm.muon_rownorm(M, R, ws)
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        ref = muon_ref.rownorm(M0[i])
        assert_f32_close(to_np(R[i]), ref, what=f"R {shapes[i]}")
        assert np.array_equal(to_np(M[i]), M0[i].astype(np.float64))  # M untouched


@pytest.mark.parametrize("wdt,udt", [("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32"), ("f32", "bf16")])
def test_apply_parity(wdt, udt):
    shapes = SHAPES_EW
    W0, _ = inputs(shapes, wdt, "bf16", 0)
    rng = np.random.default_rng(6)
    U0 = [quantize_np((rng.standard_normal(s) * 0.05).astype(np.float32), udt) for s in shapes]
    W = [to_dev(w, wdt) for w in W0]
    U = [to_dev(u, udt) for u in U0]
    mm.muon_apply(W, U, 0.2, 0.02, 0.01)
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(shapes):
        s = 0.2 * math.sqrt(max(a, b))
        ref = muon_ref.apply_update(W0[i], U0[i], s, 0.02, 0.01)
        if wdt == "f32":
            assert_f32_close(to_np(W[i]), ref, what=f"W {shapes[i]}")
        else:
            assert_bf16_close(to_np(W[i]), ref, apply_terms(W0[i], U0[i], s, 0.02, 0.01), what=f"W {shapes[i]}")


# ---------------------------------------------------------------------------
# RowNorm step (fused momentum + RowNorm + apply), wide and tall, ragged
# ---------------------------------------------------------------------------
# Tall-matrix routes of a RowNorm step: the default two row-contiguous passes with
# the second re-reading M from L2, the single-pass cluster kernel, the plain two-pass kernels.
TALL_PATHS = {"l2pass": 0, "cluster": mm.MUON_DEBUG_TALL_CLUSTER, "two_pass": mm.MUON_DEBUG_NO_CLUSTER}


ROWNORM_CASES = [(dt, dt, path) for path in TALL_PATHS for dt in ("bf16", "f32")] + \
    [("bf16", "f32", "l2pass"), ("f32", "bf16", "l2pass")]


@pytest.mark.parametrize("wdt,gdt,path", ROWNORM_CASES)
def test_rownorm_step_parity(wdt, gdt, path):
    """Wide rows (single pass) and tall columns on each tall route, ragged and degenerate
    shapes.  For the L2 two-pass kernel: (4608, 1536) has 12 column blocks x 36 row blocks
    (more chunks than the pass-2 lag), the two (1000, 300) share one launch with a ragged
    last column block and row block, (40000, 8) has 313 row blocks.  For the cluster
    kernel (40000, 8) takes 16-column strips and (70000, 8) is too tall for its shared
    memory.  (13, 7) and (517, 1) have B % 4 != 0 and take the plain two-pass kernels.
    Rows of 6145..12288 columns take the 512-thread launch unless W and G are both fp32:
    (5, 10240) five whole chunks per thread, (3, 8196) one thread busy in the fifth chunk
    round, (2, 12288) six whole chunks, (3, 11000) a part-filled sixth round, (4, 9999) the
    element-load kernel; with fp32 W and G the widths above 8192 keep the 3-chunk launch."""
    shapes = [(256, 1024), (300, 1000), (1000, 300), (1536, 1536), (7, 13), (13, 7), (1, 517), (517, 1),
              (3, 20000), (129, 129), (4608, 1536), (300, 36), (40000, 8), (70000, 8), (33, 4), (1000, 300),
              (5, 10240), (3, 8196), (2, 12288), (3, 11000), (4, 9999)]
    W0, Gs = inputs(shapes, wdt, gdt, 2)
    M0 = rand_M(shapes, seed=8, zero_line=True)
    W = [to_dev(w, wdt) for w in W0]
    M = [to_dev(m, "f32") for m in M0]
    G = [to_dev(g, gdt) for g in Gs[1]]
    ws = mm.alloc_workspace(shapes)
    mm.muon_debug_set(TALL_PATHS[path], 0)
    try:
        br = mm.muon_periodic_step(W, G, M, 1, ws, K=3)
    finally:
        mm.muon_debug_set(0, 0)
    assert br == mm.MUON_BRANCH_ROWNORM
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        refW, refM, refresh = muon_ref.periodic_step(W0[i], M0[i], Gs[1][i], 1, 3, 0.15, 0.95, 0.02, 0.01)
        assert not refresh
        assert_f32_close(to_np(M[i]), refM, what=f"M {shapes[i]}")
        if wdt == "f32":
            assert_f32_close(to_np(W[i]), refW, what=f"W {shapes[i]}")
        else:
            a, b = shapes[i]
            terms = apply_terms(W0[i], muon_ref.rownorm(refM), muon_ref.update_scale(a, b, False, 0.15), 0.02, 0.01)
            assert_bf16_close(to_np(W[i]), refW, terms, what=f"W {shapes[i]}")
    assert mm.muon_check_status(ws) == mm.MUON_OK


# ---------------------------------------------------------------------------
# Newton-Schulz
# ---------------------------------------------------------------------------
NS_SHAPES = [(256, 1024), (1024, 256), (300, 1000), (1000, 300), (520, 1100), (384, 384), (130, 2000),
             (33, 100), (100, 33), (1, 64), (64, 1), (8, 8)]


def mixed_momentum(shape, steps, seed=0):
    a, b = shape
    M = np.zeros((a, b))
    for t in range(steps):
        M = 0.95 * M + quantize_np(gradient_np(a, b, SCALES8, seed, 0, t), "bf16")
    return M.astype(np.float32)


@pytest.mark.parametrize("mode,tol", [("bf16", TOL_NS5_BF16), ("f32", TOL_NS5_F32)])
@pytest.mark.parametrize("steps", [1, 4])
def test_ns5_parity(mode, tol, steps):
    shapes = NS_SHAPES
    M0 = [mixed_momentum(s, steps, seed=i) for i, s in enumerate(shapes)]
    M = [to_dev(m, "f32") for m in M0]
    odt = torch.bfloat16 if mode == "bf16" else torch.float32
    O = [torch.full(s, 9.0, device=dev(), dtype=odt) for s in shapes]
    ws = mm.alloc_workspace(shapes, mode)
    mm.muon_ns5_batched(M, O, ws, ns5_mode=mode)
    torch.cuda.synchronize()
    assert mm.muon_check_status(ws) == mm.MUON_OK
    worst = {}
    for i in range(len(shapes)):
        ref = muon_ref.newton_schulz(M0[i].astype(np.float64))
        err = rel_fro(to_np(O[i]), ref)
        worst[shapes[i]] = err
        assert err <= tol, (shapes[i], err)
        # the bf16 path keeps a*X in higher precision in the early iterations (fp32 M,
        # then the bf16 residual of X); on matrices spanning several tiles that holds
        # its error at 4e-3 to 6.5e-3 measured (a CPU emulation of the same rounding
        # points predicts 3.4e-3 to 4.7e-3 before O's own bf16 rounding); without the
        # residual it would be 1e-2 to 2e-2.  Degenerate 1 x n, n x 1 and 8 x 8
        # inputs sit near 1.1e-2 to 1.7e-2.
        if mode == "bf16" and min(shapes[i]) >= 128:
            assert err <= 8e-3, (shapes[i], err)
        assert np.array_equal(to_np(M[i]), M0[i].astype(np.float64))
    print(f"ns5 {mode} steps={steps}: " + ", ".join(f"{k[0]}x{k[1]} {v:.2e}" for k, v in worst.items()))


@pytest.mark.parametrize("steps", [1, 4])
def test_ns5_one_cta_tiles_parity(steps):
    """The one-CTA form of the tensor-core GEMMs (128 x 256 tiles, selected by a test
    hook; the default runs 2-CTA clusters with tcgen05 cta_group::2 on 256 x 256 tiles)
    against the oracle, on the shapes of the default-form test above: ragged n (300,
    520, 130: a pair tile whose second CTA is partly or wholly past the last row), n <
    128, tall and wide."""
    shapes = NS_SHAPES
    M0 = [mixed_momentum(s, steps, seed=i) for i, s in enumerate(shapes)]
    M = [to_dev(m, "f32") for m in M0]
    O = [torch.full(s, 9.0, device=dev(), dtype=torch.bfloat16) for s in shapes]
    ws = mm.alloc_workspace(shapes)
    mm.muon_debug_set(mm.MUON_DEBUG_NO_PAIR, 0)
    try:
        mm.muon_ns5_batched(M, O, ws)
    finally:
        mm.muon_debug_set(0, 0)
    torch.cuda.synchronize()
    assert mm.muon_check_status(ws) == mm.MUON_OK
    for i in range(len(shapes)):
        err = rel_fro(to_np(O[i]), muon_ref.newton_schulz(M0[i].astype(np.float64)))
        assert err <= TOL_NS5_BF16, (shapes[i], err)
        if min(shapes[i]) >= 128:
            assert err <= 8e-3, (shapes[i], err)


def test_ns5_zero_matrix_and_scale_invariance():
    shapes = [(64, 128), (128, 64), (300, 1000)]
    M0 = [np.zeros(shapes[0], np.float32), mixed_momentum(shapes[1], 1), mixed_momentum(shapes[2], 1)]
    M1 = [m * np.float32(64.0) for m in M0]   # exact power-of-two scaling
    O0 = [torch.empty(s, device=dev(), dtype=torch.bfloat16) for s in shapes]
    O1 = [torch.empty(s, device=dev(), dtype=torch.bfloat16) for s in shapes]
    ws = mm.alloc_workspace(shapes)
    mm.muon_ns5_batched([to_dev(m, "f32") for m in M0], O0, ws)
    mm.muon_ns5_batched([to_dev(m, "f32") for m in M1], O1, ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(O0[0]).item() == 0
    for i in (1, 2):
        assert torch.equal(O0[i], O1[i]), "NS5 must be invariant to a power-of-two scale of M"


# ---------------------------------------------------------------------------
# whole refresh step with the apply fused into the last GEMM
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dt,mode", [("bf16", "bf16"), ("f32", "f32"), ("bf16", "f32"), ("f32", "bf16")])
def test_refresh_step_parity(dt, mode):
    shapes = [(256, 1024), (1024, 256), (300, 1000), (1000, 300), (129, 129), (33, 100)]
    W0, Gs = inputs(shapes, dt, dt, 1)
    M0 = [mixed_momentum(s, 3, seed=10 + i) for i, s in enumerate(shapes)]
    W = [to_dev(w, dt) for w in W0]
    M = [to_dev(m, "f32") for m in M0]
    G = [to_dev(g, dt) for g in Gs[0]]
    ws = mm.alloc_workspace(shapes, mode)
    br = mm.muon_periodic_step(W, G, M, 3, ws, K=3, ns5_mode=mode)
    assert br == mm.MUON_BRANCH_NS5
    torch.cuda.synchronize()
    tol = TOL_NS5_BF16 if mode == "bf16" else TOL_NS5_F32
    for i, (a, b) in enumerate(shapes):
        refW, refM, refresh = muon_ref.periodic_step(W0[i], M0[i], Gs[0][i], 3, 3, 0.15, 0.95, 0.02, 0.01)
        assert refresh
        assert_f32_close(to_np(M[i]), refM, what=f"M {shapes[i]}")
        dW = refW - W0[i]
        got = to_np(W[i])
        # update error within the NS5 tolerance, plus the storage rounding of W
        ulp = 2.0 ** -23 if dt == "f32" else 2.0 ** -7
        round_budget = np.linalg.norm(np.abs(refW)) * ulp
        assert np.linalg.norm(got - refW) <= tol * np.linalg.norm(dW) + round_budget, shapes[i]


@pytest.mark.parametrize("eta", [0.02, 1.0])
def test_refresh_step_bf16_w_implied_direction(eta):
    """The fused apply of the last UPDATE on bf16 W, checked through the direction it
    applied: O = (W_prev*(1 - eta*lam) - W_new)/(eta*0.2*sqrt(max(A, B))) against the
    oracle's NS5 output within the NS5 tolerance plus half a bf16 ulp of W_new per
    element.  At eta = 1 the update dominates W and the rounding budget is small, so
    the bound pins O itself.  Shapes cover each store branch of the epilogue: wide rows
    with 32-byte vectors (256 x 1024), 16-byte vectors (300 x 1000), element stores
    (520 x 1100, 129 x 129, 33 x 100), and tall matrices stored transposed."""
    shapes = [(256, 1024), (1024, 256), (300, 1000), (1000, 300), (520, 1100), (1100, 520), (129, 129), (33, 100)]
    W0, Gs = inputs(shapes, "bf16", "bf16", 1, seed=4)
    M0 = [mixed_momentum(s, 3, seed=20 + i) for i, s in enumerate(shapes)]
    W = [to_dev(w, "bf16") for w in W0]
    M = [to_dev(m, "f32") for m in M0]
    G = [to_dev(g, "bf16") for g in Gs[0]]
    ws = mm.alloc_workspace(shapes)
    assert mm.muon_periodic_step(W, G, M, 0, ws, K=3, eta=eta) == mm.MUON_BRANCH_NS5
    torch.cuda.synchronize()
    errs = {}
    for i, (a, b) in enumerate(shapes):
        refW64, refM, _ = muon_ref.periodic_step(W0[i], M0[i], Gs[0][i], 0, 3, 0.15, 0.95, eta, 0.01, w_dtype="f64")
        assert_f32_close(to_np(M[i]), refM, what=f"M {shapes[i]}")
        s = muon_ref.update_scale(a, b, True, 0.15)
        errs[shapes[i]] = check_implied_direction(to_np(W[i]), W0[i], refW64, eta, 0.01, s, TOL_NS5_BF16,
                                                  what=str(shapes[i]))
    print(f"eta={eta}: " + ", ".join(f"{k[0]}x{k[1]} {v:.2e}" for k, v in errs.items()))


# Shape groups (same short and long side) beyond the 8 one Newton-Schulz launch
# takes, and a group beyond the 512 matrices of one launch table.
MANY_GROUP_SHAPES = [(32, 64), (48, 80), (64, 96), (72, 200), (96, 96), (100, 300), (300, 100), (130, 260),
                     (128, 512), (200, 330), (256, 384), (40, 1000)] + [(8, 16)] * 515 + [(16, 8)] * 5


def test_ns5_more_groups_and_matrices_than_one_launch_takes():
    shapes = MANY_GROUP_SHAPES
    M0 = [mixed_momentum(s, 2, seed=i) for i, s in enumerate(shapes)]
    M = [to_dev(m, "f32") for m in M0]
    O = [torch.full(s, 9.0, device=dev(), dtype=torch.bfloat16) for s in shapes]
    ws = mm.alloc_workspace(shapes)
    mm.muon_ns5_batched(M, O, ws)
    torch.cuda.synchronize()
    assert mm.muon_check_status(ws) == mm.MUON_OK
    for i, s in enumerate(shapes):
        err = rel_fro(to_np(O[i]), muon_ref.newton_schulz(M0[i].astype(np.float64)))
        assert err <= TOL_NS5_BF16, (i, s, err)


@pytest.mark.parametrize("mode", ["bf16", "f32"])
def test_refresh_step_more_groups_and_matrices_than_one_launch_takes(mode):
    shapes = MANY_GROUP_SHAPES
    W0, Gs = inputs(shapes, "f32", "f32", 1, seed=7)
    M0 = [mixed_momentum(s, 2, seed=100 + i) for i, s in enumerate(shapes)]
    W = [to_dev(w, "f32") for w in W0]
    M = [to_dev(m, "f32") for m in M0]
    G = [to_dev(g, "f32") for g in Gs[0]]
    ws = mm.alloc_workspace(shapes, mode)
    assert mm.muon_periodic_step(W, G, M, 3, ws, K=3, ns5_mode=mode) == mm.MUON_BRANCH_NS5
    torch.cuda.synchronize()
    assert mm.muon_check_status(ws) == mm.MUON_OK
    tol = TOL_NS5_BF16 if mode == "bf16" else TOL_NS5_F32
    for i, (a, b) in enumerate(shapes):
        refW64, refM, _ = muon_ref.periodic_step(W0[i], M0[i], Gs[0][i], 3, 3, 0.15, 0.95, 0.02, 0.01, w_dtype="f64")
        assert_f32_close(to_np(M[i]), refM, what=f"M {i} {shapes[i]}")
        check_implied_direction(to_np(W[i]), W0[i], refW64, 0.02, 0.01, muon_ref.update_scale(a, b, True, 0.15),
                                tol, what=f"{i} {shapes[i]}")


# ---------------------------------------------------------------------------
# schedule, determinism, resume, vanilla Muon
# ---------------------------------------------------------------------------
def run_steps(shapes, dt, steps, K=3, mode="bf16", start_state=None, start_step=0, seed=0, buckets=None):
    """buckets: [(first, end)] runs of the matrix list, each taken by its own call."""
    W0, Gs = inputs(shapes, dt, dt, start_step + steps, seed=seed)
    if start_state is None:
        W = [to_dev(w, dt) for w in W0]
        M = [torch.zeros(s, device=dev()) for s in shapes]
    else:
        W, M = [w.clone() for w in start_state[0]], [m.clone() for m in start_state[1]]
    ws = mm.alloc_workspace(shapes, mode)
    branches = []
    for t in range(start_step, start_step + steps):
        G = [to_dev(g, dt) for g in Gs[t]]
        if buckets is None:
            branches.append(mm.muon_periodic_step(W, G, M, t, ws, K=K, ns5_mode=mode))
        else:
            brs = {mm.muon_periodic_step(W[a:b], G[a:b], M[a:b], t, ws, K=K, ns5_mode=mode) for a, b in buckets}
            assert len(brs) == 1
            branches.append(brs.pop())
    torch.cuda.synchronize()
    assert mm.muon_check_status(ws) == mm.MUON_OK
    return W, M, branches


def test_determinism_bit_exact():
    shapes = [(300, 1000), (1000, 300), (256, 256)]
    W1, M1, b1 = run_steps(shapes, "bf16", 4)
    W2, M2, b2 = run_steps(shapes, "bf16", 4)
    assert b1 == b2 == [1, 0, 0, 1]
    for a, b in zip(W1 + M1, W2 + M2):
        assert torch.equal(a, b)


@pytest.mark.parametrize("mode", ["bf16", "f32"])
def test_bucketed_calls_match_one_call(mode):
    """A step taken in buckets of consecutive matrices (one call each, one workspace, as
    the end-to-end benchmark streams them) is bit-identical to one call over all: every
    matrix's arithmetic is its own, whatever else shares the launches."""
    shapes = [(300, 1000), (1000, 300), (256, 256), (40, 520), (520, 40), (1, 300), (384, 1280), (1280, 384)]
    Wa, Ma, ba = run_steps(shapes, "bf16", 4, mode=mode)
    Wb, Mb, bb = run_steps(shapes, "bf16", 4, mode=mode, buckets=[(0, 3), (3, 4), (4, 8)])
    assert ba == bb == [1, 0, 0, 1]
    for a, b in zip(Wa + Ma, Wb + Mb):
        assert torch.equal(a, b)


def test_resume_bit_exact():
    shapes = [(300, 1000), (1000, 300)]
    Wa, Ma, _ = run_steps(shapes, "bf16", 6)
    Wb, Mb, _ = run_steps(shapes, "bf16", 3)
    state = ([w.cpu().clone() for w in Wb], [m.cpu().clone() for m in Mb])   # checkpoint to host
    state = ([w.to(dev()) for w in state[0]], [m.to(dev()) for m in state[1]])
    Wc, Mc, br = run_steps(shapes, "bf16", 3, start_state=state, start_step=3)
    assert br == [1, 0, 0]
    for a, b in zip(Wa + Ma, Wc + Mc):
        assert torch.equal(a, b)


def test_vanilla_K1_every_step_refreshes():
    shapes = [(64, 256), (256, 64)]
    _, _, br = run_steps(shapes, "bf16", 4, K=1)
    assert br == [1, 1, 1, 1]


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------
def test_empty_and_degenerate():
    assert mm.muon_periodic_step([], [], [], 0, torch.empty(256, dtype=torch.uint8, device=dev())) == 1
    shapes = [(0, 16), (16, 0), (1, 1), (1, 300), (300, 1)]
    W0, Gs = inputs(shapes, "bf16", "bf16", 2)
    W = [to_dev(w, "bf16") for w in W0]
    M = [torch.zeros(s, device=dev()) for s in shapes]
    ws = mm.alloc_workspace(shapes)
    refW = [w.astype(np.float64) for w in W0]
    refM = [np.zeros(s) for s in shapes]
    for t in range(2):
        G = [to_dev(g, "bf16") for g in Gs[t]]
        mm.muon_periodic_step(W, G, M, t, ws)
        for i in range(len(shapes)):
            refW[i], refM[i], _ = muon_ref.periodic_step(refW[i], refM[i], Gs[t][i], t, w_dtype="bf16")
    torch.cuda.synchronize()
    for i, s in enumerate(shapes):
        if 0 in s:
            continue
        assert_f32_close(to_np(M[i]), refM[i], what=f"M {s}")
        # a 1 x n or n x 1 matrix: NS5 of a rank-1 input, RowNorm of one line
        assert np.linalg.norm(to_np(W[i]) - refW[i]) <= 3e-2 * np.linalg.norm(refW[i] - W0[i]) + \
            np.linalg.norm(np.abs(refW[i])) * 2.0 ** -8, s


def test_zero_gradient_is_pure_weight_decay():
    shapes = [(64, 128), (128, 64)]
    W0, _ = inputs(shapes, "f32", "f32", 0)
    W = [to_dev(w, "f32") for w in W0]
    M = [torch.zeros(s, device=dev()) for s in shapes]
    G = [torch.zeros(s, device=dev()) for s in shapes]
    ws = mm.alloc_workspace(shapes, "f32")
    for t in range(3):
        mm.muon_periodic_step(W, G, M, t, ws, ns5_mode="f32")
    torch.cuda.synchronize()
    for i in range(2):
        assert_f32_close(to_np(W[i]), W0[i] * (1 - 0.02 * 0.01) ** 3, what="decay")


def test_misaligned_views_take_the_scalar_path():
    """Row length not a multiple of 4 and a base offset by one element.

    Teacher-forced: before each step the GPU state is set to the oracle's state."""
    shape = (37, 53)
    n = shape[0] * shape[1]
    base_w = torch.zeros(1 + n, dtype=torch.bfloat16, device=dev())
    base_g = torch.zeros(1 + n, dtype=torch.bfloat16, device=dev())
    base_m = torch.zeros(1 + n, dtype=torch.float32, device=dev())
    W0, Gs = inputs([shape], "bf16", "bf16", 3)
    W, G, M = base_w[1:].view(shape), base_g[1:].view(shape), base_m[1:].view(shape)
    ws = mm.alloc_workspace([shape])
    refW, refM = W0[0].astype(np.float64), np.zeros(shape)
    for t in range(3):
        W.copy_(to_dev(refW.astype(np.float32), "bf16"))
        M.copy_(to_dev(refM.astype(np.float32), "f32"))
        G.copy_(to_dev(Gs[t][0], "bf16"))
        mm.muon_periodic_step([W], [G], [M], t, ws)
        prevW = refW
        refW, refM, refresh = muon_ref.periodic_step(refW, refM.astype(np.float32), Gs[t][0], t, w_dtype="bf16")
        torch.cuda.synchronize()
        assert_f32_close(to_np(M), refM, what=f"M step {t}")
        if refresh:
            assert np.linalg.norm(to_np(W) - refW) <= TOL_NS5_BF16 * np.linalg.norm(refW - prevW) + \
                np.linalg.norm(np.abs(refW)) * 2.0 ** -8
        else:
            U = muon_ref.rownorm(refM)
            sc = muon_ref.update_scale(*shape, False, 0.15)
            assert_bf16_close(to_np(W), muon_ref.apply_update(prevW, U, sc, 0.02, 0.01),
                              apply_terms(prevW, U, sc, 0.02, 0.01), what=f"W step {t}")
    assert mm.muon_check_status(ws) == mm.MUON_OK


# ---------------------------------------------------------------------------
# device-side bounded waits: an expired wait is reported, the context survives
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("pair", [0, 1])
def test_stalled_producer_times_out_and_context_survives(pair):
    """The load warp(s) issue nothing: every consumer's bounded wait expires (in the
    2-CTA form, on both CTAs of each pair), the status reads MUON_ERR_TIMEOUT, and the
    next call on the same context is exact."""
    shapes = [(256, 512)]
    M = [to_dev(mixed_momentum(shapes[0], 1), "f32")]
    O = [torch.empty(shapes[0], device=dev(), dtype=torch.bfloat16)]
    ws = mm.alloc_workspace(shapes)
    flags = 0 if pair else mm.MUON_DEBUG_NO_PAIR
    mm.muon_debug_set(mm.MUON_DEBUG_STALL_PRODUCER | flags, 50)
    try:
        mm.muon_ns5_batched(M, O, ws)
        assert mm.muon_check_status(ws) == mm.MUON_ERR_TIMEOUT
    finally:
        mm.muon_debug_set(0, 0)
    # the status word was cleared and the context still works
    mm.muon_debug_set(flags, 0)
    try:
        mm.muon_ns5_batched(M, O, ws)
    finally:
        mm.muon_debug_set(0, 0)
    assert mm.muon_check_status(ws) == mm.MUON_OK
    ref = muon_ref.newton_schulz(to_np(M[0]))
    assert rel_fro(to_np(O[0]), ref) <= TOL_NS5_BF16


def test_tall_pass2_wait_times_out_and_context_survives():
    """The tall-matrix kernel publishes no column norms under the stall hook: its pass-2
    waits expire, the status word reports it, and the next step on the same context is exact."""
    shapes = [(1000, 300), (4608, 1536)]
    W0, Gs = inputs(shapes, "bf16", "bf16", 2)
    M0 = rand_M(shapes, seed=14)
    W = [to_dev(w, "bf16") for w in W0]
    M = [to_dev(m, "f32") for m in M0]
    G = [to_dev(g, "bf16") for g in Gs[1]]
    ws = mm.alloc_workspace(shapes)
    mm.muon_debug_set(mm.MUON_DEBUG_STALL_PRODUCER, 50)
    try:
        mm.muon_periodic_step(W, G, M, 1, ws)
        assert mm.muon_check_status(ws) == mm.MUON_ERR_TIMEOUT
    finally:
        mm.muon_debug_set(0, 0)
    W = [to_dev(w, "bf16") for w in W0]
    M = [to_dev(m, "f32") for m in M0]
    mm.muon_periodic_step(W, G, M, 1, ws)
    assert mm.muon_check_status(ws) == mm.MUON_OK
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(shapes):
        refW, refM, _ = muon_ref.periodic_step(W0[i], M0[i], Gs[1][i], 1, 3, 0.15, 0.95, 0.02, 0.01)
        assert_f32_close(to_np(M[i]), refM, what=f"M {shapes[i]}")
        terms = apply_terms(W0[i], muon_ref.rownorm(refM), muon_ref.update_scale(a, b, False, 0.15), 0.02, 0.01)
        assert_bf16_close(to_np(W[i]), refW, terms, what=f"W {shapes[i]}")


def test_tall_matrices_spanning_several_launches():
    """130 tall matrices of one shape take two launches of the tall-matrix kernel (at most
    128 per launch), reusing its control words; each matrix has two ragged row tiles."""
    shapes = [(260, 8)] * 130 + [(520, 12)] * 2
    W0, Gs = inputs(shapes, "bf16", "bf16", 2)
    M0 = rand_M(shapes, seed=15)
    runs = []
    for _ in range(2):
        W = [to_dev(w, "bf16") for w in W0]
        M = [to_dev(m, "f32") for m in M0]
        G = [to_dev(g, "bf16") for g in Gs[1]]
        ws = mm.alloc_workspace(shapes)
        mm.muon_periodic_step(W, G, M, 1, ws)
        assert mm.muon_check_status(ws) == mm.MUON_OK
        torch.cuda.synchronize()
        runs.append((W, M))
    W, M = runs[0]
    for i, (a, b) in enumerate(shapes):
        refW, refM, _ = muon_ref.periodic_step(W0[i], M0[i], Gs[1][i], 1, 3, 0.15, 0.95, 0.02, 0.01)
        assert_f32_close(to_np(M[i]), refM, what=f"M {i}")
        terms = apply_terms(W0[i], muon_ref.rownorm(refM), muon_ref.update_scale(a, b, False, 0.15), 0.02, 0.01)
        assert_bf16_close(to_np(W[i]), refW, terms, what=f"W {i}")
    for x, y in zip(runs[0][0] + runs[0][1], runs[1][0] + runs[1][1]):
        assert torch.equal(x, y)


def test_rownorm_overlap_matches_serial():
    """Wide-row kernels on the library's second stream give the same bits as running serially."""
    shapes = [(1536, 1536), (1536, 6144), (4608, 1536), (6144, 1536), (300, 1000), (1000, 300)]
    W0, Gs = inputs(shapes, "bf16", "bf16", 2)
    M0 = rand_M(shapes, seed=12)
    outs = []
    for flag in (0, mm.MUON_DEBUG_NO_OVERLAP):
        W = [to_dev(w, "bf16") for w in W0]
        M = [to_dev(m, "f32") for m in M0]
        G = [to_dev(g, "bf16") for g in Gs[1]]
        ws = mm.alloc_workspace(shapes)
        mm.muon_debug_set(flag, 0)
        try:
            mm.muon_periodic_step(W, G, M, 1, ws)
        finally:
            mm.muon_debug_set(0, 0)
        torch.cuda.synchronize()
        outs.append((W, M))
    for a, b in zip(outs[0][0] + outs[0][1], outs[1][0] + outs[1][1]):
        assert torch.equal(a, b)


def test_cuda_graph_capture_matches_eager():
    """Both branches captured into CUDA graphs (no allocation, no synchronisation inside
    the calls) replay to the same bits as eager calls."""
    shapes = [(1536, 1536), (1536, 6144), (4608, 1536), (300, 1000), (1000, 300)]
    W0, Gs = inputs(shapes, "bf16", "bf16", 3)
    M0 = rand_M(shapes, seed=13)

    def fresh():
        return ([to_dev(w, "bf16") for w in W0], [to_dev(m, "f32") for m in M0])

    G = [to_dev(g, "bf16") for g in Gs[0]]
    ws = mm.alloc_workspace(shapes)
    # eager reference: a refresh step then a RowNorm step
    We, Me = fresh()
    mm.muon_periodic_step(We, G, Me, 0, ws)
    mm.muon_periodic_step(We, G, Me, 1, ws)
    torch.cuda.synchronize()
    # captured: the same two steps as two graphs
    Wg, Mg = fresh()
    Wc, Mc = fresh()      # scratch copies used while capturing (capture does not execute)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graphs = []
    for step in (0, 1):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            mm.muon_periodic_step(Wg, G, Mg, step, ws)
        graphs.append(g)
    torch.cuda.synchronize()
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    assert mm.muon_check_status(ws) == mm.MUON_OK
    for a, b in zip(We + Me, Wg + Mg):
        assert torch.equal(a, b)


# ---------------------------------------------------------------------------
# Eq. (6) Update Norm and update-RMS telemetry
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dt,mode", [("bf16", "bf16"), ("f32", "f32")])
def test_update_norm_refresh_step_parity(dt, mode):
    # (1000, 296) is tall with 8-aligned rows: the vectorised apply with ragged tiles;
    # (1000, 300), (129, 129) and (33, 100) take the element-wise apply
    shapes = [(256, 1024), (1024, 256), (300, 1000), (1000, 300), (129, 129), (33, 100), (1000, 296)]
    W0, Gs = inputs(shapes, dt, dt, 1)
    M0 = [mixed_momentum(s, 3, seed=20 + i) for i, s in enumerate(shapes)]
    W = [to_dev(w, dt) for w in W0]
    M = [to_dev(m, "f32") for m in M0]
    G = [to_dev(g, dt) for g in Gs[0]]
    ws = mm.alloc_workspace(shapes, mode)
    rms = torch.full((len(shapes),), -1.0, device=dev())
    br = mm.muon_periodic_step(W, G, M, 3, ws, K=3, ns5_mode=mode, scale_mode="update_norm", update_rms=rms)
    assert br == mm.MUON_BRANCH_NS5
    torch.cuda.synchronize()
    assert mm.muon_check_status(ws) == mm.MUON_OK
    tol = TOL_NS5_BF16 if mode == "bf16" else TOL_NS5_F32
    for i, (a, b) in enumerate(shapes):
        refW, refM, refresh, refrms = muon_ref.periodic_step(W0[i], M0[i], Gs[0][i], 3, 3, 0.15, 0.95, 0.02, 0.01,
                                                             scale_mode="update_norm", telemetry=True)
        assert refresh
        assert_f32_close(to_np(M[i]), refM, what=f"M {shapes[i]}")
        ulp = 2.0 ** -23 if dt == "f32" else 2.0 ** -7
        dW = refW - W0[i]
        assert np.linalg.norm(to_np(W[i]) - refW) <= tol * np.linalg.norm(dW) + np.linalg.norm(np.abs(refW)) * ulp, \
            shapes[i]
        assert abs(float(rms[i]) - refrms) <= tol * refrms, (shapes[i], float(rms[i]), refrms)
        # Eq. (6): the applied direction has RMS 0.2 exactly -> |dW + eta*lam*W| has RMS eta*0.2
        got_dir = (to_np(W[i]) - W0[i] * (1 - 0.02 * 0.01)) / -0.02
        assert abs(muon_ref.rms(got_dir) - 0.2) <= tol * 0.2 + np.linalg.norm(np.abs(refW)) * ulp / 0.02 / math.sqrt(a * b)


@pytest.mark.parametrize("path", list(TALL_PATHS))
def test_update_rms_telemetry(path):
    # (3, 10240) counts its nonzero rows in the 512-thread wide-row kernel
    shapes = [(256, 1024), (1000, 300), (4608, 1536), (1536, 6144), (300, 36), (13, 7), (0, 5), (40000, 8),
              (3, 10240)]
    W0, Gs = inputs(shapes, "bf16", "bf16", 2)
    M0 = rand_M(shapes, seed=21, zero_line=True)
    for i, (a, b) in enumerate(shapes):   # keep the zero line zero through the momentum step
        if a > 2 and b > 2:
            if a <= b:
                Gs[1][i][1, :] = 0.0
            else:
                Gs[1][i][:, 1] = 0.0
    W = [to_dev(w, "bf16") for w in W0]
    M = [to_dev(m, "f32") for m in M0]
    ws = mm.alloc_workspace(shapes)
    rms = torch.full((len(shapes),), -1.0, device=dev())
    mm.muon_debug_set(TALL_PATHS[path], 0)
    try:
        # RowNorm step (scale_mode update_norm equals Eq. (7) when no line is zero; here some are)
        G = [to_dev(g, "bf16") for g in Gs[1]]
        mm.muon_periodic_step(W, G, M, 1, ws, update_rms=rms)
    finally:
        mm.muon_debug_set(0, 0)
    torch.cuda.synchronize()
    for i, s in enumerate(shapes):
        if 0 in s:
            assert float(rms[i]) == 0.0
            continue
        refW, refM, _, refrms = muon_ref.periodic_step(W0[i], M0[i], Gs[1][i], 1, telemetry=True, w_dtype="bf16")
        assert abs(float(rms[i]) - refrms) <= 1e-6 * refrms, (s, float(rms[i]), refrms)
    # refresh step telemetry against the oracle's RMS(O)
    rms.fill_(-1.0)
    G = [to_dev(g, "bf16") for g in Gs[0]]
    M2 = [to_dev(m, "f32") for m in M0]
    W2 = [to_dev(w, "bf16") for w in W0]
    mm.muon_periodic_step(W2, G, M2, 0, ws, update_rms=rms)
    torch.cuda.synchronize()
    for i, s in enumerate(shapes):
        if 0 in s:
            continue
        *_, refrms = muon_ref.periodic_step(W0[i], M0[i], Gs[0][i], 0, telemetry=True)
        assert abs(float(rms[i]) - refrms) <= TOL_NS5_BF16 * refrms, (s, float(rms[i]), refrms)


# ---------------------------------------------------------------------------
# AdamW beside Muon (biases, norms, out-of-block parameters)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("pdt,gdt", [("bf16", "bf16"), ("f32", "f32"), ("f32", "bf16")])
def test_adamw_parity(pdt, gdt):
    sizes = [1, 7, 1536, 4097, 9216, 100003]
    rng = np.random.default_rng(30)
    P0 = [quantize_np((rng.standard_normal(k) * 0.02).astype(np.float32), pdt) for k in sizes]
    P = [to_dev(p, pdt) for p in P0]
    m = [torch.zeros(k, device=dev()) for k in sizes]
    v = [torch.zeros(k, device=dev()) for k in sizes]
    refP = [p.astype(np.float64) for p in P0]
    refm = [np.zeros(k) for k in sizes]
    refv = [np.zeros(k) for k in sizes]
    lr, wd = 1e-4, 0.01
    for t in range(1, 5):
        Gn = [quantize_np((rng.standard_normal(k) * 10.0 ** rng.uniform(-4, -1)).astype(np.float32), gdt) for k in sizes]
        # teacher forcing on p: the GPU starts each step from the oracle's parameter
        for i in range(len(sizes)):
            P[i].copy_(to_dev(refP[i].astype(np.float32), pdt))
        mm.muon_adamw_step(P, [to_dev(g, gdt) for g in Gn], m, v, t, lr, weight_decay=wd)
        torch.cuda.synchronize()
        for i, k in enumerate(sizes):
            prev = refP[i]
            refP[i], refm[i], refv[i] = muon_ref.adamw_step(refP[i], Gn[i], refm[i], refv[i], t, lr, weight_decay=wd)
            assert_f32_close(to_np(m[i]), refm[i], what=f"m {k} t={t}")
            assert_f32_close(to_np(v[i]), refv[i], what=f"v {k} t={t}")
            step = prev - refP[i]
            terms = np.abs(prev) + np.abs(step)
            if pdt == "f32":
                d = np.abs(to_np(P[i]) - refP[i])
                assert np.all(d <= 1e-5 * terms + 1e-30), (k, t, float(np.max(d / (terms + 1e-30))))
            else:
                assert_bf16_close(to_np(P[i]), refP[i], terms, what=f"p {k} t={t}")
            refP[i] = muon_ref.round_to_storage(refP[i], pdt)


def test_periodic_muon_checkpoint_resumes_bit_exact():
    """A wrapper checkpoint (momentum, AdamW moments, step) taken after 2 steps and loaded
    into a fresh optimizer continues exactly like the uninterrupted run; a checkpoint
    from a different K is refused."""
    shapes = [(256, 512), (512, 256)]
    W0, Gs = inputs(shapes, "bf16", "bf16", 5)
    aux0 = [np.linspace(-1, 1, 300, dtype=np.float32), np.linspace(0.5, 2, 77, dtype=np.float32)]
    aux_g = [[np.sin(np.arange(a.size) * (t + 1)).astype(np.float32) * 1e-2 for a in aux0] for t in range(5)]

    def make():
        W = [to_dev(w, "bf16") for w in W0]
        A = [torch.from_numpy(a.copy()).to(dev()) for a in aux0]
        return W, A, mm.PeriodicMuon(W, aux_params=A)

    Wa, Aa, opt_a = make()
    for t in range(5):
        opt_a.step([to_dev(g, "bf16") for g in Gs[t]], [torch.from_numpy(g).to(dev()) for g in aux_g[t]])
    Wb, Ab, opt_b = make()
    for t in range(2):
        opt_b.step([to_dev(g, "bf16") for g in Gs[t]], [torch.from_numpy(g).to(dev()) for g in aux_g[t]])
    torch.cuda.synchronize()
    sd = {k: ([x.cpu() for x in v] if isinstance(v, list) else v) for k, v in opt_b.state_dict().items()}
    Wc = [w.clone() for w in Wb]
    Ac = [a.clone() for a in Ab]
    opt_c = mm.PeriodicMuon(Wc, aux_params=Ac)
    opt_c.load_state_dict(sd)
    for t in range(2, 5):
        opt_c.step([to_dev(g, "bf16") for g in Gs[t]], [torch.from_numpy(g).to(dev()) for g in aux_g[t]])
    torch.cuda.synchronize()
    for x, y in zip(Wa + Aa + opt_a.M, Wc + Ac + opt_c.M):
        assert torch.equal(x, y)
    with pytest.raises(ValueError):
        mm.PeriodicMuon([w.clone() for w in Wb], K=4, aux_params=[a.clone() for a in Ab]).load_state_dict(sd)


def test_periodic_muon_wrapper_matches_direct_calls():
    """The stateful wrapper (momentum buffers, workspace, step counter, auxiliary AdamW)
    gives the same bits as calling the entry points directly."""
    shapes = [(300, 1000), (1000, 300)]
    W0, Gs = inputs(shapes, "bf16", "bf16", 4)
    rng = np.random.default_rng(40)
    B0 = [(rng.standard_normal(a) * 0.01).astype(np.float32) for a, _ in shapes]
    Bg = [[(rng.standard_normal(a) * 1e-3).astype(np.float32) for a, _ in shapes] for _ in range(4)]
    Wa = [to_dev(w, "bf16") for w in W0]
    Ba = [to_dev(b, "f32") for b in B0]
    opt = mm.PeriodicMuon(Wa, aux_params=Ba, aux_lr=1e-4)
    Wb = [to_dev(w, "bf16") for w in W0]
    Bb = [to_dev(b, "f32") for b in B0]
    Mb = [torch.zeros(s, device=dev()) for s in shapes]
    mb = [torch.zeros(a, device=dev()) for a, _ in shapes]
    vb = [torch.zeros(a, device=dev()) for a, _ in shapes]
    ws = mm.alloc_workspace(shapes)
    for t in range(4):
        G = [to_dev(g, "bf16") for g in Gs[t]]
        bg = [to_dev(g, "f32") for g in Bg[t]]
        assert opt.step(G, bg) == (1 if t % 3 == 0 else 0)
        mm.muon_periodic_step(Wb, G, Mb, t, ws)
        mm.muon_adamw_step(Bb, bg, mb, vb, t + 1, 1e-4, weight_decay=0.01)
    torch.cuda.synchronize()
    assert opt.check() == mm.MUON_OK
    for a, b in zip(Wa + Ba + opt.M, Wb + Bb + Mb):
        assert torch.equal(a, b)
    sd = opt.state_dict()
    assert sd["step"] == 4 and len(sd["aux_m"]) == 2
