"""NaN and Inf in the gradient: deterministic propagation, matching the oracle's
positions, and the opt-in finite check of muon_periodic_step_ex.

The failure is made on the host: NaN or Inf is written into G before it is copied
to the device.  Nothing here faults, traps or stalls the GPU.

Reading (the pages are silent on non-finite inputs): the direction is M divided by
its norm as written, and only an exactly zero norm gives a zero direction.  A NaN
in a line of M makes that line's norm NaN, so on a RowNorm step the whole line of W
becomes NaN; an Inf makes the norm Inf, so the finite entries of that line get a zero
direction (pure weight decay) and the Inf entry NaN.  On a refresh step ||M||_F is
non-finite and NS5 spreads it to every entry of the matrix."""
import numpy as np
import pytest
import torch

from oracle import muon_ref
from parity_util import (TOL_NS5_BF16, apply_terms, assert_bf16_close, assert_f32_close, dev, inputs, to_dev,
                         to_np)

pytestmark = pytest.mark.gpu

mm = pytest.importorskip("matrix_aware_optimizer_muon_gb300")

# wide (rows kernel), tall (tall-matrix routes), square, a 7000-column row (the 512-thread
# wide-row kernel), a tall matrix with B % 4 != 0 (the plain two-pass kernels), and a clean
# wide matrix that must stay unaffected
SHAPES = [(192, 320), (320, 192), (256, 256), (4, 7000), (300, 130), (130, 1000)]
TALL_PATHS = {"l2pass": 0, "cluster": mm.MUON_DEBUG_TALL_CLUSTER, "two_pass": mm.MUON_DEBUG_NO_CLUSTER}
NAN, INF = float("nan"), float("inf")
# (step, matrix, row, col, value) written into G on the host
INJECT = [(1, 0, 5, 17, NAN), (1, 1, 40, 7, INF), (1, 3, 2, 6500, NAN), (1, 4, 250, 129, -INF),
          (3, 2, 100, 200, NAN)]
STEPS = 4   # refresh, RowNorm, RowNorm, refresh (K = 3)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mm.load_library()
    torch.cuda.set_device(0)
    yield
    mm.muon_debug_set(0, 0)


def _gradients():
    W0, Gs = inputs(SHAPES, "bf16", "bf16", STEPS, seed=5)
    for t, i, r, c, v in INJECT:
        Gs[t][i] = Gs[t][i].copy()
        Gs[t][i][r, c] = v
    return W0, Gs


def _run(check, path=0):
    """Runs the steps; returns per-step (W, M) host copies as float64 and the statuses."""
    W0, Gs = _gradients()
    W = [to_dev(w, "bf16") for w in W0]
    M = [torch.zeros(s, device=dev()) for s in SHAPES]
    ws = mm.alloc_workspace(SHAPES)
    states, statuses, raw = [], [], None
    mm.muon_debug_set(path, 0)
    try:
        for t in range(STEPS):
            G = [to_dev(g, "bf16") for g in Gs[t]]
            br = mm.muon_periodic_step(W, G, M, t, ws, K=3, check_finite=check)
            assert br == (mm.MUON_BRANCH_NS5 if t % 3 == 0 else mm.MUON_BRANCH_ROWNORM)
            statuses.append(mm.muon_check_status(ws))
            states.append(([to_np(w) for w in W], [to_np(m) for m in M]))
    finally:
        mm.muon_debug_set(0, 0)
    raw = ([w.view(torch.int16).cpu() for w in W], [m.view(torch.int32).cpu() for m in M])
    return W0, Gs, states, statuses, raw


def _same_nonfinite(got, ref, what):
    assert np.array_equal(np.isnan(got), np.isnan(ref)), f"{what}: NaN positions differ " \
        f"({int(np.isnan(got).sum())} on the GPU, {int(np.isnan(ref).sum())} in the oracle)"
    assert np.array_equal(np.isposinf(got), np.isposinf(ref)) and np.array_equal(np.isneginf(got), np.isneginf(ref)), \
        f"{what}: Inf positions differ"


@pytest.mark.parametrize("path", list(TALL_PATHS))
def test_nonfinite_gradient_propagates_like_the_oracle(path):
    W0, Gs, states, statuses, _ = _run(True, TALL_PATHS[path])
    prevW = [w.astype(np.float64) for w in W0]
    prevM = [np.zeros(s) for s in SHAPES]
    for t in range(STEPS):
        for i, (a, b) in enumerate(SHAPES):
            # teacher-forced: the oracle steps from the GPU's previous state
            with np.errstate(invalid="ignore", over="ignore"):
                refW, refM, refresh = muon_ref.periodic_step(prevW[i], prevM[i], Gs[t][i], t, 3, 0.15, 0.95, 0.02,
                                                             0.01, w_dtype="bf16")
            gotW, gotM = states[t][0][i], states[t][1][i]
            what = f"step {t} matrix {SHAPES[i]}"
            _same_nonfinite(gotM, refM, "M " + what)
            _same_nonfinite(gotW, refW, "W " + what)
            fin = np.isfinite(refM)
            assert_f32_close(gotM[fin], refM[fin], what="M " + what)
            finW = np.isfinite(refW)
            if refresh:
                if finW.all():
                    dW = refW - prevW[i]
                    assert np.linalg.norm(gotW - refW) <= TOL_NS5_BF16 * np.linalg.norm(dW) + \
                        np.linalg.norm(refW) * 2.0 ** -7, what
                else:
                    assert not finW.any(), f"{what}: a refresh of a non-finite momentum is NaN everywhere"
            else:
                with np.errstate(invalid="ignore"):
                    U = muon_ref.rownorm(refM)
                terms = apply_terms(prevW[i], U, muon_ref.update_scale(a, b, False, 0.15), 0.02, 0.01)
                assert_bf16_close(gotW[finW], refW[finW], terms[finW], what="W " + what)
            prevW[i], prevM[i] = gotW, gotM
    # the finite check saw the non-finite norms from step 1 on, and nothing at step 0
    assert statuses == [mm.MUON_OK] + [mm.MUON_ERR_NONFINITE] * (STEPS - 1)
    # every injected matrix ends all-NaN after the second refresh; the clean one stays finite
    last_W = states[-1][0]
    for i in (0, 1, 2, 3, 4):
        assert np.isnan(last_W[i]).all()
    assert np.isfinite(last_W[5]).all()


def test_nonfinite_results_are_bit_exact_and_independent_of_the_check():
    _, _, _, st1, raw1 = _run(True)
    _, _, _, st2, raw2 = _run(True)
    _, _, _, st3, raw3 = _run(False)
    assert st1 == st2 == [mm.MUON_OK] + [mm.MUON_ERR_NONFINITE] * (STEPS - 1)
    assert st3 == [mm.MUON_OK] * STEPS   # the check is opt-in
    for r in (raw2, raw3):
        for a, b in zip(raw1[0] + raw1[1], r[0] + r[1]):
            assert torch.equal(a, b)


def test_finite_inputs_report_no_error_with_the_check_on():
    W0, Gs = inputs(SHAPES, "bf16", "bf16", STEPS, seed=6)
    W = [to_dev(w, "bf16") for w in W0]
    M = [torch.zeros(s, device=dev()) for s in SHAPES]
    ws = mm.alloc_workspace(SHAPES)
    for t in range(STEPS):
        mm.muon_periodic_step(W, [to_dev(g, "bf16") for g in Gs[t]], M, t, ws, K=3, check_finite=True)
        assert mm.muon_check_status(ws) == mm.MUON_OK
