"""Parity at the workloads' full sizes, in the launch configuration the benchmark
times (all matrices of a set in one muon_periodic_step call per step).  The
oracle checks sampled matrices one by one; the GPU runs the whole set."""
import numpy as np
import pytest
import torch

from oracle import muon_ref
from parity_util import (TOL_NS5_BF16, TOL_NS5_F32, apply_terms, assert_bf16_close, assert_f32_close,
                         check_implied_direction, dev, inputs, to_dev, to_np)
from synth import WORKLOADS, gradient_np, gradient_torch, quantize_np, weight_init_np, weight_init_torch

pytestmark = pytest.mark.gpu

mm = pytest.importorskip("matrix_aware_optimizer_muon_gb300")


def oracle_step(prevW, prevM, G, t, w_dtype):
    """The oracle's step with W both as stored (w_dtype) and unrounded (fp64)."""
    W64, M, refresh = muon_ref.periodic_step(prevW, prevM, G, t, w_dtype="f64")
    return muon_ref.round_to_storage(W64, w_dtype), W64, M, refresh


def check_step_w(got, refW, prevW, refresh, w_dtype, ns_mode, refM=None, refW64=None):
    if not refresh:
        if w_dtype == "f32":
            assert_f32_close(got, refW, what="W rownorm step")
        else:
            a, b = refW.shape
            terms = apply_terms(prevW, muon_ref.rownorm(refM), muon_ref.update_scale(a, b, False, 0.15), 0.02, 0.01)
            assert_bf16_close(got, refW, terms, what="W rownorm step")
        return
    tol = TOL_NS5_BF16 if ns_mode == "bf16" else TOL_NS5_F32
    ulp = 2.0 ** -7 if w_dtype == "bf16" else 2.0 ** -23
    err = np.linalg.norm(got - refW)
    lim = tol * np.linalg.norm(refW - prevW) + np.linalg.norm(np.abs(refW)) * ulp
    assert err <= lim, (err, lim)
    if refW64 is not None and w_dtype == "bf16":
        # the direction the fused apply used, within the NS5 tolerance plus half a bf16
        # ulp of W per element (the bound above lets the W rounding hide O's error)
        a, b = refW.shape
        check_implied_direction(got, prevW, refW64, 0.02, 0.01, muon_ref.update_scale(a, b, True, 0.15), tol,
                                what=f"implied O {a}x{b}")


def test_fp32_single_matrix_three_steps():
    """256x1024 fp32, 3 steps (1 NS5 refresh + 2 RowNorm), fp32 NS5 mode, free-running."""
    wl = WORKLOADS["fp32-256x1024"]
    shapes = [(m.rows, m.cols) for m in wl.matrices]
    W0, Gs = inputs(shapes, "f32", "f32", wl.steps, scales=wl.spike_scales)
    W = [to_dev(w, "f32") for w in W0]
    M = [torch.zeros(s, device=dev()) for s in shapes]
    ws = mm.alloc_workspace(shapes, "f32")
    refW, refM = W0[0].astype(np.float64), np.zeros(shapes[0])
    for t in range(wl.steps):
        br = mm.muon_periodic_step(W, [to_dev(Gs[t][0], "f32")], M, t, ws, K=wl.K, gamma=wl.gamma, mu=wl.mu,
                                   eta=wl.eta, lam=wl.lam, ns5_mode="f32")
        prevW = refW
        refW, refM, refresh = muon_ref.periodic_step(refW, refM, Gs[t][0], t, wl.K, wl.gamma, wl.mu, wl.eta,
                                                     wl.lam, w_dtype="f32")
        assert br == int(refresh)
        torch.cuda.synchronize()
        assert_f32_close(to_np(M[0]), refM, what=f"M step {t}")
        got = to_np(W[0])
        if refresh:
            check_step_w(got, refW, prevW, True, "f32", "f32")
        else:
            # free-running: W carries the refresh step's 1e-4-level difference
            err = np.linalg.norm(got - refW) / np.linalg.norm(refW - W0[0])
            assert err <= 1e-4, err
    assert mm.muon_check_status(ws) == mm.MUON_OK


def test_bf16_64x1536_six_steps_sampled():
    """64 square bf16 matrices, 6 steps; 4 sampled matrices checked every step (teacher-forced W)."""
    wl = WORKLOADS["bf16-64x1536sq"]
    shapes = [(m.rows, m.cols) for m in wl.matrices]
    sample = [0, 21, 42, 63]
    W = [to_dev(quantize_np(weight_init_np(a, b, 0, i), "bf16"), "bf16") for i, (a, b) in enumerate(shapes)]
    M = [torch.zeros(s, device=dev()) for s in shapes]
    ws = mm.alloc_workspace(shapes)
    refW = {i: to_np(W[i]) for i in sample}
    refM = {i: np.zeros(shapes[i]) for i in sample}
    for t in range(wl.steps):
        Gn = {}
        G = []
        for i, (a, b) in enumerate(shapes):
            g = quantize_np(gradient_np(a, b, wl.spike_scales, 0, i, t), "bf16")
            if i in sample:
                Gn[i] = g
            G.append(to_dev(g, "bf16"))
        for i in sample:                       # teacher forcing: GPU W starts from the oracle's W
            W[i].copy_(to_dev(refW[i].astype(np.float32), "bf16"))
        br = mm.muon_periodic_step(W, G, M, t, ws, K=wl.K)
        torch.cuda.synchronize()
        for i in sample:
            prevW = refW[i]
            refW[i], refW64, refM[i], refresh = oracle_step(refW[i], refM[i], Gn[i], t, "bf16")
            assert br == int(refresh)
            assert_f32_close(to_np(M[i]), refM[i], what=f"M {i} step {t}")
            check_step_w(to_np(W[i]), refW[i], prevW, refresh, "bf16", "bf16", refM[i], refW64)
    assert mm.muon_check_status(ws) == mm.MUON_OK


def test_mmdit_1_3b_full_set_one_period():
    """All 160 matrices of the 1.3B MMDiT set (the benchmark's launch configuration),
    one K=3 period on device-generated inputs; one matrix per shape group checked."""
    wl = WORKLOADS["mmdit-1.3b"]
    shapes = [(m.rows, m.cols) for m in wl.matrices]
    seed = 77
    d = dev()
    W = [weight_init_torch(torch, d, a, b, seed, i, torch.bfloat16) for i, (a, b) in enumerate(shapes)]
    M = [torch.zeros(s, device=d) for s in shapes]
    ws = mm.alloc_workspace(shapes)
    sample = {}
    for i, s in enumerate(shapes):
        sample.setdefault(s, i)
    sample = sorted(sample.values())
    refW = {i: to_np(W[i]) for i in sample}          # inputs from the generator, not from the kernels
    refM = {i: np.zeros(shapes[i]) for i in sample}
    for t in range(3):
        G = [gradient_torch(torch, d, a, b, wl.spike_scales, seed, i, t, torch.bfloat16)
             for i, (a, b) in enumerate(shapes)]
        Gn = {i: to_np(G[i]) for i in sample}
        for i in sample:
            W[i].copy_(torch.from_numpy(refW[i].astype(np.float32)).to(d, torch.bfloat16))
        br = mm.muon_periodic_step(W, G, M, t, ws)
        torch.cuda.synchronize()
        for i in sample:
            prevW = refW[i]
            refW[i], refW64, refM[i], refresh = oracle_step(refW[i], refM[i], Gn[i], t, "bf16")
            assert br == int(refresh)
            assert_f32_close(to_np(M[i]), refM[i], what=f"M {shapes[i]} step {t}")
            check_step_w(to_np(W[i]), refW[i], prevW, refresh, "bf16", "bf16", refM[i], refW64)
        del G
    assert mm.muon_check_status(ws) == mm.MUON_OK


def test_mmdit_1_3b_rownorm_invariants_all_matrices():
    """Property at any size: after a RowNorm step with eta=1, lambda=0, the update
    W_old - W_new is gamma*0.2*sqrt(m) times unit lines (fp32 W, every matrix)."""
    wl = WORKLOADS["mmdit-1.3b"]
    shapes = [(m.rows, m.cols) for m in wl.matrices][:10]
    d = dev()
    W = [torch.zeros(s, device=d) for s in shapes]
    M = [torch.randn(s, device=d) * 1e-2 for s in shapes]
    G = [torch.randn(s, device=d) * 1e-3 for s in shapes]
    ws = mm.alloc_workspace(shapes, "f32")
    mm.muon_periodic_step(W, G, M, 1, ws, K=3, gamma=0.15, eta=1.0, lam=0.0, ns5_mode="f32")
    torch.cuda.synchronize()
    for (a, b), w in zip(shapes, W):
        u = -w.double() / (0.15 * 0.2 * max(a, b) ** 0.5)
        norms = u.norm(dim=1 if a <= b else 0)
        assert torch.allclose(norms, torch.ones_like(norms), atol=1e-5), (a, b)


def _sampled_period(wl_key, sample_shapes, seed, steps=3):
    """All matrices of the set on the GPU for `steps` steps; the first matrix of each
    shape in `sample_shapes` is checked against the oracle every step."""
    wl = WORKLOADS[wl_key]
    shapes = [(m.rows, m.cols) for m in wl.matrices]
    d = dev()
    torch.cuda.empty_cache()
    W = [weight_init_torch(torch, d, a, b, seed, i, torch.bfloat16) for i, (a, b) in enumerate(shapes)]
    M = [torch.zeros(s, device=d) for s in shapes]
    ws = mm.alloc_workspace(shapes)
    sample = {}
    for i, s in enumerate(shapes):
        if s in sample_shapes:
            sample.setdefault(s, i)
    sample = sorted(sample.values())
    refW = {i: to_np(W[i]) for i in sample}
    refM = {i: np.zeros(shapes[i]) for i in sample}
    G = [torch.empty(s, device=d, dtype=torch.bfloat16) for s in shapes]
    for t in range(steps):
        for i, (a, b) in enumerate(shapes):
            gradient_torch(torch, d, a, b, wl.spike_scales, seed, i, t, torch.bfloat16, out=G[i])
        Gn = {i: to_np(G[i]) for i in sample}
        for i in sample:
            W[i].copy_(torch.from_numpy(refW[i].astype(np.float32)).to(d, torch.bfloat16))
        br = mm.muon_periodic_step(W, G, M, t, ws)
        torch.cuda.synchronize()
        for i in sample:
            prevW = refW[i]
            refW[i], refW64, refM[i], refresh = oracle_step(refW[i], refM[i], Gn[i], t, "bf16")
            assert br == int(refresh)
            assert_f32_close(to_np(M[i]), refM[i], what=f"M {shapes[i]} step {t}")
            check_step_w(to_np(W[i]), refW[i], prevW, refresh, "bf16", "bf16", refM[i], refW64)
    assert mm.muon_check_status(ws) == mm.MUON_OK
    del W, M, G, ws
    torch.cuda.empty_cache()


def test_mmdit_4b_full_set_sampled():
    """4B MMDiT set (170 matrices, H=2560): one K=3 period, square and tall 6H x H sampled."""
    H = 2560
    _sampled_period("mmdit-4b", {(H, H), (6 * H, H), (H, 4 * H)}, seed=91)


def test_mmdit_15b_full_set_sampled():
    """15B MMDiT set (440 matrices, H=3072, about 240 GB with the workspace): one
    refresh and one RowNorm step, square and tall 3H x H sampled."""
    H = 3072
    free, total = torch.cuda.mem_get_info()
    if free < 250e9:
        pytest.skip(f"needs ~250 GB free, {free / 1e9:.0f} GB available")
    _sampled_period("mmdit-15b", {(H, H), (3 * H, H)}, seed=92, steps=2)
