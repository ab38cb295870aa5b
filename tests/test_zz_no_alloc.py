"""muon_fro_norm_noalloc: the Frobenius norm for callers that cannot allocate
device memory (its scratch is a fixed array inside the library, not a caller
workspace).  Checked against muon_fro_norm, the workspace entry point, and against
the fp64 oracle, on two calls in a row with different matrix lists (the fixed
scratch keeps the previous call's contents, which must not leak into the next
result).  Collected last so
that a run stopping at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

mm = pytest.importorskip("matrix_aware_optimizer_muon_gb300")

TOL = 1e-5


def _lists():
    rng = np.random.default_rng(21)
    a = [(256, 1024), (1000, 300), (7, 13), (1, 517), (0, 9), (129, 129)]
    b = [(1536, 1536), (64, 40000), (300, 1000)]
    out = []
    for shapes in (a, b):
        out.append([torch.from_numpy((rng.standard_normal(s) * 1e-2).astype(np.float32)).cuda() for s in shapes])
    return out


def test_noalloc_fro_norm_matches_workspace_entry_point_twice():
    """Two calls in a row, each checked against muon_fro_norm and against the fp64
    oracle's ||M||_F (the Frobenius norm of X_0 = M/||M||_F, "Muon is Scalable for LLM
    Training" notes, section 2.1)."""
    from oracle import muon_ref
    mm.load_library()
    torch.cuda.set_device(0)
    for M in _lists():
        n = len(M)
        ws = mm.alloc_workspace([tuple(m.shape) for m in M])
        want = torch.full((n,), -1.0, device="cuda")
        got = torch.full((n,), -2.0, device="cuda")
        mm.muon_fro_norm(M, want, ws)
        mm.muon_fro_norm_noalloc(M, got)
        torch.cuda.synchronize()
        w, g = want.cpu().numpy(), got.cpu().numpy()
        assert np.all(np.abs(g - w) <= TOL * np.maximum(np.abs(w), 1e-30)), (g, w)
        ref = np.array([muon_ref.frobenius_norm(m.cpu().numpy().astype(np.float64)) for m in M])
        assert np.all(np.abs(g - ref) <= TOL * np.maximum(ref, 1e-30)), (g, ref)


def test_noalloc_rejects_what_the_workspace_entry_point_rejects():
    """An unknown dtype code and a list of mixed dtypes give MUON_ERR_UNSUPPORTED from
    both entry points (checked on the host, before any launch)."""
    from matrix_aware_optimizer_muon_gb300._lib import MuonMatrix
    lib = mm.load_library()
    m = torch.zeros(8, 8, device="cuda")
    out = torch.empty(2, device="cuda")
    ws = mm.alloc_workspace([(8, 8), (8, 8)])
    for dts in ([(7, 1), (7, 1)], [(1, 1), (0, 0)]):
        arr = (MuonMatrix * 2)()
        for i, (wd, gd) in enumerate(dts):
            arr[i] = MuonMatrix(None, None, m.data_ptr(), 8, 8, wd, gd)
        assert lib.muon_fro_norm_noalloc(arr, 2, out.data_ptr(), None) == mm.MUON_ERR_UNSUPPORTED
        assert lib.muon_fro_norm(arr, 2, out.data_ptr(), ws.data_ptr(), ws.numel(), None) == \
            mm.MUON_ERR_UNSUPPORTED


def test_noalloc_rejects_lists_beyond_its_fixed_scratch():
    mm.load_library()
    big = torch.empty(0, device="cuda")
    from matrix_aware_optimizer_muon_gb300._lib import MuonMatrix
    arr = (MuonMatrix * 1)()
    arr[0] = MuonMatrix(None, None, big.data_ptr() or 256, 65536, 65536 * 2 + 128, 1, 1)   # 1024 x 1025 tiles
    out = torch.empty(1, device="cuda")
    st = mm.load_library().muon_fro_norm_noalloc(arr, 1, out.data_ptr(), None)
    assert st == mm.MUON_ERR_UNSUPPORTED
