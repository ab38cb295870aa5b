"""muon_fro_norm_noalloc: the Frobenius norm for callers that cannot allocate
device memory (its scratch is a fixed array inside the library, not a caller
workspace).  Checked against muon_fro_norm, the workspace entry point, on two
calls in a row with different matrix lists (the fixed scratch keeps the previous
call's contents, which must not leak into the next result).  Collected last so
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


def test_noalloc_rejects_lists_beyond_its_fixed_scratch():
    mm.load_library()
    big = torch.empty(0, device="cuda")
    from matrix_aware_optimizer_muon_gb300._lib import MuonMatrix
    arr = (MuonMatrix * 1)()
    arr[0] = MuonMatrix(None, None, big.data_ptr() or 256, 65536, 65536 * 2 + 128, 1, 1)   # 1024 x 1025 tiles
    out = torch.empty(1, device="cuda")
    st = mm.load_library().muon_fro_norm_noalloc(arr, 1, out.data_ptr(), None)
    assert st == mm.MUON_ERR_UNSUPPORTED
