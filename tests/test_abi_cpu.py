"""C ABI checks that need no GPU: the library loads, exports every symbol that
include/muon.h declares, validates arguments before touching a device, and
reports the Periodic schedule (branch) bit-exactly for any step."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "muon.h")


@pytest.fixture(scope="session")
def lib():
    from matrix_aware_optimizer_muon_gb300 import build as b
    from matrix_aware_optimizer_muon_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        b.build()
    return _lib.load_library()


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(muon_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_spec_entry_points():
    names = header_functions()
    for n in ["muon_momentum", "muon_fro_norm", "muon_ns5_batched", "muon_rownorm", "muon_apply",
              "muon_periodic_step"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in header_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_status_strings(lib):
    from matrix_aware_optimizer_muon_gb300 import _lib
    assert lib.muon_abi_version() == 2
    for st in range(0, -8, -1):
        s = _lib.status_str(st)
        assert s and s != "unknown status"
    assert _lib.status_str(-99) == "unknown status"


def _mats(shapes, w_dt=1, g_dt=1, ptr=1 << 20):
    from matrix_aware_optimizer_muon_gb300._lib import MuonMatrix
    arr = (MuonMatrix * max(len(shapes), 1))()
    for i, (r, c) in enumerate(shapes):
        arr[i] = MuonMatrix(ptr, ptr, ptr, r, c, w_dt, g_dt)
    return arr


def _step(lib, mats, n, step, K, mode=0, ws=None, nbytes=0):
    br = ctypes.c_int(-7)
    st = lib.muon_periodic_step(mats, n, step, K, 0.15, 0.95, 0.02, 0.01, mode, ws, nbytes, None,
                                ctypes.byref(br))
    return st, br.value


def test_schedule_is_step_mod_K(lib):
    """Branch for steps 0..120 and far steps equals the oracle's step % K == 0."""
    from oracle import muon_ref
    empty = _mats([])
    for K in (1, 2, 3, 4, 7):
        for step in list(range(121)) + [2 ** 40, 2 ** 40 + 1, 3 * 10 ** 12, 3 * 10 ** 12 + 2]:
            st, br = _step(lib, empty, 0, step, K)
            assert st == 0
            assert br == (1 if muon_ref.is_refresh(step, K) else 0), (K, step)


def test_refresh_count_K3(lib):
    empty = _mats([])
    for T in (3, 6, 9, 30):
        cnt = sum(_step(lib, empty, 0, s, 3)[1] for s in range(T))
        assert cnt == -(-T // 3)


def test_argument_validation_before_device(lib):
    from matrix_aware_optimizer_muon_gb300 import _lib as L
    m = _mats([(4, 8)])
    assert _step(lib, m, 1, 0, 0)[0] == L.MUON_ERR_INVALID          # K < 1
    assert _step(lib, m, 1, -1, 3)[0] == L.MUON_ERR_INVALID         # step < 0
    assert _step(lib, m, -1, 0, 3)[0] == L.MUON_ERR_INVALID         # n < 0
    assert _step(lib, m, 1, 0, 3, mode=7)[0] == L.MUON_ERR_UNSUPPORTED
    bad = _mats([(4, 8), (4, 8)])
    bad[1].w_dtype = 0                                             # mixed dtypes
    assert _step(lib, bad, 2, 0, 3)[0] == L.MUON_ERR_UNSUPPORTED
    neg = _mats([(-1, 8)])
    assert _step(lib, neg, 1, 0, 3)[0] == L.MUON_ERR_INVALID
    null = _mats([(4, 8)], ptr=0)
    assert _step(lib, null, 1, 0, 3)[0] == L.MUON_ERR_INVALID
    odd = _mats([(4, 8)], ptr=(1 << 20) + 1)                       # misaligned bf16 pointer
    assert _step(lib, odd, 1, 0, 3)[0] == L.MUON_ERR_INVALID
    bigdt = _mats([(4, 8)], w_dt=5)
    assert _step(lib, bigdt, 1, 0, 3)[0] == L.MUON_ERR_UNSUPPORTED
    assert lib.muon_debug_set(0, -1) == L.MUON_ERR_INVALID
    assert lib.muon_debug_set(0, 0) == L.MUON_OK
    assert lib.muon_workspace_init(None, 0, None) == L.MUON_ERR_WORKSPACE
    assert lib.muon_check_status(None, 0, None) == L.MUON_ERR_WORKSPACE


def test_valid_call_without_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from matrix_aware_optimizer_muon_gb300 import _lib as L
    m = _mats([(4, 8)])
    st, br = _step(lib, m, 1, 0, 3)
    assert st == L.MUON_ERR_NO_DEVICE and br == 1


def test_workspace_size_plan(lib):
    from matrix_aware_optimizer_muon_gb300 import muon_workspace_size
    assert muon_workspace_size([]) == 0
    a = muon_workspace_size([(256, 1024)])
    b = muon_workspace_size([(256, 1024), (256, 1024)])
    # two same-shape matrices share one group: the NS5 part doubles, the header does not
    assert a < b < 2 * a + 4096
    # bf16 mode: 3 n x m bf16 buffers (X ping-pong + its residual, updated in place) and 2 n x n
    assert a >= 3 * 256 * 1024 * 2 + 2 * 256 * 256 * 2
    assert a < 4 * 256 * 1024 * 2
    # fp32 mode: 2 n x m fp32 and 2 n x n fp32
    f = muon_workspace_size([(256, 1024)], "f32")
    assert f >= 2 * 256 * 1024 * 4 + 2 * 256 * 256 * 4
    # tall and wide share the NS5 plan; only the RowNorm line partials differ
    assert abs(muon_workspace_size([(1024, 256)]) - a) <= 64 * 1024
    # ragged sizes pad the leading dimension to 8 elements
    assert muon_workspace_size([(5, 1001)]) >= 3 * 5 * 1008 * 2
    # empty matrices cost nothing but the header
    assert muon_workspace_size([(0, 100), (100, 0)]) <= 4096
    with pytest.raises(Exception):
        muon_workspace_size([(-1, 3)])
    # 1.3B MMDiT set: about 3 x 1.36e9 x 2 bytes for NS5 buffers
    from synth import WORKLOADS
    shapes = [(m.rows, m.cols) for m in WORKLOADS["mmdit-1.3b"].matrices]
    sz = muon_workspace_size(shapes)
    assert 3 * 1.35e9 * 2 < sz < 3 * 1.37e9 * 2 + 2e9
