"""GB300 (sm_103a) Muon / Periodic Row-wise Muon optimizer step.

The compute runs in libmuon_gb300.so (hand-written CUDA); this package is its
ctypes binding plus a small stateful wrapper.  See include/muon.h for the C ABI.
"""
from ._lib import (MUON_BRANCH_NS5, MUON_BRANCH_ROWNORM, MUON_DEBUG_NO_CLUSTER, MUON_DEBUG_NO_OVERLAP, MUON_DEBUG_TALL_CLUSTER, MUON_DEBUG_NO_PAIR, MUON_DEBUG_STALL_PRODUCER, MUON_DTYPE_BF16,
                   MUON_DTYPE_F32, MUON_ERR_CUDA, MUON_ERR_INVALID, MUON_ERR_NO_DEVICE, MUON_ERR_NONFINITE, MUON_ERR_TIMEOUT,
                   MUON_ERR_UNSUPPORTED, MUON_ERR_WORKSPACE, MUON_NS5_BF16, MUON_NS5_F32, MUON_OK, MUON_SCALE_ADJUSTED_LR, MUON_SCALE_UPDATE_NORM, MuonError,
                   MuonMatrix, alloc_workspace, load_library, make_matrices, muon_apply, muon_check_status,
                   muon_debug_set, muon_init, muon_fro_norm, muon_fro_norm_noalloc, muon_momentum, muon_ns5_batched, muon_periodic_step,
                   muon_rownorm, muon_workspace_init, muon_workspace_size, status_str,
                   muon_profile_events, muon_launch_count, muon_adamw_step)
from .optim import PeriodicMuon

__all__ = [n for n in dir() if not n.startswith("_")]
