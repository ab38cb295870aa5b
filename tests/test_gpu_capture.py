"""CUDA-graph capture of a host thread's first library calls.

A new host thread calls muon_init(), then captures its very first
muon_periodic_step calls (a refresh step and a RowNorm step over wide and tall
matrices, so that the RowNorm step forks its second stream) into two CUDA graphs.
Replaying them must give the same bits as the same two steps run eagerly."""
import threading

import pytest
import torch

from parity_util import dev, inputs, to_dev

pytestmark = pytest.mark.gpu

mm = pytest.importorskip("matrix_aware_optimizer_muon_gb300")

SHAPES = [(300, 1000), (1000, 300), (256, 256), (96, 7000)]


def test_first_calls_of_a_fresh_thread_capture_after_muon_init():
    mm.load_library()
    torch.cuda.set_device(0)
    W0, Gs = inputs(SHAPES, "bf16", "bf16", 2, seed=9)
    G = [[to_dev(g, "bf16") for g in Gs[t]] for t in range(2)]

    # eager reference on this thread
    We = [to_dev(w, "bf16") for w in W0]
    Me = [torch.zeros(s, device=dev()) for s in SHAPES]
    wse = mm.alloc_workspace(SHAPES)
    for t in range(2):
        mm.muon_periodic_step(We, G[t], Me, t, wse, K=3)
    torch.cuda.synchronize()

    Wg = [to_dev(w, "bf16") for w in W0]
    Mg = [torch.zeros(s, device=dev()) for s in SHAPES]
    wsg = mm.alloc_workspace(SHAPES)
    torch.cuda.synchronize()
    err = []

    def worker():
        try:
            torch.cuda.set_device(0)
            mm.muon_init()
            s = torch.cuda.Stream()
            graphs = []
            for t in range(2):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    mm.muon_periodic_step(Wg, G[t], Mg, t, wsg, K=3)
                graphs.append(g)
            for g in graphs:
                g.replay()
            torch.cuda.synchronize()
        except Exception as e:   # reported on the main thread
            err.append(e)

    th = threading.Thread(target=worker)
    th.start()
    th.join()
    assert not err, err
    assert mm.muon_check_status(wsg) == mm.MUON_OK
    for a, b in zip(We + Me, Wg + Mg):
        assert torch.equal(a, b)
