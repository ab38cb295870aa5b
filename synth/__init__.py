"""Seeded synthetic workloads for the Muon optimizer step.

This module serves both the CUDA path and the oracle: it only makes inputs
(weights W0 and per-step gradients G) and describes the parameter-set shapes.
It holds none of the optimizer's arithmetic.

Shapes follow the MMDiT parameter sets of "Scaling Muon for Diffusion
Transformers" (agihunt summary, the experimental-setup paragraph: double-stream
MMDiT at 1.3B/4B/15B; Muon on the 2-D weights of the Transformer blocks).  Per
stream and per block the 2-D weights are qkv (3H x H), proj (H x H),
MLP-up (4H x H), MLP-down (H x 4H) and the adaLN modulation (6H x H).

Gradient recipe: G = N(0, sigma^2) + sum_i s_i u_i v_i^T with u_i, v_i ~ N(0, 1);
weights W0 ~ N(0, 0.02^2).  Every draw is keyed by (seed, matrix index, step), so
any single matrix can be regenerated alone.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Sequence, Tuple

import numpy as np

W_INIT_STD = 0.02
NOISE_STD = 1e-3


@dataclasses.dataclass(frozen=True)
class MatrixSpec:
    name: str
    rows: int   # A (out features)
    cols: int   # B (in features)


@dataclasses.dataclass(frozen=True)
class Workload:
    key: str
    description: str
    matrices: Tuple[MatrixSpec, ...]
    w_dtype: str          # "bf16" | "f32"
    g_dtype: str          # "bf16" | "f32"
    steps: int
    spike_scales: Tuple[float, ...]
    K: int = 3
    gamma: float = 0.15
    mu: float = 0.95
    eta: float = 0.02
    lam: float = 0.01

    @property
    def n_params(self) -> int:
        return sum(m.rows * m.cols for m in self.matrices)

    def shape_groups(self) -> List[Tuple[Tuple[int, int], int]]:
        """(rows, cols) -> count, in first-appearance order."""
        seen = {}
        for m in self.matrices:
            seen[(m.rows, m.cols)] = seen.get((m.rows, m.cols), 0) + 1
        return list(seen.items())


def mmdit_matrices(H: int, blocks: int) -> Tuple[MatrixSpec, ...]:
    out = []
    for b in range(blocks):
        for stream in ("img", "txt"):
            p = f"block{b}.{stream}"
            out.append(MatrixSpec(f"{p}.qkv", 3 * H, H))
            out.append(MatrixSpec(f"{p}.proj", H, H))
            out.append(MatrixSpec(f"{p}.mlp_up", 4 * H, H))
            out.append(MatrixSpec(f"{p}.mlp_down", H, 4 * H))
            out.append(MatrixSpec(f"{p}.adaln", 6 * H, H))
    return tuple(out)


def _geometric(n: int, s0: float, r: float) -> Tuple[float, ...]:
    return tuple(s0 * r ** i for i in range(n))


WORKLOADS = {
    "fp32-256x1024": Workload(
        "fp32-256x1024",
        "single fp32 matrix 256x1024, rank-4 spike at 1e-2, 3 steps",
        (MatrixSpec("w", 256, 1024),), "f32", "f32", 3, (1e-2,) * 4),
    "bf16-64x1536sq": Workload(
        "bf16-64x1536sq",
        "64 square bf16 matrices 1536x1536, rank-8 geometric spike 1e-2*0.5^i, 6 steps",
        tuple(MatrixSpec(f"w{i}", 1536, 1536) for i in range(64)), "bf16", "bf16", 6,
        _geometric(8, 1e-2, 0.5)),
    "mmdit-1.3b": Workload(
        "mmdit-1.3b",
        "1.3B-class MMDiT Muon set, H=1536, 16 double-stream blocks, bf16 W/G, fp32 M, 6 steps",
        mmdit_matrices(1536, 16), "bf16", "bf16", 6, _geometric(8, 1e-2, 0.5)),
    "mmdit-4b": Workload(
        "mmdit-4b",
        "4B-class MMDiT Muon set, H=2560, 17 double-stream blocks, bf16 W/G, fp32 M, 9 steps",
        mmdit_matrices(2560, 17), "bf16", "bf16", 9, _geometric(8, 1e-2, 0.5)),
    "mmdit-15b": Workload(
        "mmdit-15b",
        "15B-class MMDiT Muon set, H=3072, 44 double-stream blocks, bf16 W/G, fp32 M, 30 steps",
        mmdit_matrices(3072, 44), "bf16", "bf16", 30, (1e-2,) * 16),
}
# Index order of the parameter sets as the workload list gives them.
WORKLOAD_ORDER = ("fp32-256x1024", "bf16-64x1536sq", "mmdit-1.3b", "mmdit-4b", "mmdit-15b")


def _seq(seed: int, tag: int, index: int, step: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, index, step])))


def weight_init_np(rows: int, cols: int, seed: int, index: int) -> np.ndarray:
    """W0 ~ N(0, 0.02^2) as float32, keyed by (seed, index)."""
    g = _seq(seed, 1, index, 0)
    return (g.standard_normal((rows, cols), dtype=np.float32) * np.float32(W_INIT_STD))


def gradient_np(rows: int, cols: int, spike_scales: Sequence[float], seed: int, index: int,
                step: int) -> np.ndarray:
    """G = N(0, 1e-3^2) + sum_i s_i u_i v_i^T as float32, keyed by (seed, index, step).

    Noise, then u_i, then v_i are drawn in that order from the keyed stream.
    """
    g = _seq(seed, 2, index, step)
    G = g.standard_normal((rows, cols), dtype=np.float32) * np.float32(NOISE_STD)
    r = len(spike_scales)
    if r:
        U = g.standard_normal((rows, r), dtype=np.float32)
        V = g.standard_normal((cols, r), dtype=np.float32)
        U = U * np.asarray(spike_scales, dtype=np.float32)[None, :]
        G += U @ V.T
    return G


def to_bf16_bits_np(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest even); return the uint16 bit pattern."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    out = ((u + rounding) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32_np(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def quantize_np(x: np.ndarray, dtype: str) -> np.ndarray:
    """Values as the storage dtype holds them, returned as float32."""
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f32_np(to_bf16_bits_np(x))
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# torch device generators (fast, for full-size runs); same recipe, own stream.
# ---------------------------------------------------------------------------

def _torch_gen(torch, device, seed: int, tag: int, index: int, step: int):
    g = torch.Generator(device=device)
    g.manual_seed(int(np.random.SeedSequence([seed, tag, index, step]).generate_state(1)[0]))
    return g


def weight_init_torch(torch, device, rows, cols, seed, index, dtype):
    g = _torch_gen(torch, device, seed, 1, index, 0)
    w = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32) * W_INIT_STD
    return w.to(dtype)


def gradient_torch(torch, device, rows, cols, spike_scales, seed, index, step, dtype, out=None):
    g = _torch_gen(torch, device, seed, 2, index, step)
    G = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32) * NOISE_STD
    r = len(spike_scales)
    if r:
        U = torch.randn((rows, r), generator=g, device=device, dtype=torch.float32)
        V = torch.randn((cols, r), generator=g, device=device, dtype=torch.float32)
        U = U * torch.tensor(spike_scales, device=device, dtype=torch.float32)[None, :]
        G.addmm_(U, V.t())
    if out is not None:
        out.copy_(G)
        return out
    return G.to(dtype)
