"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Every tensor is produced on the CPU from its own
``torch.Generator`` (X: seed 0, W: seed 1, labels: seed 2), drawn in fp32 and
rounded once to bf16 (round-to-nearest-even), so the CUDA path and the CPU
oracle read the very same bits.

Workload shapes come from the pages:
  * "Strength reduction: fold transpose into a subsequent GEMM call" -- the
    traced projection: activation bf16[384, 2, 13824] (viewed [768, 13824]),
    weight bf16[5120, 13824] in its stored layout, output bf16[384, 2, 5120].
  * "Schedule a small matmul op as a reduction (or pointwise) op" -- the RoPE
    K=1 matmul of a [64, 1] inverse-frequency column and a [1, 4096] row of
    positions (int64 cast to float).
  * "Allow reductions in matmul epilogues" -- a matmul whose epilogue is the
    row-wise cross-entropy over N (LM-head shapes: N is a vocabulary size).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

SEED_X, SEED_W, SEED_LABELS = 0, 1, 2


def bf16_normal(shape, std: float, seed: int) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 on the CPU, rounded once to bf16."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    t = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def labels_uniform(M: int, N: int, seed: int = SEED_LABELS) -> torch.Tensor:
    """int32[M], uniform over [0, N)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randint(0, N, (M,), generator=g, dtype=torch.int64).to(torch.int32)


def k1_operands(M: int = 64, N: int = 4096, head_dim: int = 128):
    """RoPE K=1 operands: a[i] = 1/10000^(2i/head_dim) (fp64, rounded once to
    fp32), b[j] = float(j) for positions j = 0..N-1.  Returns (a [M,1], b [1,N])."""
    a = torch.tensor([10000.0 ** (-(2.0 * i) / head_dim) for i in range(M)],
                     dtype=torch.float64).to(torch.float32).reshape(M, 1)
    b = torch.arange(N, dtype=torch.int64).to(torch.float32).reshape(1, N)
    return a, b


def rope_operands(H: int = 64, S: int = 4096, max_position: int = 0):
    """Inputs of the RoPE segment: inv_freq bf16 [H] = 1/10000^(2i/(2H)) (fp64,
    rounded to fp32, then to bf16) and int64 position ids [S] = 0, 1, ..., wrapping at
    `max_position` when it is positive (several sequences back to back)."""
    inv = torch.tensor([10000.0 ** (-(2.0 * i) / (2 * H)) for i in range(H)],
                       dtype=torch.float64).to(torch.float32).to(torch.bfloat16)
    pos = torch.arange(S, dtype=torch.int64)
    if max_position > 0:
        pos = pos % max_position
    return inv, pos


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    x_std: float
    w_std: float
    x_shape: tuple          # shape the activation is drawn in (viewed [M, K])
    path: str               # "gemm_nt", "xent_grad", "xent_loss", "k1", "tiny"
    description: str


WORKLOADS = {
    "tiny": Workload("tiny", 64, 256, 128, 1.0, 1.0 / math.sqrt(128), (64, 128), "tiny",
                     "X bf16[64,128]~N(0,1), W bf16[256,128]~N(0,1/128), labels U[0,256)"),
    "nt_projection": Workload("nt_projection", 768, 5120, 13824, 0.02, 0.02, (384, 2, 13824),
                              "gemm_nt",
                              "X bf16[384,2,13824] viewed [768,13824], W bf16[5120,13824], "
                              "both N(0,1)*0.02; out bf16[768,5120]"),
    "k1_rope": Workload("k1_rope", 64, 4096, 1, 0.0, 0.0, (64, 1), "k1",
                        "a fp32[64,1]=1/10000^(2i/128), b fp32[1,4096]=0..4095; out fp32[64,4096]"),
    "xent_grad": Workload("xent_grad", 4096, 32768, 4096, 1.0, 1.0 / 64.0, (4096, 4096),
                          "xent_grad",
                          "X bf16[4096,4096]~N(0,1), W bf16[32768,4096]~N(0,1/4096), "
                          "labels U[0,32768); loss fp32[4096] + grad bf16[4096,32768]"),
    "xent_loss": Workload("xent_loss", 8192, 128256, 4096, 1.0, 1.0 / 64.0, (8192, 4096),
                          "xent_loss",
                          "X bf16[8192,4096]~N(0,1), W bf16[128256,4096]~N(0,1/4096), "
                          "labels U[0,128256); loss fp32[8192] only"),
}


def make_gemm_inputs(M: int, N: int, K: int, x_std: float = 1.0, w_std: float = 1.0,
                     x_shape=None):
    """(X [M,K] or x_shape, W [N,K]) bf16 CPU tensors, seeds 0 and 1."""
    x = bf16_normal(x_shape if x_shape is not None else (M, K), x_std, SEED_X)
    w = bf16_normal((N, K), w_std, SEED_W)
    return x, w


def make_workload(name: str):
    """Inputs for a named workload as CPU tensors: dict with x, w, labels (or a, b)."""
    wl = WORKLOADS[name]
    if wl.path == "k1":
        a, b = k1_operands(wl.M, wl.N)
        return {"a": a, "b": b}
    x, w = make_gemm_inputs(wl.M, wl.N, wl.K, wl.x_std, wl.w_std, wl.x_shape)
    out = {"x": x, "w": w}
    if wl.path in ("tiny", "xent_grad", "xent_loss"):
        out["labels"] = labels_uniform(wl.M, wl.N)
    return out
