"""Seeded synthetic inputs shaped like the MXFP8 training workloads.

This module is shared by the CUDA path's tests and benchmark and by the
oracle's tests.  It holds no quantization or GEMM arithmetic: it only draws
BF16 tensors and MoE routings from seeded generators.

Workloads (shapes follow the linear and MoE-expert matmuls that the
torchtitan-npu low-precision tutorial quantizes -- "nn.Linear" layers and
"MoE 专家层 (Grouped MM)" -- and the DeepSeek-V4-Flash expert sizes of the
MindSpeed RFC's MoE use case, section 2.2):

  linear_fwd_small  X [256, 512] ~N(0,1) with outliers, W [512, 512] ~N(0, 0.02^2)
  linear_train      X [8192, 4096] (outliers), W [4096, 4096], dY [8192, 4096] ~N(0, 1e-3^2)
  weight_32x32      W [7168, 7168]; X, dY [4096, 7168]
  moe_grouped       16384 tokens, hidden 4096, 128 experts, top-8, Zipf(1.1) loads
                    (4 experts empty); gate_up W [128, 4096, 4096], down W [128, 4096, 2048]
  sweep_<K>         M = 16384, K = N in {4096, 7168, 16384}; X, dY = 0.5 * Student-t(3)

"Outliers": every entry independently, with probability 1e-3, is multiplied
by 100.  Seeds: tensor index i of workload w uses seed 1000*w + i (w = 1..5;
the small linear case uses w = 0).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

WORKLOAD_IDS = {"linear_fwd_small": 0, "linear_train": 2, "weight_32x32": 3,
                "moe_grouped": 4, "sweep_4096": 5, "sweep_7168": 5, "sweep_16384": 5}
TENSOR_INDEX = {"X": 0, "W": 1, "dY": 2, "routing": 3, "H": 4, "W_down": 5}


def seed_for(workload: str, tensor: str, sub: int = 0) -> int:
    return 1000 * WORKLOAD_IDS[workload] + TENSOR_INDEX[tensor] + 100 * sub


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in float32, returned as bf16."""
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def normal_with_outliers(shape, seed: int, p: float = 1e-3, factor: float = 100.0,
                         device="cpu") -> torch.Tensor:
    """N(0,1); each entry independently with probability p multiplied by factor."""
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    u = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    x = torch.where(u < p, x * factor, x)
    return x.to(torch.bfloat16)


def student_t(shape, seed: int, df: int = 3, scale: float = 0.5, device="cpu") -> torch.Tensor:
    """scale * Z / sqrt(chi2_df / df), Z and the df normals of chi2 from one generator."""
    g = _gen(seed, device)
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(df):
        n = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        chi2.addcmul_(n, n)
    return (scale * z / torch.sqrt(chi2 / df)).to(torch.bfloat16)


@dataclass
class Routing:
    """Rows sorted by expert.  token_of_row[r] is the token that row r copies;
    offsets[g] .. offsets[g+1] are the rows of expert g."""
    token_of_row: torch.Tensor      # int64 [tokens * topk]
    offsets: torch.Tensor           # int64 [experts + 1]
    experts: int
    empty_experts: list = field(default_factory=list)


def moe_routing(tokens: int, experts: int, topk: int, seed: int, zipf_s: float = 1.1,
                n_empty: int = 4) -> Routing:
    """Top-k routing with Zipf(s) expert popularity.

    Expert popularity by rank r = 1..E is w_r ~ r^-s; ranks are assigned to
    expert ids by a seeded permutation and n_empty seeded experts get weight 0
    so that empty groups occur.  Each token draws topk distinct experts by the
    Gumbel-top-k trick on log w.  Rows are then sorted by expert (stable in
    token order)."""
    g = _gen(seed, "cpu")
    perm = torch.randperm(experts, generator=g)
    ranks = torch.arange(1, experts + 1, dtype=torch.float64)
    logw_by_rank = -zipf_s * torch.log(ranks)
    logw = torch.empty(experts, dtype=torch.float64)
    logw[perm] = logw_by_rank
    empty = torch.randperm(experts, generator=g)[:n_empty]
    logw[empty] = -math.inf
    u = torch.rand((tokens, experts), generator=g, dtype=torch.float64).clamp_(1e-300, 1.0)
    gumbel = -torch.log(-torch.log(u))
    score = logw.unsqueeze(0) + gumbel
    chosen = torch.topk(score, topk, dim=1).indices          # [tokens, topk], distinct
    expert_of_row = chosen.reshape(-1)
    token_ids = torch.arange(tokens).repeat_interleave(topk)
    order = torch.sort(expert_of_row, stable=True).indices
    counts = torch.bincount(expert_of_row, minlength=experts)
    offsets = torch.zeros(experts + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(counts, 0)
    return Routing(token_ids[order].contiguous(), offsets, experts, sorted(empty.tolist()))


def linear_fwd_small(device="cpu"):
    w = "linear_fwd_small"
    return {"X": normal_with_outliers((256, 512), seed_for(w, "X"), device=device),
            "W": normal((512, 512), 0.02, seed_for(w, "W"), device=device)}


def linear_train(device="cpu", M=8192, N=4096, K=4096):
    w = "linear_train"
    return {"X": normal_with_outliers((M, K), seed_for(w, "X"), device=device),
            "W": normal((N, K), 0.02, seed_for(w, "W"), device=device),
            "dY": normal((M, N), 1e-3, seed_for(w, "dY"), device=device)}


def weight_32x32(device="cpu", M=4096, N=7168, K=7168):
    w = "weight_32x32"
    return {"W": normal((N, K), 0.02, seed_for(w, "W"), device=device),
            "X": normal_with_outliers((M, K), seed_for(w, "X"), device=device),
            "dY": normal((M, N), 1e-3, seed_for(w, "dY"), device=device)}


def moe_grouped(device="cpu", tokens=16384, hidden=4096, inter=2048, experts=128, topk=8,
                weights=True):
    """Routed inputs for the expert GEMMs: A = X rows gathered in expert order
    [tokens*topk, hidden]; H = the down-projection input [tokens*topk, inter];
    gate_up weights [E, 2*inter, hidden]; down weights [E, hidden, inter]
    (omitted when weights=False)."""
    w = "moe_grouped"
    routing = moe_routing(tokens, experts, topk, seed_for(w, "routing"))
    x = normal_with_outliers((tokens, hidden), seed_for(w, "X"), device=device)
    a = x.index_select(0, routing.token_of_row.to(device))
    h = normal((tokens * topk, inter), 1.0, seed_for(w, "H"), device=device)
    out = {"A": a, "H": h, "routing": routing}
    if weights:
        out["W_gate_up"] = normal((experts, 2 * inter, hidden), 0.02, seed_for(w, "W"), device=device)
        out["W_down"] = normal((experts, hidden, inter), 0.02, seed_for(w, "W_down"), device=device)
    return out


def sweep(K: int, device="cpu", M=16384):
    w = f"sweep_{K}"
    return {"X": student_t((M, K), seed_for(w, "X"), device=device),
            "W": normal((K, K), 0.02, seed_for(w, "W"), device=device),
            "dY": student_t((M, K), seed_for(w, "dY"), device=device)}
