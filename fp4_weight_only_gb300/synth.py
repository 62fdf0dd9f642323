"""Seeded synthetic inputs: BF16 activations and BF16 weights.

This module draws random numbers only; it holds none of the method's
arithmetic (no quantisation, scaling or products).  The same tensors feed the
CUDA path and the CPU oracle.

Workloads follow the shapes and value distributions of the Petit blog's GEMM
study ("Detailed performance analysis": Llama-3-70B weight matrices at m = 16
and m = 256): activations ~ N(0, 1), weights ~ N(0, 0.02), optionally a small
fraction of activation outliers ~ N(0, 20).  No dataset or trained weights are
involved.
"""

import torch

# Llama-3-70B linear layers, (n, k) with W stored [n, k] (out, in).
LLAMA3_70B_SHAPES = {
    "qkv": (10240, 8192),
    "o": (8192, 8192),
    "gate_up": (57344, 8192),
    "down": (8192, 28672),
}


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def activations(m, k, seed=0, device="cpu", outlier_frac=0.0, outlier_std=20.0):
    """A [m, k] bf16 ~ N(0, 1); a fraction ``outlier_frac`` of entries is
    replaced by N(0, outlier_std) draws."""
    g = _gen(seed, device)
    a = torch.randn((m, k), generator=g, device=device, dtype=torch.float32)
    if outlier_frac > 0.0:
        go = _gen(seed + 2, device)
        pick = torch.rand((m, k), generator=go, device=device) < outlier_frac
        big = torch.randn((m, k), generator=go, device=device, dtype=torch.float32)
        a = torch.where(pick, big * outlier_std, a)
    return a.to(torch.bfloat16)


def weights(n, k, seed=1, device="cpu", std=0.02):
    """W [n, k] bf16 ~ N(0, std)."""
    g = _gen(seed, device)
    w = torch.randn((n, k), generator=g, device=device, dtype=torch.float32)
    return (w * std).to(torch.bfloat16)


def one_hot_activations(m, k, cols, device="cpu"):
    """A [m, k] bf16 with A[i, cols[i]] = 1 and zeros elsewhere."""
    a = torch.zeros((m, k), dtype=torch.bfloat16, device=device)
    idx = torch.as_tensor(cols, dtype=torch.long, device=device)
    a[torch.arange(m, device=device), idx] = 1.0
    return a


def moe_expert_offsets(tokens, experts, top_k, seed=0, skew=1.0):
    """Synthetic MoE routing: each of `tokens` tokens picks `top_k` distinct
    experts with probability proportional to 1 / (rank + 1)^skew (a seeded,
    Zipf-like popularity over a seeded expert order).  Returns the E + 1
    row offsets of the expert-grouped activation matrix (tokens * top_k
    rows)."""
    g = _gen(seed, "cpu")
    order = torch.randperm(experts, generator=g)
    weights = torch.empty(experts)
    weights[order] = 1.0 / (torch.arange(experts, dtype=torch.float32) + 1.0) ** skew
    counts = torch.zeros(experts, dtype=torch.int64)
    for _ in range(tokens):
        picked = torch.multinomial(weights, top_k, replacement=False, generator=g)
        counts[picked] += 1
    offsets = [0]
    for c in counts.tolist():
        offsets.append(offsets[-1] + c)
    return offsets
