"""Seeded synthetic Q, K, V for the attention workloads.

This module only draws random numbers: it holds none of the attention or
quantization arithmetic, and both the CUDA path and the CPU oracle take their
inputs from it, so they see identical bytes.

The SageAttention3 pages measure on real model activations (CogVideoX,
HunyuanVideo, Mochi, Flux, SD3.5, Qwen2.5, Llama3.2) that are not available;
these seeded shapes and value patterns stand in for them: an LLM-prefill shape
with per-channel K offsets and outlier channels, video-DiT shapes with a
per-head K mean offset or rare large entries.

Recipe (identical on every machine): ``torch.Generator('cpu').manual_seed(seed)``,
float32 draws in the order Q, K, V, then the pattern draws, cast to bf16 last.
"N(0, s)" means standard deviation s.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    causal: bool
    pattern: str

    @property
    def ops(self) -> float:
        """4*B*H*N^2*D, causal counted at half."""
        o = 4.0 * self.B * self.H * self.N * self.N * self.D
        return o / 2 if self.causal else o

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "N": self.N, "D": self.D,
                "causal": self.causal, "pattern": self.pattern}


WORKLOADS = {
    "small": Workload("attn_fwd B1 H2 N512 D128 iid", 1, 2, 512, 128, False, "iid"),
    "llm": Workload("attn_fwd B4 H32 N4096 D128 k-channel-outliers", 4, 32, 4096, 128, False,
                    "k_channel_outliers"),
    "llm_causal": Workload("attn_fwd B4 H32 N8192 D128 causal k-channel-outliers", 4, 32, 8192,
                           128, True, "k_channel_outliers"),
    "dit": Workload("attn_fwd B2 H48 N17776 D64 k-head-mean", 2, 48, 17776, 64, False,
                    "k_head_mean"),
    "dit_long": Workload("attn_fwd B1 H24 N32768 D128 sparse-outliers", 1, 24, 32768, 128, False,
                         "sparse_outliers"),
}

# SageBwd (8-bit attention for training) shapes: the pages fine-tune Llama3.2
# (1B: 32 query heads of 64) and Qwen2.5 (3B: 16 query heads of 128) and time
# Llama-1B training on 8K/16K-token micro-batches.  One 8K-token sequence per
# micro-batch, causal; grouped K/V heads are taken as one K/V head per query
# head.
TRAIN_WORKLOADS = {
    "train_small": Workload("attn_train B1 H2 N512 D64 iid", 1, 2, 512, 64, False, "iid"),
    "train_llama1b": Workload("attn_train B1 H32 N8192 D64 causal iid", 1, 32, 8192, 64, True, "iid"),
    "train_qwen3b": Workload("attn_train B1 H16 N8192 D128 causal k-channel-outliers", 1, 16, 8192, 128, True,
                             "k_channel_outliers"),
    # half the heads of the Llama-1B and Qwen-3B shapes: the cases the
    # full-set profiles capture
    "train_llama1b_h16": Workload("attn_train B1 H16 N8192 D64 causal iid", 1, 16, 8192, 64, True, "iid"),
    "train_qwen3b_h8": Workload("attn_train B1 H8 N8192 D128 causal k-channel-outliers", 1, 8, 8192, 128, True,
                                "k_channel_outliers"),
}


def make_qkv(B: int, H: int, N: int, D: int, pattern: str = "iid", seed: int = 0):
    """Return bf16 CPU tensors q, k, v of shape [B, H, N, D] (contiguous)."""
    g = torch.Generator("cpu").manual_seed(seed)
    shape = (B, H, N, D)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if pattern == "iid":
        pass
    elif pattern == "k_channel_outliers":
        # per-(b,h,channel) offset N(0,4) broadcast over tokens, then 1% of the
        # channels (Bernoulli mask) multiplied by 20, offset included
        off = torch.randn((B, H, 1, D), generator=g, dtype=torch.float32) * 4.0
        mask = torch.rand((B, H, 1, D), generator=g, dtype=torch.float32) < 0.01
        k = (k + off) * torch.where(mask, 20.0, 1.0)
    elif pattern == "k_head_mean":
        # one scalar mean per head, N(0,2), added to every K entry of that head
        mu = torch.randn((B, H, 1, 1), generator=g, dtype=torch.float32) * 2.0
        k = k + mu
    elif pattern == "sparse_outliers":
        # each entry of each tensor replaced with probability 0.001 by N(0,30)
        outs = []
        for t in (q, k, v):
            m = torch.rand(shape, generator=g, dtype=torch.float32) < 0.001
            big = torch.randn(shape, generator=g, dtype=torch.float32) * 30.0
            outs.append(torch.where(m, big, t))
        q, k, v = outs
    elif pattern == "zeros_q":
        q = torch.zeros_like(q)
    elif pattern == "equal_k":
        k = k[:, :, :1, :].expand(shape).contiguous()
    else:
        raise ValueError(f"unknown pattern {pattern!r}")
    return (q.to(torch.bfloat16).contiguous(), k.to(torch.bfloat16).contiguous(),
            v.to(torch.bfloat16).contiguous())


def make_workload(w: Workload, seed: int = 0):
    return make_qkv(w.B, w.H, w.N, w.D, w.pattern, seed)


def make_dout(B: int, H: int, N: int, D: int, seed: int = 0, std: float = 0.01):
    """Output gradient dO for the training shapes: bf16 N(0, std) of shape
    [B, H, N, D], from its own generator (seed + 7919) so that Q, K, V stay
    those of make_qkv with the same seed."""
    g = torch.Generator("cpu").manual_seed(seed + 7919)
    d = torch.randn((B, H, N, D), generator=g, dtype=torch.float32) * std
    return d.to(torch.bfloat16).contiguous()
