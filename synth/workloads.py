"""Shapes of the synthetic VLA workloads.

Each projection is an nn.Linear: weights [N, K], input [M, K], output [M, N].
Projections that read the same tensor (q/k/v read the attention input,
gate/up read the MLP input) share one synthetic input.

Families (hidden size, MLP size, attention layout):
  * gemma2b_prefix   : 2048 hidden, 16384 MLP, 8 query heads x 256, 1 KV head
                       (the VLA's vision-language backbone, 816 prefix tokens);
  * gemma300m_expert : 1024 hidden, 4096 MLP (GeGLU), q/k/v/o 1024 x 1024
                       (the iterative action expert, 50 action tokens);
  * llama2_7b        : 4096 hidden, 11008 MLP (SwiGLU), 32 heads.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Projection:
    name: str
    N: int
    K: int
    input: str  # which distinct input tensor of the layer feeds it


_FAMILIES = {
    "gemma2b_prefix": [
        Projection("q", 2048, 2048, "attn_in"),
        Projection("k", 256, 2048, "attn_in"),
        Projection("v", 256, 2048, "attn_in"),
        Projection("o", 2048, 2048, "o_in"),
        Projection("gate", 16384, 2048, "mlp_in"),
        Projection("up", 16384, 2048, "mlp_in"),
        Projection("down", 2048, 16384, "down_in"),
    ],
    "gemma300m_expert": [
        Projection("q", 1024, 1024, "attn_in"),
        Projection("k", 1024, 1024, "attn_in"),
        Projection("v", 1024, 1024, "attn_in"),
        Projection("o", 1024, 1024, "o_in"),
        Projection("gate", 4096, 1024, "mlp_in"),
        Projection("up", 4096, 1024, "mlp_in"),
        Projection("down", 1024, 4096, "down_in"),
    ],
    "llama2_7b": [
        Projection("q", 4096, 4096, "attn_in"),
        Projection("k", 4096, 4096, "attn_in"),
        Projection("v", 4096, 4096, "attn_in"),
        Projection("o", 4096, 4096, "o_in"),
        Projection("gate", 11008, 4096, "mlp_in"),
        Projection("up", 11008, 4096, "mlp_in"),
        Projection("down", 4096, 11008, "down_in"),
    ],
}

# The projections kept at eight bits in the mixed-precision backbone
# (attention output and feed-forward down projection).
W8A8_PROJECTIONS = ("o", "down")


def layer_projections(family: str):
    return list(_FAMILIES[family])


def input_width(family: str, input_name: str) -> int:
    for p in _FAMILIES[family]:
        if p.input == input_name:
            return p.K
    raise KeyError(input_name)


WORKLOADS = {
    # 1: one W4A4 linear, 16 tokens
    "single_w4a4_16x256": dict(
        M=16, N=256, K=256, hadamard_block=64, act_dist="normal", n_outliers=4,
        outlier_scale=20.0, w_std=0.02, seed=0),
    # 2: batch-1 action expert, weight-only int4 group 128
    "expert_w4a16": dict(
        family="gemma300m_expert", M=50, layers=18, steps=10, group_size=128,
        act_dist="normal", n_outliers=0, outlier_scale=1.0, w_std=0.02,
        spike_frac=0.001, spike_scale=10.0, seed=0),
    # 3: prefix backbone, W4A4 (q,k,v,gate,up) + W8A8 (o, down)
    "prefix_w4a4_w8a8": dict(
        family="gemma2b_prefix", M=816, layers=18, hadamard_block=128,
        act_dist="student_t4", outlier_frac=0.01, outlier_scale=30.0,
        w_std=0.02, seed=0),
    # 4: Llama-2-7B-shaped, every projection at W8A8, W4A4 and W4A16
    "llama2_7b": dict(
        family="llama2_7b", Ms=(1, 64, 512), layers=32, hadamard_block=128,
        group_size=128, act_dist="normal", outlier_frac=0.005,
        outlier_scale=50.0, w_std=0.02, seed=0),
    # 5: full control step: prefix once, then the expert for 10 denoising
    #    steps at W4A4 with static per-step scales and again at W4A16
    "pi05_control_step": dict(
        prefix="prefix_w4a4_w8a8", expert="expert_w4a16", steps=10,
        calib_draws=8, hadamard_block=128, seed=0),
}


def n_outliers(K: int, frac: float) -> int:
    """Outlier channel count for a fraction of K channels (nearest integer)."""
    return int(round(frac * K))
