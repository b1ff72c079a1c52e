"""Named synthetic workloads: shapes, element types, tree recipes, acceptance rules.

Each entry describes one Medusa verify step at a model shape.  The pages that
define the method measure on Vicuna-7B/13B/33B with MT-Bench and AlpacaEval
prompts ("Medusa: Simple LLM Inference Acceleration Framework with Multiple
Decoding Heads", Results; explainer "085 | Medusa", section 四); neither the
weights nor the prompts are available here, so random tensors of those model
shapes stand in for them.

Tree recipes:
  ("cartesian", s, max_nodes)  every path with rank i_k <= s_k, breadth-first,
                               cut after max_nodes non-root nodes (None = all)
  ("greedy", budget, R)        greedy sparse tree from the synthetic per-head
                               accuracy table a_k^(i) = 0.6 * 0.7^(k-1) * 0.5^(i-1)
"""
from __future__ import annotations

WORKLOADS = {
    # Tiny fp32 step: the case the oracle finishes in well under a second.
    "tiny_fp32": dict(
        dtype="f32", d=256, V=1024, H=4, Dh=64, B=1, L=(64,), K=3,
        tree=("cartesian", (2, 2, 2), None), mode="greedy",
        w1_std=0.02, lm_std="inv_sqrt_d", w2="lm_plus_noise", w2_noise_std=0.01,
    ),
    # Tiny bf16 step on the tensor-core paths (Dh 128; 300 prefix + 15 tree keys
    # give the attention a ragged third key tile, V = 2048 sixteen vocabulary tiles).
    "tiny_bf16": dict(
        dtype="bf16", d=256, V=2048, H=2, Dh=128, B=1, L=(300,), K=3,
        tree=("cartesian", (2, 2, 2), None), mode="greedy",
        w1_std="inv_sqrt_d", lm_std="inv_sqrt_d", w2="independent",
    ),
    # Vicuna-7B-shaped single-sequence step (the headline).
    "vicuna7b_L1024_tree64": dict(
        dtype="bf16", d=4096, V=32000, H=32, Dh=128, B=1, L=(1024,), K=4,
        tree=("greedy", 64, 10), mode="greedy",
        w1_std="inv_sqrt_d", lm_std="inv_sqrt_d", w2="independent",
    ),
    # Vicuna-13B-shaped step with typical acceptance.
    "vicuna13b_L2048_tree64_typical": dict(
        dtype="bf16", d=5120, V=32000, H=40, Dh=128, B=1, L=(2048,), K=5,
        tree=("greedy", 64, 10), mode="typical", eps=0.09, delta=0.3, temperature=0.7,
        w1_std="inv_sqrt_d", lm_std="inv_sqrt_d", w2="independent",
    ),
    # Tree-size sweep at the 7B shape, long prefix.
    "vicuna7b_L4096_tree64": dict(
        dtype="bf16", d=4096, V=32000, H=32, Dh=128, B=1, L=(4096,), K=4,
        tree=("greedy", 64, 10), mode="greedy",
        w1_std="inv_sqrt_d", lm_std="inv_sqrt_d", w2="independent",
    ),
    "vicuna7b_L4096_dense256": dict(
        dtype="bf16", d=4096, V=32000, H=32, Dh=128, B=1, L=(4096,), K=4,
        tree=("cartesian", (4, 4, 4, 4), 256), mode="greedy",
        w1_std="inv_sqrt_d", lm_std="inv_sqrt_d", w2="independent",
    ),
    # 33B-shaped batch of 4 ragged sequences, typical acceptance.
    "vicuna33b_bs4_ragged": dict(
        dtype="bf16", d=6656, V=32000, H=52, Dh=128, B=4, L=("uniform", 512, 8192), K=5,
        tree=("greedy", 64, 10), mode="typical", eps=0.09, delta=0.3, temperature=0.7,
        w1_std="inv_sqrt_d", lm_std="inv_sqrt_d", w2="independent",
    ),
}

HEADLINE = "vicuna7b_L1024_tree64"


def get(name: str) -> dict:
    w = dict(WORKLOADS[name])
    w["name"] = name
    return w
