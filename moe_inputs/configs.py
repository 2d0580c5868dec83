"""Layer shapes and input recipes.

Shapes follow the layers the DeepSeekMoE pages describe:
- the DeepSeek-V3 MoE layer: hidden 7168, 256 fine-grained routed experts of
  intermediate size 2048, 8 routed + 1 shared expert active per token
  ("DeepSeekMoE架构解析", section 1; "DeepSeek-V3：MoE大模型架构");
- the January-2024 DeepSeekMoE 16B layer: 2 shared + 64 routed experts,
  2 + 6 active per token, gates not renormalised (course chapter "MoE",
  sections 2 and 4).
Initialisation std 0.006 comes from the V3 walk-through, section 4.1.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

F32 = "f32"
BF16 = "bf16"
E4M3 = "e4m3"

SIGMOID = 0
SOFTMAX = 1


@dataclass(frozen=True)
class LayerCfg:
    name: str
    T: int          # tokens in the batch
    d: int          # hidden size
    E: int          # routed experts
    K: int          # routed experts chosen per token (K_r)
    S: int          # shared experts
    I: int          # expert intermediate size (routed and shared)
    act: str        # activation / token dtype
    wgt: str        # weight and centroid dtype
    x_std: float = 1.0
    w_std: float = 0.02
    bias_range: float = 0.0      # bias ~ U(-r, r); 0 means bias = 0
    normalize: int = 1           # 1: renormalise chosen gates; 0: 2024 variant
    score_func: int = SIGMOID    # SIGMOID (V3) or SOFTMAX (2024)
    add_residual: int = 1
    gamma: float = 1e-3
    seed: int = 0
    zipf_s: float = 0.0          # > 0: expert popularity ~ rank^-zipf_s (see gen.py)
    n_groups: int = 0            # node-limited routing: expert groups (0 = off)
    topk_groups: int = 0         # groups kept per token

    def with_(self, **kw) -> "LayerCfg":
        return replace(self, **kw)

    @property
    def rows_total(self) -> int:
        """Rows of the expert-ordered activation buffers: T*K routed + S*T shared."""
        return self.T * self.K + self.S * self.T

    def gemm_flops(self) -> int:
        """Algorithmic FLOPs of the expert GEMMs: 6*d*I per (token, expert) pair."""
        return 6 * self.d * self.I * (self.T * self.K + self.T * self.S)

    def router_flops(self) -> int:
        return 2 * self.T * self.d * self.E


CONFIGS = {
    # tiny correctness layer, fp32
    "tiny": LayerCfg("tiny", T=64, d=256, E=16, K=4, S=1, I=128, act=F32, wgt=F32,
                     w_std=0.02, bias_range=0.0, normalize=1),
    # V3-shaped decode batch: weight streaming
    "v3_decode": LayerCfg("v3_decode", T=128, d=7168, E=256, K=8, S=1, I=2048,
                          act=BF16, wgt=BF16, w_std=0.006, bias_range=0.01),
    # V3-shaped prefill batch: the throughput workload
    "v3_prefill": LayerCfg("v3_prefill", T=8192, d=7168, E=256, K=8, S=1, I=2048,
                           act=BF16, wgt=BF16, w_std=0.006, bias_range=0.01),
    # V3 layer with Zipf-skewed expert popularity and FP8 block-scaled weights
    "v3_skewed_fp8": LayerCfg("v3_skewed_fp8", T=16384, d=7168, E=256, K=8, S=1, I=2048,
                              act=BF16, wgt=E4M3, w_std=0.006, bias_range=0.0,
                              zipf_s=1.1),
    # DeepSeekMoE-16B-shaped layer, softmax scores, no renormalisation
    "dsmoe16b": LayerCfg("dsmoe16b", T=32768, d=2048, E=64, K=6, S=2, I=1408,
                         act=BF16, wgt=BF16, w_std=0.02, bias_range=0.0,
                         normalize=0, score_func=SOFTMAX),
}


def get_config(name: str) -> LayerCfg:
    return CONFIGS[name]


def small_cases() -> dict:
    """Reduced layers that the oracle finishes in seconds, yet span several
    tiles of every kernel, ragged expert groups and ragged token tails."""
    v3 = CONFIGS["v3_prefill"]
    return {
        "tiny": CONFIGS["tiny"],
        "small_bf16": v3.with_(name="small_bf16", T=512, d=512, E=32, K=4, S=1, I=256,
                               w_std=0.03),
        "ragged_bf16": v3.with_(name="ragged_bf16", T=301, d=384, E=24, K=3, S=2, I=384,
                                w_std=0.03, bias_range=0.02),
        "softmax_norenorm": CONFIGS["dsmoe16b"].with_(name="softmax_norenorm", T=640,
                                                      d=256, E=64, K=6, S=2, I=128),
        "sigmoid_norenorm": v3.with_(name="sigmoid_norenorm", T=256, d=256, E=16, K=2,
                                     S=1, I=128, normalize=0, w_std=0.03),
        "wide_e": v3.with_(name="wide_e", T=200, d=256, E=512, K=16, S=1, I=128,
                           w_std=0.03, bias_range=0.01),
        "tiny_f32_ragged": CONFIGS["tiny"].with_(name="tiny_f32_ragged", T=37, d=96,
                                                 E=8, K=3, S=2, I=40),
        # node-limited routing: 8 groups of 4 experts, 3 kept (V3 uses 8 nodes, 4 kept)
        "grouped_bf16": v3.with_(name="grouped_bf16", T=512, d=512, E=32, K=4, S=1, I=256,
                                 w_std=0.03, bias_range=0.01, n_groups=8, topk_groups=3),
        # FP8 block-scaled experts, Zipf-skewed routing (one expert takes every token)
        "small_fp8": CONFIGS["v3_skewed_fp8"].with_(name="small_fp8", T=600, d=512, E=32,
                                                    K=4, S=1, I=384, w_std=0.03),
        "ragged_fp8": CONFIGS["v3_skewed_fp8"].with_(name="ragged_fp8", T=301, d=384, E=24,
                                                     K=3, S=2, I=256, w_std=0.03, zipf_s=0.0,
                                                     bias_range=0.02),
    }
