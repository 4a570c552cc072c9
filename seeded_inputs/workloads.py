"""Workload recipes: shapes, seeds and value distributions of the synthetic inputs.

Kimi-K3 MoE layer shape (LazyLoRA README, "The engine" and the LoRA paragraph of
"File map": 896 routed experts, top-16, experts in the latent space 3584 -> 3072
-> 3584; "Running a 2.78-Trillion-Parameter Model Across Two Desks", Act II:
latent width 3,584, 17.55 MB per MXFP4 expert).

Value distributions:
  * x ~ N(0, 1), router W ~ N(0, 1/d), rounded to the stated dtype;
  * MXFP4 codes uniform over all 16 E2M1 codes; E8M0 scale bytes uniform in
    [scale_lo, scale_hi] (2^(byte-127));
  * RVQ3: three stages of 256 x 8 fp16 codebooks, stage s (1-based) ~ N(0, (0.02/s)^2),
    one set per layer; codes uniform in 0..255 (WASTE README, "3 bits per expert
    weight": residual vector quantisation, 3 stages of 256-entry codebooks over
    8-dim vectors, 3.00 bits/weight);
  * prefill skew: an additive Zipf(s = 1) logit bias b[e] = -ln(e + 1).
The tiny layer's scale range 2^-8..2^-2 is the one its description fixes.  For the
K3-shaped layers no range is given; 2^-9..2^-6 (bytes 118..121) gives expert
weights of rms ~0.026 (the RVQ layer's codebooks give ~0.023) and keeps the
six-layer residual stack finite (SwiGLU is quadratic in its input, so the tiny
layer's range would overflow fp32 by the fourth layer).
"""
import math
from dataclasses import dataclass, replace


@dataclass(frozen=True)
class LayerRecipe:
    name: str
    d: int
    ff: int
    E: int
    k: int
    T: int
    quant: str = "mxfp4"  # "mxfp4" | "rvq3"
    x_dtype: str = "bf16"  # "f32" | "bf16"
    w_dtype: str = "bf16"
    seed: int = 0
    x_sigma: float = 1.0
    scale_lo: int = 118
    scale_hi: int = 121
    bias: str = "none"  # "none" | "zipf"
    zipf_s: float = 1.0
    act: str = "swiglu"  # "swiglu" | "situ"
    n_shared: int = 0  # shared experts: records E .. E + n_shared - 1, every token, weight 1
    bias_mode: str = "logit"  # "logit": the bias enters selection and gates | "select": selection only

    @property
    def w_sigma(self):
        return 1.0 / math.sqrt(self.d)

    def with_(self, **kw):
        return replace(self, **kw)


K3 = dict(d=3584, ff=3072, E=896, k=16)

WORKLOADS = {
    # d=256, ff=128, E=16, top-4, 8 tokens, fp32 x and router W, seed 0
    "tiny": LayerRecipe("tiny", d=256, ff=128, E=16, k=4, T=8, x_dtype="f32", w_dtype="f32", seed=0,
                        scale_lo=119, scale_hi=125),
    # K3 layer, decode batch 1, all 896 MXFP4 experts resident
    "k3_mxfp4_decode": LayerRecipe("k3_mxfp4_decode", T=1, seed=1, **K3),
    # the same decode layer with 64 experts (1.1 GB): the small case for detailed
    # profiler captures; one token still streams 16 experts (281 MB > L2)
    "k3_mxfp4_decode_e64": LayerRecipe("k3_mxfp4_decode_e64", T=1, seed=1, **dict(K3, E=64)),
    "k3_rvq3_decode_e64": LayerRecipe("k3_rvq3_decode_e64", T=1, seed=2, quant="rvq3", **dict(K3, E=64)),
    "k3_rvq3_decode_b8_e64": LayerRecipe("k3_rvq3_decode_b8_e64", T=8, seed=2, quant="rvq3", **dict(K3, E=64)),
    # K3 layer with RVQ3 experts, decode batch 1 and batch 8
    "k3_rvq3_decode_b1": LayerRecipe("k3_rvq3_decode_b1", T=1, seed=2, quant="rvq3", **K3),
    "k3_rvq3_decode_b8": LayerRecipe("k3_rvq3_decode_b8", T=8, seed=2, quant="rvq3", **K3),
    # the K3 MoE block with its 2 shared experts beside the 896 routed ones and
    # the score-correction bias (here the Zipf prior) steering the selection
    # only; decode batch 1 (18 records per token), and a small parity case
    "k3_mxfp4_decode_shared2": LayerRecipe("k3_mxfp4_decode_shared2", T=1, seed=4, bias="zipf", bias_mode="select",
                                           n_shared=2, **K3),
    "k3_mxfp4_prefill_shared2_e64": LayerRecipe("k3_mxfp4_prefill_shared2_e64", T=40, seed=4, bias="zipf",
                                                bias_mode="select", n_shared=2, **dict(K3, E=64)),
    # K3 prefill, 512 tokens: Zipf-skewed routing and the uniform control
    "k3_mxfp4_prefill_zipf": LayerRecipe("k3_mxfp4_prefill_zipf", T=512, seed=3, bias="zipf", **K3),
    "k3_mxfp4_prefill_uniform": LayerRecipe("k3_mxfp4_prefill_uniform", T=512, seed=3, **K3),
    # small cases of the prefill kernels for detailed profiler captures (64
    # experts, 1.1 GB): Zipf-skewed buckets of up to ~500 tokens, and 40 tokens
    # (about 10 per expert, the size of a uniform 512-token bucket over 896)
    "k3_mxfp4_prefill_zipf_e64": LayerRecipe("k3_mxfp4_prefill_zipf_e64", T=512, seed=3, bias="zipf",
                                             **dict(K3, E=64)),
    "k3_mxfp4_prefill_b40_e64": LayerRecipe("k3_mxfp4_prefill_b40_e64", T=40, seed=3, **dict(K3, E=64)),
}

STACK_LAYERS = 6
STACK_T = 64


def stack_layer(layer):
    """Layer `layer` (0-based) of the six-layer K3 stack: its own seed, 64 tokens."""
    return LayerRecipe(f"k3_mxfp4_stack_l{layer}", T=STACK_T, seed=100 + layer, **K3)


def get_workload(name):
    return WORKLOADS[name]
