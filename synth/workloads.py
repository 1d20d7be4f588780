"""The five layer shapes the MoE forward is built and measured on.

Each entry fixes the shapes, the routing variant and the input recipe; the
token count T is chosen per run.  Routing variants (Cross-Platform Fused MoE
Dispatch in Triton, review: the method runs the standard softmax/sigmoid
router with top-k selection of Mixtral, DeepSeek-V3 and Qwen2-MoE layers):

* tiny / mixtral: softmax over all E, top-k, weights renormalised over the k.
* qwen2: softmax over all 64, top-8, raw softmax weights, plus one always-on
  shared SwiGLU expert scaled by sigmoid(x . w_s).
* skew: softmax with renormalised top-4 and a per-expert logit bias log(p_e),
  p_e proportional to rank^-alpha.
* deepseek: sigmoid scores, group-limited top-8 (8 groups of 32, group score
  = sum of its top-2, keep 4 groups), weights normalised to sum 1 then x2.5,
  plus one shared SwiGLU expert (scale 1).
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    F: int
    E: int
    k: int
    score: str = "softmax"          # "softmax" | "sigmoid"
    renormalize: bool = True
    route_scale: float = 1.0
    n_group: int = 1                # 1 = plain top-k
    topk_group: int = 1
    group_topn: int = 0
    F_shared: int = 0               # 0 = no shared expert
    shared_gate: bool = False       # shared expert scaled by sigmoid(x . w_s)
    alpha: float | None = None      # Zipf skew exponent (adds a logit bias)
    activation: str = "silu"        # gate activation: "silu" (SwiGLU) or "gelu" (GEGLU)
    seed: int = 0

    def with_T(self, T: int) -> "Workload":
        return replace(self, T=T)

    @property
    def label(self) -> str:
        s = f"{self.name} T={self.T} H={self.H} F={self.F} E={self.E} k={self.k}"
        if self.F_shared:
            s += f" Fs={self.F_shared}"
        if self.alpha is not None:
            s += f" alpha={self.alpha:g}"
        if self.activation != "silu":
            s += f" act={self.activation}"
        return s

    # Algorithmic work of one forward over T tokens (elementwise work excluded).
    def flops(self) -> float:
        f = self.T * (2.0 * self.H * self.E + self.k * 6.0 * self.H * self.F)
        if self.F_shared:
            f += self.T * 6.0 * self.H * self.F_shared
            if self.shared_gate:
                f += self.T * 2.0 * self.H
        return f

    def compulsory_bytes(self, active_experts: int) -> float:
        """x read + router weights + weights of experts with >= 1 routed row + out."""
        b = 2.0 * self.T * self.H * 2 + 2.0 * self.E * self.H
        b += active_experts * 6.0 * self.H * self.F
        if self.F_shared:
            b += 6.0 * self.H * self.F_shared
            if self.shared_gate:
                b += 2.0 * self.H
        if self.alpha is not None:
            b += 4.0 * self.E
        return b


TINY = Workload("tiny", T=128, H=512, F=1024, E=8, k=2)
MIXTRAL = Workload("mixtral", T=4096, H=4096, F=14336, E=8, k=2)
QWEN2 = Workload("qwen2", T=512, H=3584, F=2560, E=64, k=8, renormalize=False,
                 F_shared=20480, shared_gate=True)
SKEW = Workload("skew", T=512, H=2048, F=1408, E=64, k=4, alpha=0.0)
DEEPSEEK = Workload("deepseek", T=8192, H=7168, F=2048, E=256, k=8, score="sigmoid",
                    route_scale=2.5, n_group=8, topk_group=4, group_topn=2, F_shared=2048)

# The second Mixtral shape the review lists ("Mixtral-8x7B/22B"): the published
# Mixtral-8x22B expert layer.
MIXTRAL22B = Workload("mixtral22b", T=4096, H=6144, F=16384, E=8, k=2)

WORKLOADS = {w.name: w for w in (TINY, MIXTRAL, QWEN2, SKEW, DEEPSEEK, MIXTRAL22B)}

# Token counts each workload is run at.
T_SWEEP = {"tiny": (128,), "mixtral": (1, 32, 128, 512, 4096), "qwen2": (128, 256, 512),
           "skew": (128, 256, 512), "deepseek": (512, 2048, 8192), "mixtral22b": (1, 32, 128, 512, 4096)}

# Expert-count sweep (the review's Table 5 remark: d_ffn is scaled down as the
# expert count rises to keep total compute about constant; the target is not
# stated).  Reading: E * F is held at the Mixtral-shaped layer's 8 * 14336, so
# the expert parameters (and the weight bytes a small batch streams) stay
# constant; H = 4096, top-2 softmax routing as Mixtral.
EXPERT_SWEEP_E = (8, 16, 32, 64, 128)


def expert_sweep(E: int, T: int) -> Workload:
    if E not in EXPERT_SWEEP_E:
        raise ValueError(E)
    return Workload(f"esweep{E}", T=T, H=4096, F=8 * 14336 // E, E=E, k=2)
SKEW_ALPHAS = (0.0, 1.0, 2.0)


def workload(name: str, T: int | None = None, **kw) -> Workload:
    w = WORKLOADS[name]
    if T is not None:
        w = w.with_T(T)
    if kw:
        w = replace(w, **kw)
    return w
