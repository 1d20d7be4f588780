"""CPU oracle of the single-GPU Mixture-of-Experts layer forward.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's CPU
baseline leg import this package; the product path (the CUDA library and its
Python binding) never does, and shares no code with it.  It is plain numpy in
float64, slow and written to be checked by eye against the method's
definition.

``traffic_model_bytes`` (the fused/unfused byte model) is pinned by counting
the bytes an executed fused and unfused SwiGLU sequence moves; the 35 %
figure the review quotes does not follow from the byte counts it prints and
stays unreproduced (parity unpinned for that one figure).
"""
from .moe_oracle import (  # noqa: F401
    Routing,
    widen,
    router_logits,
    router_scores,
    select_experts,
    selection_margin,
    routing_weights,
    permute,
    activate,
    swiglu_expert,
    combine,
    route,
    forward,
    forward_tokens,
    dense_masked_forward,
    traffic_model_bytes,
)
