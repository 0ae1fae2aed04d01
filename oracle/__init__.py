"""fp64 CPU oracle of the routed Mixture-of-Experts FFN step.

TEST INFRASTRUCTURE ONLY. This package is the plain, slow, obviously correct
definition of what the GPU library computes. Only the tests, the smoke check
and the benchmark's CPU-baseline leg may import it; the library never does,
and it shares no code with the library (the only common dependency is the
seeded input generator, which holds no arithmetic of the method).

See ``oracle.moe`` for the functions and the passages each one follows.
"""
from .moe import (  # noqa: F401
    f16_bits_to_f64, bf16_bits_to_f64, dequant_q4g64, dequant_q2g64, dequant_q8g64,
    router_weights_f64, router_logits, select_topk, routing_weights, silu,
    expert_ffn, moe_token, moe_tokens, RouteInfo, LFUCache, lfu_trace,
    layer_dense_f64, sigmoid_scores, sigmoid_keys, routing_weights_sigmoid, route_keys,
)
