"""fp64 CPU oracle for tree verification — test infrastructure only.

Imported by the tests, the smoke check and the benchmark's CPU-baseline leg;
never by the product path.
"""
from .treeverify_oracle import *  # noqa: F401,F403
from .treeverify_oracle import (tree_build_mask, tree_verify_attn, tree_accept_greedy,  # noqa: F401
                                tree_accept_sampling, kv_commit_path, node_plan, node_plan_wor, softmax_t,
                                inverse_cdf, accept_test, ancestors_or_self, bf16_to_f64,
                                tree_is_valid, draft_entropy, branch_width, top_tokens,
                                log_softmax_at, tree_expand_level, tree_build_dynamic,
                                kv_prune_pages, dequantize_q4, tree_verify_attn_q4,
                                f64_to_bf16_bits_via_f32, quantize_q4, q3_code_values, q3_pack,
                                dequantize_q3, tree_verify_attn_q3, quantize_q3)
