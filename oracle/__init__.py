"""CPU oracle for decode-step attention over a paged KV cache.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only the test suite, the package's smoke
check and the benchmark's CPU-baseline / reference arm may import this package.
The CUDA library never calls it, and it never calls the CUDA library: the two
share no code. The only thing both sides consume is the seeded input generator
in ``workloads``, which holds no attention arithmetic.

Everything here is plain numpy in float64 (bf16 inputs are widened exactly).
Each function restates the operation from the pages it cites:

* SwiftLLM page (l189.com), section 3.1 "PagedAttention and KV cache management"
  and section 5.1 (attention takes the query, the block tables and the context
  lengths): pages of fixed size addressed through a per-request block table.
* TokenSpeed deep dive (wth2jhl.online), section 7 "MLA decode", fig. 3 and
  section 7.1: split-KV partial outputs carry a log-sum-exp and are reduced by it.
* tokenspeed 딥다이브 (fiv.co.kr), section 6-4: fp8 token-group quantization
  (scale = group max / fp8 max, clamp, cast; reconstruction = code * scale).
* TokenSpeed deep dive (wth2jhl.online), section 0 and the closing section:
  tree speculation (draft tokens verified in one step under an ancestor mask).
* TokenSpeed deep dive (wth2jhl.online), section 4.1, and tokenspeed 딥다이브
  (fiv.co.kr), section 6-3: sliding-window KV groups (the last
  ``sliding_window_tokens`` tokens, placeholders in front of the window).
* Tokasaurus blog (Stanford), "Dynamic prefix identification and exploration":
  shared-prefix (Hydragen / cascade) attention over greedily found shared prefixes.

Pins for every function live in ``tests/test_oracle_*.py``; each function's
docstring names the pins that tie it to something other than itself.
"""

from .attention import (
    gather_sequence,
    decode_attention,
    decode_attention_window,
    fold_sq_factor,
    multi_query_decode_attention,
    tree_ancestors,
    tree_verify_decode_attention,
    mla_decode_attention,
    mla_multi_query_decode_attention,
    merge_states,
    merge_states_many,
    kv_append,
)
from .prefix_groups import check_prefix_groups, check_prefix_forest, shared_depth_brute_force, PrefixGroups
from .fp8 import (
    e4m3_decode,
    e4m3_encode,
    quantize_token_groups,
    dequantize,
    kv_append_fp8,
    decode_attention_fp8,
    mla_decode_attention_fp8,
)

__all__ = [
    "gather_sequence",
    "decode_attention",
    "fold_sq_factor",
    "multi_query_decode_attention",
    "tree_ancestors",
    "tree_verify_decode_attention",
    "mla_decode_attention",
    "mla_multi_query_decode_attention",
    "merge_states",
    "merge_states_many",
    "kv_append",
    "check_prefix_groups",
    "check_prefix_forest",
    "shared_depth_brute_force",
    "e4m3_decode",
    "e4m3_encode",
    "quantize_token_groups",
    "dequantize",
    "kv_append_fp8",
    "decode_attention_fp8",
    "mla_decode_attention_fp8",
    "PrefixGroups",
]
