"""Plain double-precision CPU oracle for paged mixed-codec decode attention.

TEST INFRASTRUCTURE ONLY.  This package is the independent checker of the CUDA
library: only the test suite, the smoke check and the benchmark's CPU-baseline
leg may import it.  The product path never calls into it, and it shares no code
with the CUDA sources (no kernels, headers, helpers, tables or constants).

It follows three web pages:

* "ARGUS: Heterogeneous KV-cache memory management" (argus-cache 0.5.1 on PyPI),
  sections "Why decode is slow" and "Direct paged attention": codec tiers,
  an exact online softmax over one page at a time with grouped-query
  attention, a structure-of-arrays page table; "Pluggable tiers" (the INT2
  and 1-bit tiers as unsigned_affine with bits = 2 and bits = 1) and "v0.5: model-independent KV
  placement" with the "HuggingFace example" (sliding-window masks, sink
  tokens).
* "feat(kvcache): host-RAM KV tier for sparse-attention models" (FreeToken
  PR #499 and its discussion), sections "Why this works for sparse attention",
  "Design", the update that stores "e4m3 codes + fp32 scales", and the
  comment on in-place host placement: top-k page selection over a compressed
  slab, a logical-to-physical block table, windowed prefill folded by
  log2-sum-exp into a float32 accumulator.
* "Storage contracts for hybrid KV cache offloading", section "Stored-byte
  savings are not a latency result": the transfer lower bound S_wire / B used
  for the roofline.

Attention results are the plain softmax definition evaluated in float64 on the
dequantised stored values; codec encoders are spelled out one IEEE-fp32
operation at a time so that the GPU codes can be compared bit for bit.

Parity pins (see tests/test_oracle_pins.py): every function here is checked
against something other than itself -- a library routine (torch softmax / SDPA
in float64, torch's float8_e4m3fn and bfloat16 conversions), a brute-force
search, an algebraic identity (fold of any partition, block-table permutation
invariance), closed-form special cases, or numbers printed on the pages.
"""

from .codecs import (  # noqa: F401
    CODEC_FP16, CODEC_BF16, CODEC_FP8_E4M3, CODEC_INT8, CODEC_INT4_G32, CODEC_INT2_G32, CODEC_INT1_G32,
    e4m3_value, e4m3_table, e4m3_encode, f16_bits_to_f64, bf16_bits_to_f64,
    round_to_bf16, f64_to_bf16_bits, quantize_unit_fp8, quantize_unit_int8,
    quantize_group_int4, quantize_group_int2, quantize_group_int1, quantize_pages, dequant_page,
)
from .attention import (  # noqa: F401
    softmax_attention, paged_decode, fold_lse, window_attention, visible_positions,
    gather_window, paged_window_attention, staging_moves_less,
)
from .selection import compressed_key_scores, select_pages  # noqa: F401
