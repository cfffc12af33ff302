"""Plain fp64 CPU oracle for exact softmax attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run anything in this package.  The
product path (the CUDA library and its Python binding) never imports it, and this
package imports nothing from the product path.

Every function is written from the pages' statement of the method, in float64,
materialising the score matrix S and the probability matrix P on purpose:

* ``attn_fwd_ref``  -- the plain definition O = softmax(scale*Q*K^T) * V and the
  per-row log-sum-exp.
* ``attn_bwd_ref``  -- the textbook gradient of that definition (the pages say only
  that the backward recomputes S and P from Q, K and the saved statistics; the
  formulas are the derivative of the definition above).
* ``attn_rows_ref`` -- the same definition for selected query rows of one head, for
  checks at sequence lengths where whole heads are too costly in float64.
* ``online_softmax_stats`` / ``online_attention_row`` / ``attn_fwd_tiled_ref`` --
  the streaming (m, l) recurrence, used only to check the oracle's own algebra.
* ``attn_cross_head_fwd`` / ``attn_cross_fwd_ref`` -- the definition with Nq query
  rows against Nk keys (causal mask aligned bottom-right) and with grouped key/value
  heads (``kv_head_of``); ``attn_gqa_bwd_ref`` -- its gradient for grouped heads.
* ``merge_partials`` -- attention over a union of disjoint key ranges from the
  attention over each range (the split-key combine).
* ``butterfly_mask`` / ``attn_masked_head_fwd`` / ``attn_masked_head_bwd`` -- the
  definition with a boolean visibility mask, and the fixed butterfly block pattern of
  block-sparse attention.
* ``fp8`` -- the E4M3 format (``e4m3_encode`` / ``e4m3_decode``), the fixed random
  rotation of Q and K (``rotate_exact``, ``rotate_fp32``), block quantization
  (``quantize_blocks`` / ``dequantize_blocks``) and the FP8 forward's reference
  (``attn_fp8_ref``: exact attention on the de-quantised inputs).

Parity pins: every function here is pinned by tests in ``tests/test_oracle_*pins.py``
against printed worked examples, closed forms, invariants, library routines and
central finite differences.  No function is "parity unpinned".
"""

from .attention import (  # noqa: F401
    softmax_two_pass,
    online_softmax_stats,
    online_attention_row,
    attn_fwd_ref,
    attn_fwd_tiled_ref,
    attn_bwd_ref,
    attn_head_fwd,
    attn_head_bwd,
    attn_rows_ref,
    attn_cross_head_fwd,
    attn_cross_fwd_ref,
    attn_gqa_bwd_ref,
    kv_head_of,
    merge_partials,
    butterfly_pairs_visible,
    butterfly_mask,
    attn_masked_head_fwd,
    attn_masked_head_bwd,
)
from .fp8 import (  # noqa: F401
    E4M3_MAX,
    QUANT_BLOCK,
    e4m3_values,
    e4m3_decode,
    e4m3_encode,
    hadamard,
    rotate_exact,
    rotate_fp32,
    quantize_blocks,
    dequantize_blocks,
    attn_fp8_ref,
)
