"""CPU oracle for paged KV-cache attention (test infrastructure only).

Plain, slow, obviously-correct numpy float64 restatement of what the paged
attention path computes.  It exists to check the CUDA library and is imported
only by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py``; the product package never imports it.

Sources (web pages this method is described on):
  [p1] flash-attention #824 "Add support for small page sizes" -- the
       reproduction snippet calling ``flash_attn_with_kvcache`` with a paged
       cache, ``k=``/``v=`` append, ``cache_seqlens``, ``block_table``,
       ``causal=True``; the illegal-memory-access discussion.
  [p2] vLLM #6052 "Unify the kernel used in flash attention backend" -- one
       varlen launch for prefill + decode; cumulative query lengths padded
       with (0, 0) entries for CUDA graphs.
  [p3] flash-attention #1000 "Inappropriate Number of Splits Predicted by
       determine_num_splits" -- split-KV decode on a preallocated contiguous
       cache whose real length comes from ``cache_seqlens``.
  [p4] vLLM #3010 "Introduce flash-attn (>= 2.5.0)" -- paged decode and
       prefill + cache-write benchmarks.
Rotary embedding of the new tokens (``rotary.py``) is only named on [p1]; it
follows the published RoFormer definition, see that module.

Parity pins live in ``tests/test_oracle_pins.py``.  Every function here is
pinned (golden worked examples under ``tests/golden/``, closed forms,
torch's CPU scaled_dot_product_attention on contiguous inputs, brute force,
invariants); none is "parity unpinned".
"""

from .attention import (  # noqa: F401
    PAGE_SIZE,
    kv_head_of,
    visible_keys,
    gather_pages,
    logical_kv,
    attend_rows,
    append_kv,
    fwd_kvcache,
    fwd_varlen,
    split_then_combine,
    combine_splits,
)
from .rotary import round_to, rotary, rotate_new_tokens  # noqa: F401
