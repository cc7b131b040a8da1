"""Float64 CPU oracle for INT4-KV attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code with the CUDA path (no kernels, headers, helpers, tables or
constant generators) and imports nothing from the product package.

Modules
-------
codec      -- symmetric INT4 per-(token, kv-head) quantizer, nibble packing,
              dequantization (the KV-cache format).
attention  -- unfused attention over the dequantized cache: GQA, causal
              (bottom-right aligned), variable lengths, paged gather, and the
              log-sum-exp merge of split partials.
codec3, codec2 -- the INT3 and INT2 per-row codecs.
headwise   -- headwise mixed 2/4-bit precision: priorities and the bit plan.
flashq     -- the int8 decode buffer with a universal scale, and its flush.
baselines  -- the comparison paths: attention over an FP16 cache, and the
              cache dequantized to FP16 first, then attended.
progressive -- progressive INT8 -> INT4 storage: 64-token blocks, symmetric
              int8 with one FP16 scale, then channel-wise asymmetric 4-bit
              codes with an integer scale and zero point per channel.

Every function cites the passage of the source pages it follows.  Where the
pages are silent or garbled the reading taken is stated in the docstring.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against values fixed by the pages or by mathematics (hand-derived vectors,
exact-rational rounding, closed forms, an mpmath brute force, and PyTorch's
``scaled_dot_product_attention`` in float64 as the textbook special case).
"""

from . import codec, attention  # noqa: F401
