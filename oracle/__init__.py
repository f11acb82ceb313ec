"""CPU oracle for the INT8 KV cache and split-K decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, header, table or helper with the CUDA path under
``int8_kv_cache_02_gb300/`` and imports nothing from it.

What it computes, and where each step comes from:

* ``quant``     -- fp16 -> int8 absmax/127 quantization, one fp16 scale per
                   (position, kv head) as in the genie-ai-runtime INT8 KV cache
                   (release v0.1.0-alpha.12, "Path I series", rows I1-I3;
                   release v0.1.0-alpha.11, "--int8-kv triage" table) or one per
                   64 values as in Strata pull request #2698 ("What it does",
                   first bullet, ``kKVG = 64``).
* ``pool``      -- the paged KV pool with a separate scales region
                   (alpha.12 "Path I series", I1) and the append of new tokens
                   through a page table.
* ``attention`` -- decode attention that dequantizes on load (alpha.12 I3:
                   the attention reads ``k_scales[kv_pos * n_kv_heads +
                   kv_head]``), split-K partials and their per-head combine
                   (genie-ai-runtime v1.3.0, "split-K decode attention"), the
                   sliding-window mask (v1.3.0 "Details"), and the causal
                   prefill chunk over the same cache (Strata #2698, "prompt
                   chunk ... dequantize on the fly"; genie v1.3.1).

Precision: quantization decisions are taken in IEEE fp32 exactly as the
method's rounding rule states (scale ``s = fp16_rne(fp32(absmax) / 127)``,
code ``= round_half_even(fp32(x) / fp32(s))`` clamped to [-127, 127]);
attention is evaluated in fp64 over the exactly dequantized cache.

Pins: every function here is checked in ``tests/test_oracle_*.py`` against
something other than itself -- exact rational brute force over all fp16
inputs for the scale and the codes, closed forms (context length 1, identical
keys, a dominant key, hand-computed two-key softmax), invariants (key/value
permutation, split-K == single pass, paged == contiguous), the page text's
528 B/cell figure, and hand-written fixtures under ``tests/golden/``.
"""

from . import quant, pool, attention  # noqa: F401

__all__ = ["quant", "pool", "attention"]
