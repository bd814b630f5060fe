"""CPU oracle for the low-bit KV cache hot path (test infrastructure only).

This package is the slow, plain, obviously-checkable statement of what the
quantize/pack and decode-attention path computes.  It exists to check the CUDA
library, and only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it.  The product path never calls into it: the
CUDA library fails loudly when its shared object is missing rather than fall
back to anything here.

It shares no code with the CUDA path (no kernels, helpers, tables or constant
generators); the only thing both sides read is the packed-format definition in
prose, which each side implements on its own.

Sources, cited by page title and section throughout:

* "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache"
  (fdeinterviews.com): first paragraph (per-token round-to-nearest baseline),
  second paragraph (per-channel keys in 32-token groups, per-token values),
  third paragraph (full-precision window of the newest R = 128 tokens,
  quantized in blocks when it fills).
* "KV cache quantization" (synthetic.wiki): section "Keys are harder than
  values" (per-channel keys, per-token values, Pre-RoPE key quantization with
  RoPE applied after dequantization, grouped + residual split combined when
  computing attention scores); section "What they report" (asymmetric 2-bit
  scheme, attention-sink token kept in fp16, per-vector dense-and-sparse
  outlier isolation).
* "2-Bit KV Cache Quantization: Memory You Save, Recall You Risk"
  (groundy.com): section "The capacity math" (2 vs 16 bits per element);
  section "Method map: three ways to shrink the cache" (Walsh-Hadamard
  rotation as a design decision of a robust low-bit path).

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, invariants, hand-derived golden fixtures or brute force;
no function is "parity unpinned".
"""

from .kivi import (  # noqa: F401
    GROUP,
    block_bytes,
    code_location,
    code_location_table,
    pack_tile,
    unpack_tile,
    quantize_asymmetric,
    quantize_key_group,
    quantize_value_tokens,
    quantize_keys_per_token,
    quantize_dense_sparse,
    dequantize,
    rope_rotate,
    hadamard_rotate,
    hadamard_matrix,
    hadamard_unrotate,
    OracleCache,
    dense_attention,
)
