"""GB300 (sm_103a) low-bit KV cache: KIVI-style asymmetric 2/4-bit
quantization of keys (per channel, 32-token groups) and values (per token)
with an fp16 window of the newest tokens, and split-K decode attention read
straight from the packed cache.

The compute lives in libkvq.so (C ABI: include/kvq.h).  Modules:
  build  -- compiles csrc/*.cu for sm_103a into libkvq.so (in-tree)
  kvq    -- ctypes binding of the C ABI (argument marshalling only)
  synth  -- seeded synthetic workloads (shapes of the benchmark configs)
"""

__all__ = ["build", "kvq", "synth"]
