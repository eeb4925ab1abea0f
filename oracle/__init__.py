"""CPU oracle for the 4-bit paged KV cache (NVFP4 and INT4 per-token-head).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  It shares no code with the CUDA library.

The oracle restates, step by step and in plain numpy, what the pages define:

* ``formats``   -- the E2M1 element, the E4M3 block scale and the bf16 input
  type, from their bit definitions ("SGLang's 4-bit KV cache: the 56% is
  exact", Figure 2 caption and the section "The 56% survives its own scale").
* ``quant``     -- NVFP4 block quantisation (16 elements per E4M3 scale, one
  FP32 global scale) and the INT4 per-token-head encoding ("KV cache in 4
  bits", section "What we changed").
* ``pool``      -- the paged pool: request -> token -> slot -> page bytes
  (Figure 2 caption: the memory system that assigns tokens to slots).
* ``attention`` -- exact FP64 softmax attention over the dequantised cache,
  the split-KV log-sum-exp combine, the dequantisation of a cached prefix
  into an FP8 E4M3 workspace, and the chunk's attention over that prefix
  plus itself (Figure 2, the chunked prefill and extend column).

Every function is pinned by ``tests/test_oracle_*.py`` against something
other than itself (library casts, closed forms, brute force, the pages'
printed byte counts).  The one reading that no pin can fix -- the INT4 scale
bytes holding two FP32 symmetric scales -- is marked "parity unpinned" in
``quant.py``.
"""
from . import formats, quant, pool, attention  # noqa: F401
