"""sub_byte_mixed_gb300: the quantized linear layer of sub-byte mixed-precision
LLM training (SNIP's per-layer FP8/NVFP4 plan; NVFP4 = 16 E2M1 values sharing an
E4M3 scale, round-to-nearest forward, stochastic rounding backward), as
hand-written CUDA for sm_103a behind a C ABI (``include/snip.h``).

``sub_byte_mixed_gb300.snip`` is the thin ctypes binding of that ABI; it loads
``_build/libsnip.so`` and raises if the library is missing.  Importing this
package itself loads nothing, so the input generators in ``inputs`` work on
machines without a GPU.
"""
