"""CPU oracle for the grouped MoE low-precision path.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check in
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import anything from this package.  The product
library (``fp4_fp8_quantization_gb300``) never imports it, and the CUDA
code shares no code, table or constant generator with it.

Everything here is plain NumPy: element codecs are searches over the code
tables, quantizers follow the fixed sequence of IEEE fp32 operations that
define them, and the GEMMs dequantize to float64 and use a float64 matmul
per expert group.  Module map:

* ``formats``  - E2M1 / E4M3 / E8M0 / bf16 encode-decode, nibble packing.
* ``layout``   - the tiled 128x4 block-scale layout (index function) and the
                 gate/up row interleave of the fused kernel's weight.
* ``quantize`` - per-expert amax and tensor scale, NVFP4 / MXFP8 / MXFP4
                 block quantization, the grouped (ragged, padded) quantizer.
* ``gemm``     - grouped rowwise-scaled FP8 GEMM, grouped block-scaled GEMM.
* ``swiglu``   - the project's exp / reciprocal / SiLU definition (with an
                 exact fp32 fused multiply-add emulation) and the chained
                 SwiGLU + NVFP4 / MX requantization.
* ``dispatch`` - the single-rank expert dispatch: routing of top-k choices
                 to expert groups and MXFP4 quantization of the routed rows
                 (padded or fixed-slot scale layout).

Pages cited: "grouped_quantize_dynamic_scaled_fp4_async_kernel" (Mojo kernel
doc), "grouped_matmul_rowwise_dynamic_scaled_fp8" (Mojo function doc),
"max.nn.moe.NvMxf4f8Strategy" (Python class doc), "Struct_ep_dispatch_mxfp4"
(Mojo graph-op doc).

Parity unpinned: behaviour on NaN / Inf inputs (the synthetic data holds
none and the library leaves it undefined).
"""
