"""CPU fp64 oracle for the fused cascaded-reduction kernels.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never calls it, and it shares no code with the CUDA path: the only module
both sides use is the seeded input generator
(``workloads``, at the repository root), which holds none of the method's
arithmetic.

Each cascade is computed the plain, unfused way: every reduction is a
separate full pass over its input, in float64, in the order in which the
method's sources define the cascade.  Sources cited in this package:

[A] "RedFuser: An Automatic Operator Fusion Framework for Cascaded Reductions
    on AI Accelerators", ASPLOS 2026 -- the authors' abstract.
[E] "RedFuser框架：AI加速器中的算子融合技术解析" (explainer article on
    jsqmd.com): §2.1 cascade definition, §2.2 softmax cascade, §2.3
    incremental form, §3.3 execution hierarchy, §4.1 fused attention loop,
    §4.2 MoE routing, §4.3 FP8 quantised GEMM.
[S] gist.science technical summary of the same paper: "Methodologie" 1
    (fusion conditions), 2 (incremental computation), 3 (single- and
    multi-segment code generation).
[OCP] Open Compute Project "OCP 8-bit Floating Point Specification (OFP8)",
    E4M3 format (bias 7, no infinities, max normal 448, NaN = S.1111.111).

Modules: ``attention`` (safe-softmax cascade, its incremental and
multi-segment forms, the latent-KV decode), ``moe_gate`` (gate scores, top-k, softmax of the
selected scores), ``fp8_quant_gemm`` (row absmax, E4M3 quantisation, GEMM,
dequantisation).  Every function is pinned by tests under ``tests/`` against
closed forms, library routines, brute force or worked examples; none is
"parity unpinned".
"""
