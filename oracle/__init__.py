"""Plain, slow fp64 CPU oracle for the rotated low-bit KV-cache path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
and its Python binding) may import, call or link anything in this package;
only the tests, the smoke check and the CPU-baseline leg of the benchmark do.
It shares no code with the CUDA path: the one module both sides use is the
seeded input generator, which holds none of the method's arithmetic.

Modules
  fp         exact fp32 fused multiply-add emulation and IEEE fp16 rounding,
             used where a floating-point value decides an integer (a
             quantisation code): the decision is taken in the kernel's fp32
             precision, everything else in fp64.
  attention  GQA decode attention, softmax over s <= t (Output-Aware
             Rotation for INT2 KV-Cache Quantization, §3 Eqs. 1-2).
  int2       rotated INT2 group quantisation D_R(z) = Q2(zR) R^T (§3.1 Eq. 4),
             attention-equivalent key centring (§1), paged cache format,
             packed-cache decode attention.
  bgtq       Gaussian Lloyd-Max codebooks, TQ-MSE encode/decode, greedy
             RoPE-block bit allocation (Theorem 1), grouped encoding and the
             packed Block-GTQ cache (RoPE-Aware Bit Allocation for KV-Cache
             Quantization, prerequisites and method steps (1)-(4)).
  diagnostics  output-space error of a quantised cache: E_rec, E_out and
             the key/value split (Output-Aware Rotation, §3.2 Eqs. 5-10).

Every function is pinned by tests under tests/ that do not re-derive its
formula: closed forms, textbook values, invariants, brute force and exact
rational arithmetic.
"""
