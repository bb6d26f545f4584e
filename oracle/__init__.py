"""CPU oracle for exact attention: test infrastructure, not product code.

Only the tests, the smoke check and the bench's CPU-baseline / reference arm
use this package.  The CUDA library never imports, links or calls it, and it
imports nothing from the CUDA library: the two share only the seeded input
generators in ``fa_inputs``.

Contents
--------
``attention``   float64 NumPy definitions: dense, varlen and decode attention
                (materialised S, safe softmax, P V, log-sum-exp), the
                (m, d, o) state, its merge and folds, and split-KV chunk states.
``combine_f32`` a plain C fp32 fold of split-KV states in a fixed order, with
                its own exp2 / log written from textbook methods, so that a
                GPU combine with the same operation sequence can be compared
                bit for bit (loaded through ctypes; built by ``build``).

Sources: "Learning FlashAttention the Hard Way - Part 1" (cloudrift.ai),
sections "Softmax Looks Like It Breaks the Rules", "Online Softmax
Reparametrization", "FlashAttention: Not So Special", "The State", "The Merge,
and the Twist", "Numerical Analysis of the FlashAttention Kernel",
"Alternative Twist: Base 2"; "Associativity is All You Need" for split-K.
"""
