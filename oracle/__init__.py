"""FP64 CPU oracle for exact attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU
baseline leg of the benchmark may import this package.  The library's compute
path never calls it, and it shares no code with the CUDA sources: the two meet
only through the seeded input generator in ``synth``.

Contents
--------
attention   the plain definition of scaled-dot-product attention (two-pass
            softmax over a materialised score matrix) and its explicit
            chain-rule backward; the tiled online-softmax algorithm with
            conditional rescaling, written out step by step.
exp2_poly   the 2^x polynomial emulation: our own minimax fit and its error
            table.
roofline    the cycle model behind the forward and backward roofline tables.
merge       attention over a key range (split-KV partials) and the associative
            merge of such partials.
fp8         the e4m3 format, the Hadamard rotation of Q and K, power-of-two
            block scales, and the FP8 forward (online softmax with P
            rounded to e4m3) from quantised inputs.
masks       attention under a sliding-window mask and a block mask (forward
            and chain-rule backward), and the tile pairs such a mask leaves
            visible.

Every function is pinned by a CPU test against something other than itself
(brute force, finite differences, closed forms, invariants, or the numbers
printed in the pages).  No function here is "parity unpinned".
"""
