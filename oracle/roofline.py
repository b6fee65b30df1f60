"""Cycle model behind the forward and backward roofline tables.

Test infrastructure only (see the package docstring).

Source: "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
Asymmetric Hardware Scaling", Table 1 (forward) and Table 3 (backward); the
unit rates come from "FlashAttention 3 and 4: When the Bottleneck Moves",
section 3.2: 8192 BF16 tensor-core FLOPs and 16 exponentials per cycle per SM.

Reading: the pages do not print the shared-memory rate.  128 bytes per cycle
per SM is the one value that reproduces every shared-memory cell of both
tables when each matrix product reads its shared-memory operands once and the
operands kept in tensor memory (P^T and dS^T in the backward) cost nothing.
"""
from __future__ import annotations

MMA_FLOPS_PER_CLK = 8192
EXP_PER_CLK = 16
SMEM_BYTES_PER_CLK = 128
BF16 = 2
FP32 = 4


def _mma(m: int, n: int, k: int) -> float:
    return 2.0 * m * n * k / MMA_FLOPS_PER_CLK


def forward_tile(m: int, n: int, d: int) -> dict:
    """One m-row Q block against one n-key tile, head dim d (m is 128 or 256).

    Products: S = Q K^T and O += P V (P from tensor memory), each split into
    128-row products.  Shared-memory reads: the Q block once, K and V once per
    128-row product.  Exponentials: one per score.
    """
    q_tiles = m // 128
    mma = _mma(m, n, d) + _mma(m, d, n)
    smem_bytes = m * d * BF16 + q_tiles * (n * d * BF16) * 2
    return {"mma": mma, "smem": smem_bytes / SMEM_BYTES_PER_CLK, "exp": m * n / EXP_PER_CLK}


def backward_tile_1cta(m: int = 128, n: int = 128, d: int = 128) -> dict:
    """1-CTA backward step for one (Q tile, KV tile) pair.

    Five products: S^T = K Q^T, dP^T = V dO^T, dV += P^T dO, dK += dS^T Q,
    dQ = dS K.  Ten operand tiles, two of which (P^T and dS^T) live in tensor
    memory, leave eight bf16 tiles read from shared memory.  dS is written to
    shared memory once; the FP32 dQ tile is written to and read back from
    shared memory on its way to the global accumulator.
    """
    mma = 5 * _mma(m, n, d)
    operands = 8 * (m * d * BF16)
    return {"mma": mma,
            "smem_operands": operands / SMEM_BYTES_PER_CLK,
            "smem_ds_write": m * n * BF16 / SMEM_BYTES_PER_CLK,
            "smem_ds_dsmem": 0.0,
            "smem_dq": 2 * m * d * FP32 / SMEM_BYTES_PER_CLK}


def backward_tile_2cta(m: int = 256, n: int = 128, d: int = 128) -> dict:
    """2-CTA backward step, per CTA of the pair (pair tile m = 256 keys).

    Each CTA supplies its own 128-row A operand and half of every B operand.
    Per CTA: S^T and dP^T read a 128-row A tile and half a B tile; dV and dK
    take A from tensor memory and read half a B tile; the dQ product runs with
    a doubled reduction (2n keys), each CTA reading a (m/2 x 2n) dS operand and
    half of the stacked K.  dQ is half as large per CTA.  The shared-memory
    cost of the dS exchange is not modelled (the table's 384-cycle cell is
    left unexplained).
    """
    half = m // 2
    mma = 5 * _mma(half, n, d)
    a_tile = half * d * BF16
    b_half = (n // 2) * d * BF16
    ds_pair = (half // 2) * (2 * n) * BF16
    k_pair_half = (d // 2) * (2 * n) * BF16
    operands = (a_tile + b_half) * 2 + b_half * 2 + ds_pair + k_pair_half
    return {"mma": mma,
            "smem_operands": operands / SMEM_BYTES_PER_CLK,
            "smem_ds_write": half * n * BF16 / SMEM_BYTES_PER_CLK,
            "smem_dq": 2 * (half // 2) * d * FP32 / SMEM_BYTES_PER_CLK}
