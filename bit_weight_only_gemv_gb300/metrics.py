"""Byte accounting and bandwidth arithmetic for the benchmark (no GPU work).

Page "Gemma 4 on a 4 GB GPU in Plain PyTorch", section "Step 3 — Multiply
Straight From the Packed Weights", reports kernel speed as the packed bytes a
decode step reads divided by the time per step (MiB of weights per token over
milliseconds per token, in GB/s), next to a plain memory-read rate of the
same card.  The same form is used here, with the algorithmic bytes of each
call: packed codes, bf16 steps, the activation rows read and the output rows
written.  Re-reads (L2 misses of the activations, split-K partials) are not
counted.
"""

from __future__ import annotations

MIB = 1 << 20
GB = 1e9


def gemv_bytes(M: int, N: int, K: int) -> int:
    """Algorithmic bytes of one W4A16 GEMV: N*K/2 codes + N*K/16 steps + x + y."""
    return N * K // 2 + N * (K // 32) * 2 + 2 * M * K + 2 * M * N


def gemv_id_bytes(n_ids: int, x_rows: int, N: int, K: int) -> int:
    """Routed-expert GEMV: n_ids experts' codes and steps, x rows read, y written."""
    return n_ids * (N * K // 2 + N * (K // 32) * 2) + 2 * x_rows * K + 2 * n_ids * N


def gather_bytes(T: int, K: int) -> int:
    """Row gather: T rows of codes and steps read, T bf16 rows written, T ids."""
    return T * (K // 2 + (K // 32) * 2) + 2 * T * K + 4 * T


def gbps(nbytes: float, seconds: float) -> float:
    return nbytes / seconds / GB


def gemv_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K
