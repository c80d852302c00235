"""CPU oracle for the W4A16 group-32 decode path (test infrastructure only).

This package is the slow, plain, obviously-correct definition of what the CUDA
library computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it; the
product path (the C-ABI library and its Python binding) never does, and this
package imports nothing from the product.

Modules
-------
ref         dequantisation, GEMV, routed-expert GEMV (plain and with per-expert
            output vectors by real id), row gather, quantiser,
            bf16 rounding and the acceptance bound (NumPy, fp64).
lfu         the per-layer LFU expert-slot pool policy (pure Python).
magic_check.c
            exhaustive check, in plain C, of the float-bit dequantisation
            identities the kernels rely on.
"""

from .ref import (  # noqa: F401
    GROUP,
    NIBBLES_PER_WORD,
    bf16_bits_to_f64,
    bf16_rne,
    ulp_bf16,
    unpack_codes,
    pack_codes,
    dequant,
    gemv_ref,
    gemv_abs_ref,
    gemv_values_ref,
    silu_mul_ref,
    gemv_id_ref,
    gemv_id_scaled_ref,
    gather_ref,
    quantize_ref,
    within_bound,
    bound_violations,
)
from .lfu import LFUSlotPoolRef  # noqa: F401
