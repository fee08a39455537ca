"""CPU oracle (test infrastructure only; never imported by the product path).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. See ``oracle/oracle.py`` for the rules
it restates and the sources it follows.
"""
from .oracle import *  # noqa: F401,F403
from .oracle import (  # noqa: F401
    QK, Q8_0_BLOCK_BYTES, Q4_0_BLOCK_BYTES, GEMV_RTOL, GEMV_ATOL, GEMM_RTOL, GEMM_ATOL,
    f32_to_f16_bits, f16_bits_to_f32, f32_to_bf16_rne, pack_f16, quantize_q8_0,
    quantize_q4_0, pack, dequantize_q8_0, dequantize_q4_0, dequantize_f16, dequantize,
    unpack_q4_0_codes, packed_row_bytes, matmul_ref, reference, argmax_first,
)
