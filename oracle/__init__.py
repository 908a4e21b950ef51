"""CPU oracle for the GPTQ linear layer (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg may
import this package.  The product library never does.  The C source
``gptq_oracle.c`` holds the arithmetic; this module builds it with gcc and wraps
it with ctypes and numpy.
"""
from .oracle import (  # noqa: F401
    build, lib, unpack_codes, pack_codes, unpack_zeros, pack_zeros, num_groups,
    dequant, linear, check_rules, runtime_dims, runtime_layout, num_threads, set_num_threads, half_to_float,
    awq_unpack, awq_pack, awq_dequant, awq_linear, awq_to_gptq_fields, round_fp32,
    e4m3_to_float, fp8_dequant, fp8_linear, runtime_layout_fp8,
)
