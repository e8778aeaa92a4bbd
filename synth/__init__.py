"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

Holds none of the method's arithmetic: only random draws, format conversion of
the drawn values to their storage types, and the workload table.
"""
from .inputs import (CONFIGS, DECODE_TOKENS, MOE_CONFIGS, FP8_SPREAD, Workload, bf16_bits_to_f32, f32_to_bf16_bits,
                     make_inputs, make_inputs_fp8, make_inputs_moe, make_inputs_mxfp4, make_inputs_nvfp4, workload)

__all__ = ["CONFIGS", "DECODE_TOKENS", "MOE_CONFIGS", "FP8_SPREAD", "Workload", "bf16_bits_to_f32", "f32_to_bf16_bits",
           "make_inputs", "make_inputs_fp8", "make_inputs_moe", "make_inputs_mxfp4", "make_inputs_nvfp4", "workload"]
