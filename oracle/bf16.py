"""Exact decoding of bfloat16 bit patterns to float64 (oracle, test-only).

A bfloat16 value is the upper 16 bits of an IEEE-754 binary32 value, so
placing the 16 stored bits in the high half of a 32-bit word and reading that
word as binary32 reproduces the value exactly; binary32 -> binary64 is exact
as well.  The pages fix only the storage cost of such a value ("bytes per
element" p = 2 for FP16/BF16: "LLM serving (vLLM, quantized inference):
Visual walkthrough", Step 1).
"""
import numpy as np


def bf16_bits_to_f64(bits):
    """Return float64 values of an array of raw bf16 bit patterns (uint16)."""
    b = np.asarray(bits)
    if b.dtype != np.uint16:
        raise TypeError("bf16 bit patterns must be uint16")
    word = b.astype(np.uint32) << np.uint32(16)
    return word.view(np.float32).astype(np.float64)
