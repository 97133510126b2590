"""Float64 CPU oracle for sparse MLA decode (test infrastructure only).

Imported by the tests, the smoke check and the bench's CPU baseline; never by
the library. See smla_oracle for the definitions and their sources.
"""
from .smla_oracle import *  # noqa: F401,F403
from .smla_oracle import (attend, bf16_bits_to_f64, block_scales, decode, dequant_rows,  # noqa: F401
                          e4m3_decode, e4m3_encode_rne_satfinite, f32, gather_dequant,
                          pack_bf16, pack_fp8_ds, pack_fp8_tensor, physical_slots, pow2_ceil_f32,
                          bf16_rne, f64_to_bf16_bits, rms_norm_bf16, rope_bf16, store_normed_rows, q_values)
