"""Float64 CPU oracle (test infrastructure only; see ``decode_ref``)."""
from .decode_ref import (attend, bf16_to_f64, decode_ref, decode_ref_inputs, dequant_int4,
                         dequant_int8, gather_kv, merge_splits, unpack_int4)

__all__ = ["attend", "bf16_to_f64", "decode_ref", "decode_ref_inputs", "dequant_int4",
           "dequant_int8", "gather_kv", "merge_splits", "unpack_int4"]
