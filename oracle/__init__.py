"""Float64 CPU oracle for paged decode attention (GQA/MQA/MHA, MLA, split combine).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; never by the product path. It
shares no code with the CUDA library.
"""
from .decode import (FP8_E4M3, attend, attend_interval, combine_splits, decode_e4m3,  # noqa: F401
                     dequantize, gather_tokens, kv_head_of, mla_decode, num_pages, paged_decode,
                     token_locations, widen, causal_prefix, paged_decode_mtp, mla_decode_mtp,
                     encode_e4m3, quantize_e4m3, append_tokens)
