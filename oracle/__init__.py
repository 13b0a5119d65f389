"""Float64 CPU oracle for paged decode attention (GQA/MQA/MHA, MLA, split combine).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; never by the product path. It
shares no code with the CUDA library.
"""
from .decode import (attend, attend_interval, combine_splits, gather_tokens, kv_head_of,  # noqa: F401
                     mla_decode, num_pages, paged_decode, token_locations, widen)
