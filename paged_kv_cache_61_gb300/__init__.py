"""Paged decode attention for GB300 (sm_103a): GQA/MQA/MHA split-KV and absorbed MLA.

The compute path is the C-ABI shared library ``libpda.so`` built from ``csrc/``;
``paged_kv_cache_61_gb300.pda`` is its thin ctypes binding. ``synth`` draws the
seeded synthetic inputs and ``traffic`` holds the byte/FLOP accounting used by
the benchmark. Importing this package does not load the library; the first call
through ``pda`` does, and raises if it has not been built.
"""
