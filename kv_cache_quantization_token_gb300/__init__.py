"""KVarN hot path on GB300 (sm_103a): 4-bit-key / 2-bit-value KV-cache tile
compression and attention over the compressed cache.

The compute runs in the CUDA library ``libkvarn.so`` (sources in ``csrc/``);
``kvarn`` is its thin ctypes binding. ``synth`` draws the seeded inputs.
"""
