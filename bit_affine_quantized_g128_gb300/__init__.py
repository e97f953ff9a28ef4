"""1-bit affine group-quantized (g128) linear layer for GB300 (sm_103a).

The compute lives in the C-ABI library ``libq1.so`` (hand-written CUDA);
:mod:`.q1` is its thin Python binding.  The library is loaded on first use,
so that the seeded input generators in :mod:`.synth` import without it.
"""
