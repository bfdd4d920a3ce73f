"""W8A8 block-FP8 linear layers on GB300 (sm_103a).

The compute path is the C-ABI library ``libfp8bq.so`` (hand-written CUDA);
``block_scaled_fp8_group_gb300.fp8bq`` is its thin Python binding.  This file
imports nothing heavy, so ``synth`` can be used without the library.
"""
