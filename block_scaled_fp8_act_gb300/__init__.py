"""GB300-native W8A8 block-FP8 linear layer (1x128 activation / 128x128 weight scales).

The compute lives in ``libfp8act.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/fp8act.h``). ``block_scaled_fp8_act_gb300.fp8act``
is the thin ctypes binding; importing this package does not load the library.
"""
