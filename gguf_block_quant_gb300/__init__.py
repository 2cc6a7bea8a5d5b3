"""GB300-native GGUF block-quantized decode DMMV (Q8_0 / Q4_0).

The compute path is the C-ABI CUDA library built from ``csrc/`` for sm_103a
(``libzdmmv.so``); ``zdmmv`` is its thin Python binding. ``synth`` draws the
seeded synthetic inputs.
"""
