"""GB300-native decode-step token selection over fp32 logits rows.

The compute path is a C-ABI shared library of hand-written CUDA kernels for
sm_103a (``csrc/``, declared in ``include/sel.h``); ``binding`` marshals
torch CUDA tensors into its entry points. ``synth`` holds the seeded input
generators shared by the tests and the benchmark.
"""
