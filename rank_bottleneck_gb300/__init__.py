"""GB300-native forward/backward of one low-rank (CoLA-style) bottleneck decoder block.

The compute lives in ``libboostblk.so`` (CUDA for sm_103a, C ABI in
``include/boostblk.h``); ``rank_bottleneck_gb300.block`` is its Python binding and
``rank_bottleneck_gb300.synth`` draws seeded synthetic inputs.
"""
__all__ = ["block", "synth"]
