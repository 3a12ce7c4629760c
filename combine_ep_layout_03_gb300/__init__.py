"""GB300-native MoE expert-parallel token layout, dispatch and combine.

The compute path is the C-ABI library ``libeplayout.so`` (hand-written CUDA
kernels for sm_103a, declared in ``include/ep_layout.h``).  ``ep`` is its thin
Python binding; importing it loads the library and raises if it is missing.
``synth`` draws the seeded synthetic inputs.
"""
__all__ = ["ep", "synth"]
