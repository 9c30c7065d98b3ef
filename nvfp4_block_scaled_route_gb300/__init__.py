"""GB300-native NVFP4 MoE expert FFN (sm_103a).

The compute path is the C-ABI library ``libnvfp4moe.so`` built from ``csrc/``
(hand-written CUDA for sm_103a).  ``binding`` marshals arguments to it;
``synthetic`` draws seeded inputs.  Importing this package does not load the
library; ``binding.lib()`` does, and raises if it has not been built.
"""
