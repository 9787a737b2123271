"""GB300-native Adafactor step (factored second moment) as a C-ABI CUDA library.

The CUDA kernels and the C entry points live in ``csrc/``; ``binding`` is the
ctypes marshalling layer with the same names as the C entry points; ``optim``
holds the list-of-tensors step and a ``torch.optim.Optimizer`` wrapper.
"""
