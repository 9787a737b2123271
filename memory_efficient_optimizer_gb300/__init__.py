"""GB300-native Adafactor step (factored second moment) as a C-ABI CUDA library.

The CUDA kernels and the C entry points live in ``csrc/`` (declared in
``include/adafactor.h``); ``binding`` is the ctypes marshalling layer with the
same names as the C entry points; ``optim`` holds the list-of-tensors step and
a ``torch.optim.Optimizer`` wrapper.  There is no CPU fallback: without the
built library every entry point raises.
"""
from .binding import AdafactorError, library_path  # noqa: F401
from .optim import (Adafactor, AdafactorShardStep, AdafactorStep, adafactor_step,  # noqa: F401
                    init_state, make_hparams)

__all__ = ["Adafactor", "AdafactorStep", "AdafactorShardStep", "AdafactorError", "adafactor_step", "init_state",
           "make_hparams", "library_path"]
