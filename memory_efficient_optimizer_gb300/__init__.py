"""GB300-native Adafactor step (factored second moment) as a C-ABI CUDA library,
with the multi-tensor LAMB and CAME steps beside it.

The CUDA kernels and the C entry points live in ``csrc/`` (declared in
``include/adafactor.h``, ``include/lamb.h`` and ``include/came.h``); ``binding`` is the ctypes marshalling layer with the
same names as the C entry points; ``optim`` holds the list-of-tensors step and
a ``torch.optim.Optimizer`` wrapper, ``lamb`` and ``came`` the same for LAMB and CAME.  There is no CPU fallback: without the
built library every entry point raises.
"""
from .binding import AdafactorError, library_path  # noqa: F401
from .came import Came, CameStep, came_step, init_came_state, make_came_hparams  # noqa: F401
from .lamb import Lamb, LambStep, init_lamb_state, lamb_step, make_lamb_hparams  # noqa: F401
from .optim import (Adafactor, AdafactorShardStep, AdafactorStep, adafactor_step,  # noqa: F401
                    init_state, make_hparams)

__all__ = ["Adafactor", "AdafactorStep", "AdafactorShardStep", "AdafactorError", "adafactor_step", "init_state",
           "make_hparams", "library_path", "Lamb", "LambStep", "lamb_step", "init_lamb_state",
           "make_lamb_hparams", "Came", "CameStep", "came_step", "init_came_state", "make_came_hparams"]
