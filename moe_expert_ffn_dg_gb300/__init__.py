"""GB300-native (sm_103a) routed-MoE feed-forward block of a DiffusionGemma
layer: router + top-k, token->expert grouping, grouped tcgen05 GEMMs with
fused GEGLU and weighted combine, dense branch, norm sandwich and residual.

The compute runs in ``lib/libdgmoe.so`` (built by :func:`build`) behind the C
ABI of ``include/dg_moe.h``; this package is its Python binding.
"""

from .build import build, LIB  # noqa: F401
from . import binding  # noqa: F401
from .binding import DgError, load_library  # noqa: F401


def __getattr__(name):
    # the torch-level holder imports torch lazily
    if name in ("MoEBlock", "ScMlp", "params_to_device"):
        from . import block
        return getattr(block, name)
    raise AttributeError(name)
