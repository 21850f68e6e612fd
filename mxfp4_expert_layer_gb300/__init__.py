"""GB300-native MXFP4 mixture-of-experts layer (gpt-oss-style MoE block).

The compute path is the CUDA library ``libmoe_mxfp4.so`` (C ABI in
``include/moe_mxfp4.h``); this package only builds it and binds it.
"""

from . import _lib  # noqa: F401
from .build import build, LIB_PATH  # noqa: F401


def __getattr__(name):
    # torch-facing helpers are imported lazily so the C binding works without torch
    if name in ("MoELayer", "MoELayerBF16", "prepare_weights", "prepare_weights_bf16", "workspace", "route",
                "build_tile_table", "tile_rows", "max_tiles"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
