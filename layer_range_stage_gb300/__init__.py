"""GB300-native forward of one layer-range pipeline stage.

The compute path is the CUDA library ``_lib/libstage.so`` (C ABI in include/stage.h);
``binding`` marshals arguments to it.  Building: ``layer_range_stage_gb300.build.build()``.
"""
from .binding import *  # noqa: F401,F403
from .binding import StageError, lib, make_cfg  # noqa: F401
