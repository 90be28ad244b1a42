"""GB300-native decode attention of FastOCR (focal layers, top-tau image-token
selection, gather attention, Cross-Step Fixation Reuse) and R-SWA.

The compute path is libfastocr.so (CUDA, sm_103a) behind the C ABI of
include/fastocr.h; `_native` binds it with ctypes under the same names, and
`decoder.DecodeAttention` sequences the per-layer calls of a decode step.
Importing this package loads the library and fails if it is not built.
"""
from . import _native  # noqa: F401  (loads libfastocr.so or raises)
from ._native import (  # noqa: F401
    fastocr_abi_version, fastocr_create, fastocr_destroy, fastocr_device_status,
    fastocr_focal_attend, fastocr_full_attend, fastocr_profiler_reset, fastocr_profiler_select,
    fastocr_rswa_attend, fastocr_set_length_hint, fastocr_set_splits, fastocr_sparse_attend,
    make_kv)
from .decoder import (CapturedStep, DecodeAttention, ProfileSchedule, keep_capacity,  # noqa: F401
                      ring_block_table)
