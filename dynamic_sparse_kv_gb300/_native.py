"""ctypes binding of libfastocr.so: the C ABI of include/fastocr.h, same names.

Argument marshalling only -- every step of the decode-attention path runs in
the library's CUDA kernels. Tensors are PyTorch tensors on the GPU; their
data pointers are handed to the library as they are (no copies, no casts).
If the library is missing this module raises at import: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfastocr.so")

FASTOCR_OK = 0
FASTOCR_ERR_NULL = -1
FASTOCR_ERR_INVALID = -2
FASTOCR_ERR_UNSUPPORTED = -3
FASTOCR_ERR_CUDA = -4
FASTOCR_ERR_NO_DEVICE = -5
FASTOCR_ERR_ALIGN = -6
FASTOCR_DTYPE_F32 = 0
FASTOCR_DTYPE_BF16 = 1
DEV_BAD_PAGE, DEV_BAD_SEQLEN, DEV_BAD_IMG, DEV_BAD_SELECTION, DEV_INTERNAL = 1, 2, 4, 8, 16


class fastocr_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("max_img_tokens", ctypes.c_int32),
                ("num_layers", ctypes.c_int32)]


class fastocr_kv(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("seq_len", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32)]


class FastOCRError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_string(status)} (status {status})")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python dynamic_sparse_kv_gb300/build.py` "
            "(or __graft_entry__.build()) -- there is no CPU fallback")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, F64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_double
    sigs = {
        "fastocr_abi_version": ([], I32),
        "fastocr_status_string": ([I32], ctypes.c_char_p),
        "fastocr_create": ([ctypes.POINTER(fastocr_dims), ctypes.POINTER(P)], I32),
        "fastocr_destroy": ([P], I32),
        "fastocr_full_attend": ([P, P, ctypes.POINTER(fastocr_kv), P, P], I32),
        "fastocr_focal_attend": ([P, P, ctypes.POINTER(fastocr_kv), P, F64, P, P, I32, P, I32, P],
                                 I32),
        "fastocr_focal_scores": ([P, P, ctypes.POINTER(fastocr_kv), P, P, P, I32, P], I32),
        "fastocr_profile_attend": ([P, P, ctypes.POINTER(fastocr_kv), P, P, I32, P], I32),
        "fastocr_select": ([P, ctypes.POINTER(fastocr_kv), P, P, I32, F64, P, I32, P, P], I32),
        "fastocr_sparse_attend": ([P, P, ctypes.POINTER(fastocr_kv), P, P, I32, P, P, P], I32),
        "fastocr_sparse_attend_ex": ([P, P, ctypes.POINTER(fastocr_kv), P, P, I32, P, P,
                                      ctypes.c_uint32, P], I32),
        "fastocr_rswa_attend": ([P, P, ctypes.POINTER(fastocr_kv), I32, I32, P, P], I32),
        "fastocr_profiler_reset": ([P, P], I32),
        "fastocr_profiler_select": ([P, I32, ctypes.POINTER(I32), ctypes.POINTER(F64), P], I32),
        "fastocr_profiler_read": ([P, ctypes.POINTER(F64), P], I32),
        "fastocr_profiler_load": ([P, ctypes.POINTER(F64), P], I32),
        "fastocr_device_status": ([P, ctypes.POINTER(I32), P], I32),
        "fastocr_set_splits": ([P, I32, I32], I32),
        "fastocr_set_variant": ([P, I32, I32], I32),
        "fastocr_set_length_hint": ([P, I32], I32),
        "fastocr_read_probe": ([P, ctypes.c_int64, P, P], I32),
        "fastocr_copy": ([P, P, ctypes.c_int64, P], I32),
        "fastocr_focal_attend_noalloc": ([ctypes.POINTER(fastocr_dims), P,
                                          ctypes.POINTER(fastocr_kv), P, F64, P, P, I32, P, P, P],
                                         I32),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.fastocr_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != FASTOCR_OK:
        raise FastOCRError(fn, status)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def fastocr_abi_version() -> int:
    return lib.fastocr_abi_version()


def fastocr_create(batch, num_q_heads, num_kv_heads, head_dim, dtype, page_size,
                   max_pages_per_seq, max_img_tokens, num_layers) -> int:
    dims = fastocr_dims(batch, num_q_heads, num_kv_heads, head_dim, dtype, page_size,
                        max_pages_per_seq, max_img_tokens, num_layers)
    h = ctypes.c_void_p()
    _check("fastocr_create", lib.fastocr_create(ctypes.byref(dims), ctypes.byref(h)))
    return h.value


def fastocr_destroy(handle: int) -> None:
    _check("fastocr_destroy", lib.fastocr_destroy(handle))


def make_kv(k, v, block_table, seq_len) -> fastocr_kv:
    """One layer's cache descriptor; keeps no reference to the tensors."""
    return fastocr_kv(_ptr(k), _ptr(v), _ptr(block_table), _ptr(seq_len), int(k.shape[0]))


def fastocr_full_attend(handle, q, kv: fastocr_kv, out, stream=None) -> None:
    _check("fastocr_full_attend",
           lib.fastocr_full_attend(handle, _ptr(q), ctypes.byref(kv), _ptr(out), _stream(stream)))


def fastocr_focal_attend(handle, q, kv: fastocr_kv, img_range, tau, out, idx, idx_stride, k_out,
                         profile_layer=-1, stream=None) -> None:
    _check("fastocr_focal_attend",
           lib.fastocr_focal_attend(handle, _ptr(q), ctypes.byref(kv), _ptr(img_range),
                                    float(tau), _ptr(out), _ptr(idx), int(idx_stride),
                                    _ptr(k_out), int(profile_layer), _stream(stream)))


def fastocr_profile_attend(handle, q, kv: fastocr_kv, img_range, out, profile_layer,
                           stream=None) -> None:
    """Full attention that adds the layer's image mass to the profiler; no selection."""
    _check("fastocr_profile_attend",
           lib.fastocr_profile_attend(handle, _ptr(q), ctypes.byref(kv), _ptr(img_range),
                                      _ptr(out), int(profile_layer), _stream(stream)))


def fastocr_focal_scores(handle, q, kv: fastocr_kv, img_range, out, sigma, sigma_stride,
                         stream=None) -> None:
    _check("fastocr_focal_scores",
           lib.fastocr_focal_scores(handle, _ptr(q), ctypes.byref(kv), _ptr(img_range), _ptr(out),
                                    _ptr(sigma), int(sigma_stride), _stream(stream)))


def fastocr_select(handle, kv: fastocr_kv, img_range, sigma, sigma_stride, tau, idx, idx_stride,
                   k_out, stream=None) -> None:
    _check("fastocr_select",
           lib.fastocr_select(handle, ctypes.byref(kv), _ptr(img_range), _ptr(sigma),
                              int(sigma_stride), float(tau), _ptr(idx), int(idx_stride),
                              _ptr(k_out), _stream(stream)))


def fastocr_sparse_attend(handle, q, kv: fastocr_kv, img_range, idx, idx_stride, k, out,
                          stream=None) -> None:
    _check("fastocr_sparse_attend",
           lib.fastocr_sparse_attend(handle, _ptr(q), ctypes.byref(kv), _ptr(img_range),
                                     _ptr(idx), int(idx_stride), _ptr(k), _ptr(out),
                                     _stream(stream)))


SELECTION_FINAL = 1     # FASTOCR_SELECTION_FINAL
SELECTION_PENDING = 2   # FASTOCR_SELECTION_PENDING


def fastocr_sparse_attend_ex(handle, q, kv: fastocr_kv, img_range, idx, idx_stride, k, out,
                             flags: int, stream=None) -> None:
    """fastocr_sparse_attend with flags; SELECTION_FINAL: idx and k were written
    before the kernel preceding this call on the stream began."""
    _check("fastocr_sparse_attend_ex",
           lib.fastocr_sparse_attend_ex(handle, _ptr(q), ctypes.byref(kv), _ptr(img_range),
                                        _ptr(idx), int(idx_stride), _ptr(k), _ptr(out),
                                        int(flags), _stream(stream)))


def fastocr_rswa_attend(handle, q, kv: fastocr_kv, prefix_len, window, out, stream=None) -> None:
    _check("fastocr_rswa_attend",
           lib.fastocr_rswa_attend(handle, _ptr(q), ctypes.byref(kv), int(prefix_len),
                                   int(window), _ptr(out), _stream(stream)))


def fastocr_profiler_reset(handle, stream=None) -> None:
    _check("fastocr_profiler_reset", lib.fastocr_profiler_reset(handle, _stream(stream)))


def fastocr_profiler_select(handle, n_focal, num_layers, stream=None):
    """Returns (focal layer ids ascending, image mass of every layer)."""
    layers = (ctypes.c_int32 * n_focal)()
    ratio = (ctypes.c_double * num_layers)()
    _check("fastocr_profiler_select",
           lib.fastocr_profiler_select(handle, int(n_focal), layers, ratio, _stream(stream)))
    return tuple(int(x) for x in layers), [float(x) for x in ratio]


def fastocr_profiler_read(handle, num_layers, stream=None) -> list:
    """The accumulated image mass of every layer (synchronises the stream)."""
    mass = (ctypes.c_double * num_layers)()
    _check("fastocr_profiler_read", lib.fastocr_profiler_read(handle, mass, _stream(stream)))
    return [float(x) for x in mass]


def fastocr_profiler_load(handle, mass, stream=None) -> None:
    """Load the accumulated image mass of every layer (len(mass) = num_layers)."""
    arr = (ctypes.c_double * len(mass))(*[float(x) for x in mass])
    _check("fastocr_profiler_load", lib.fastocr_profiler_load(handle, arr, _stream(stream)))


def fastocr_device_status(handle, stream=None) -> int:
    s = ctypes.c_int32()
    _check("fastocr_device_status",
           lib.fastocr_device_status(handle, ctypes.byref(s), _stream(stream)))
    return int(s.value)


def fastocr_set_length_hint(handle, n_t) -> None:
    _check("fastocr_set_length_hint", lib.fastocr_set_length_hint(handle, int(n_t)))


def fastocr_set_splits(handle, mode, splits) -> None:
    _check("fastocr_set_splits", lib.fastocr_set_splits(handle, int(mode), int(splits)))


VARIANT_AUTO, VARIANT_GENERAL, VARIANT_DEEP = 0, 1, 2


def fastocr_set_variant(handle, mode, variant) -> None:
    _check("fastocr_set_variant", lib.fastocr_set_variant(handle, int(mode), int(variant)))


NOALLOC_MAX_UNITS_IMG = 65536   # FASTOCR_NOALLOC_MAX_UNITS_IMG


def fastocr_focal_attend_noalloc(dims: fastocr_dims, q, kv: fastocr_kv, img_range, tau, out, idx,
                                 idx_stride, k_out, status, stream=None) -> None:
    """Focal layer without a handle, for callers that may not allocate GPU
    memory where they run; its scratch is a fixed array inside the library."""
    _check("fastocr_focal_attend_noalloc",
           lib.fastocr_focal_attend_noalloc(ctypes.byref(dims), _ptr(q), ctypes.byref(kv),
                                            _ptr(img_range), float(tau), _ptr(out), _ptr(idx),
                                            int(idx_stride), _ptr(k_out), _ptr(status),
                                            _stream(stream)))


def fastocr_copy(dst, src, nbytes, stream=None) -> None:
    """Copy nbytes from src to dst with the SMs (device or page-locked host memory)."""
    _check("fastocr_copy", lib.fastocr_copy(_ptr(dst), _ptr(src), int(nbytes), _stream(stream)))


def fastocr_read_probe(src, nbytes, sink, stream=None) -> None:
    """Read nbytes of device memory at src once (read-only bandwidth probe)."""
    _check("fastocr_read_probe",
           lib.fastocr_read_probe(_ptr(src), int(nbytes), _ptr(sink), _stream(stream)))
