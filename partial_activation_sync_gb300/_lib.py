"""ctypes declarations of the C ABI in ``include/caat.h``.

Loading fails loudly when the CUDA library has not been built: there is no
CPU or PyTorch fallback behind these functions.
"""
import ctypes
import os

from . import build as _build

_c_i64 = ctypes.c_int64
_c_p = ctypes.c_void_p
_c_pp = ctypes.POINTER(ctypes.c_void_p)

EXPORTS = (
    "caat_select_channels",
    "caat_partial_channel_reduce",
    "caat_rowpar_linear_fwd",
    "caat_rowpar_linear_bwd_workspace",
    "caat_rowpar_linear_bwd",
    "caat_rowpar_linear_bwd_noalloc",
    "caat_rowpar_linear_fwd_compact",
    "caat_rowpar_linear_bwd_compact",
    "caat_rowpar_linear_compact_workspace",
    "caat_colpar_linear_fwd",
    "caat_colpar_linear_bwd_workspace",
    "caat_colpar_linear_bwd",
    "caat_status_string",
    "caat_get_device_status",
    "caat_last_kernel",
    "caat_launch_count",
    "caat_debug_set_wait",
    "caat_pcr_pack",
    "caat_pcr_unpack",
    "caat_rank_fold",
)

_lib = None


def load(path: str = None) -> ctypes.CDLL:
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise ImportError(
            "libcaat.so is not built (%s); run partial_activation_sync_gb300.build.build() "
            "(nvcc, sm_103a) first" % p)
    L = ctypes.CDLL(p)
    L.caat_select_channels.argtypes = [_c_i64, ctypes.c_double, ctypes.c_int, ctypes.c_uint64,
                                       _c_p, _c_p]
    L.caat_select_channels.restype = ctypes.c_int
    L.caat_partial_channel_reduce.argtypes = [ctypes.c_int, _c_i64, _c_i64, ctypes.c_int,
                                              _c_pp, _c_i64, _c_pp, _c_i64, _c_p, _c_i64, _c_p]
    L.caat_partial_channel_reduce.restype = ctypes.c_int
    L.caat_rowpar_linear_fwd.argtypes = [ctypes.c_int, _c_i64, _c_i64, _c_i64, ctypes.c_int,
                                         _c_p, _c_i64, _c_p, _c_i64, _c_i64,
                                         _c_pp, _c_i64, _c_p, _c_i64, _c_p]
    L.caat_rowpar_linear_fwd.restype = ctypes.c_int
    L.caat_rowpar_linear_bwd_workspace.argtypes = [ctypes.c_int, _c_i64, _c_i64, _c_i64, ctypes.c_int,
                                                   ctypes.c_int]
    L.caat_rowpar_linear_bwd_workspace.restype = ctypes.c_size_t
    L.caat_rowpar_linear_bwd.argtypes = [ctypes.c_int, _c_i64, _c_i64, _c_i64, ctypes.c_int,
                                         _c_p, _c_i64, _c_p, _c_i64, _c_i64,
                                         _c_pp, _c_i64, _c_p, _c_i64, _c_p, _c_i64, _c_i64,
                                         _c_p, _c_i64, ctypes.c_int, _c_p, ctypes.c_size_t, _c_p]
    L.caat_rowpar_linear_bwd.restype = ctypes.c_int
    L.caat_rowpar_linear_bwd_noalloc.argtypes = [ctypes.c_int, _c_i64, _c_i64, _c_i64, ctypes.c_int,
                                                 _c_p, _c_i64, _c_p, _c_i64, _c_i64,
                                                 _c_pp, _c_i64, _c_p, _c_i64, _c_p, _c_i64, _c_i64,
                                                 _c_p, _c_i64, ctypes.c_int, _c_p]
    L.caat_rowpar_linear_bwd_noalloc.restype = ctypes.c_int
    L.caat_rowpar_linear_fwd_compact.argtypes = [ctypes.c_int, _c_i64, _c_i64, _c_i64, ctypes.c_int,
                                                 _c_p, _c_i64, _c_p, _c_i64, _c_i64,
                                                 _c_p, _c_i64, _c_pp, _c_i64, _c_p, _c_i64,
                                                 _c_p, ctypes.c_size_t, _c_p]
    L.caat_rowpar_linear_fwd_compact.restype = ctypes.c_int
    L.caat_rowpar_linear_bwd_compact.argtypes = [ctypes.c_int, _c_i64, _c_i64, _c_i64, ctypes.c_int,
                                                 _c_p, _c_i64, _c_p, _c_i64, _c_i64,
                                                 _c_p, _c_i64, _c_pp, _c_i64,
                                                 _c_p, _c_i64, _c_p, _c_i64, _c_i64,
                                                 _c_p, _c_i64, _c_p, ctypes.c_size_t, _c_p]
    L.caat_rowpar_linear_bwd_compact.restype = ctypes.c_int
    L.caat_rowpar_linear_compact_workspace.argtypes = [ctypes.c_int, _c_i64, _c_i64, _c_i64, ctypes.c_int,
                                                       ctypes.c_int, ctypes.c_int]
    L.caat_rowpar_linear_compact_workspace.restype = ctypes.c_size_t
    L.caat_colpar_linear_fwd.argtypes = [ctypes.c_int, _c_i64, _c_i64, _c_i64, ctypes.c_int,
                                         _c_pp, _c_i64, _c_p, _c_i64, _c_i64, _c_p, _c_i64, _c_p]
    L.caat_colpar_linear_fwd.restype = ctypes.c_int
    L.caat_colpar_linear_bwd_workspace.argtypes = [ctypes.c_int, _c_i64, _c_i64, _c_i64, ctypes.c_int]
    L.caat_colpar_linear_bwd_workspace.restype = ctypes.c_size_t
    L.caat_colpar_linear_bwd.argtypes = [ctypes.c_int, _c_i64, _c_i64, _c_i64, ctypes.c_int,
                                         _c_pp, _c_i64, _c_p, _c_i64, _c_i64, _c_p, _c_i64,
                                         _c_pp, _c_i64, _c_p, _c_i64, _c_i64, _c_p, _c_i64,
                                         _c_p, ctypes.c_size_t, _c_p]
    L.caat_colpar_linear_bwd.restype = ctypes.c_int
    L.caat_status_string.argtypes = [ctypes.c_int]
    L.caat_status_string.restype = ctypes.c_char_p
    L.caat_get_device_status.argtypes = [_c_p]
    L.caat_get_device_status.restype = ctypes.c_int
    L.caat_last_kernel.argtypes = []
    L.caat_last_kernel.restype = ctypes.c_char_p
    L.caat_launch_count.argtypes = []
    L.caat_launch_count.restype = ctypes.c_uint64
    L.caat_debug_set_wait.argtypes = [ctypes.c_uint64, ctypes.c_int]
    L.caat_debug_set_wait.restype = ctypes.c_int
    L.caat_pcr_pack.argtypes = [_c_i64, _c_i64, ctypes.c_int, _c_p, _c_i64, _c_p, _c_i64, _c_p, _c_i64, _c_p]
    L.caat_pcr_pack.restype = ctypes.c_int
    L.caat_pcr_unpack.argtypes = [_c_i64, _c_i64, ctypes.c_int, _c_p, _c_i64, _c_p, _c_i64, _c_pp, ctypes.c_int,
                                  _c_i64, _c_p]
    L.caat_pcr_unpack.restype = ctypes.c_int
    L.caat_rank_fold.argtypes = [ctypes.c_int, _c_i64, _c_i64, ctypes.c_int, _c_p, _c_i64, _c_i64, _c_p, _c_i64,
                                 _c_p]
    L.caat_rank_fold.restype = ctypes.c_int
    if path is None:
        _lib = L
    return L


def ptr_array(ptrs):
    if not ptrs:
        return (ctypes.c_void_p * 1)()
    return (ctypes.c_void_p * len(ptrs))(*ptrs)
