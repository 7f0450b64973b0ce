"""Thin ctypes binding of the C ABI in include/vq_kivi.h.

Argument marshalling only: every step of the path runs in the CUDA library.
The library must have been built (``bit_kv_cache_05_gb300.build``); loading
fails loudly otherwise -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

VQ_OK = 0
VQ_ERR_ARG = -1
VQ_ERR_UNSUPPORTED = -2
VQ_ERR_CAPACITY = -3
VQ_ERR_OOM = -4
VQ_ERR_CUDA = -5
_NAMES = {VQ_ERR_ARG: "VQ_ERR_ARG", VQ_ERR_UNSUPPORTED: "VQ_ERR_UNSUPPORTED",
          VQ_ERR_CAPACITY: "VQ_ERR_CAPACITY", VQ_ERR_OOM: "VQ_ERR_OOM",
          VQ_ERR_CUDA: "VQ_ERR_CUDA"}

# every symbol include/vq_kivi.h declares
EXPORTS = ("vq_kivi_quantize", "vq_kivi_quantize_ex", "vq_kivi_append",
           "vq_kivi_decode_attend", "vq_kivi_step_host",
           "vq_kivi_free", "vq_kivi_attend_multi", "vq_kivi_last_error", "vq_kivi_lengths",
           "vq_kivi_get_params", "vq_kivi_plane_bytes", "vq_kivi_export",
           "vq_kivi_dequantize",
           "vq_kivi_cache_bytes", "vq_kivi_set_split_tokens",
           "vq_kivi_launch_count", "vq_kivi_decode_attend_static",
           "vq_kivi_device_status", "vq_kivi_decode_kernel",
           "vq_kivi_debug_fail_chunk")


class VqError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_NAMES.get(code, code)}: {msg}")
        self.code = code


class Params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("B", "H_q", "H_kv", "D", "bits", "group", "residual",
                 "max_seq")]


class Planes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("Kc", "Ks", "Kz", "Vc", "Vs", "Vz", "Kr", "Vr")]


class Options(ctypes.Structure):
    _fields_ = [("n_sink", ctypes.c_int32), ("kitty", ctypes.c_int32),
                ("kitty_hi", ctypes.c_int32), ("age_recent", ctypes.c_int32),
                ("age_mid", ctypes.c_int32), ("age_bits_recent", ctypes.c_int32),
                ("age_bits_mid", ctypes.c_int32), ("age_bits_old", ctypes.c_int32)]


class Bytes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in
                ("code_bytes", "meta_bytes", "residual_bytes", "fp16_bytes",
                 "sink_bytes", "value_fp16_bytes")]


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"CUDA library not built: {path} is missing (run "
                    "python -m bit_kv_cache_05_gb300.build)")
            _build.build()
        L = ctypes.CDLL(path)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.vq_kivi_quantize.argtypes = [ctypes.POINTER(Params), P, P, i64, P, P,
                                       ctypes.POINTER(P)]
        L.vq_kivi_quantize_ex.argtypes = [ctypes.POINTER(Params),
                                          ctypes.POINTER(Options), P, P, i64,
                                          P, P, ctypes.POINTER(P)]
        L.vq_kivi_append.argtypes = [P, P, P, i64, P, P]
        L.vq_kivi_decode_attend.argtypes = [P, P, P, ctypes.c_float, P]
        L.vq_kivi_step_host.argtypes = [P, P, P, P, P, ctypes.c_float, P]
        L.vq_kivi_attend_multi.argtypes = [P, P, i32, P, ctypes.c_float, P]
        L.vq_kivi_free.argtypes = [P]
        L.vq_kivi_last_error.restype = ctypes.c_char_p
        L.vq_kivi_lengths.argtypes = [P, P, P, P]
        L.vq_kivi_get_params.argtypes = [P, ctypes.POINTER(Params)]
        L.vq_kivi_plane_bytes.restype = ctypes.c_size_t
        L.vq_kivi_plane_bytes.argtypes = [P, ctypes.c_int]
        L.vq_kivi_export.argtypes = [P, ctypes.c_int, P, ctypes.c_size_t, P]
        L.vq_kivi_dequantize.argtypes = [P, P, P, i64, P]
        L.vq_kivi_cache_bytes.argtypes = [P, ctypes.POINTER(Bytes)]
        L.vq_kivi_set_split_tokens.argtypes = [P, i32]
        L.vq_kivi_device_status.argtypes = [P]
        L.vq_kivi_decode_kernel.argtypes = [P]
        L.vq_kivi_debug_fail_chunk.argtypes = [P, i32]
        L.vq_kivi_launch_count.restype = ctypes.c_uint64
        L.vq_kivi_decode_attend_static.argtypes = [
            ctypes.POINTER(Params), ctypes.POINTER(Planes), P, P, P,
            ctypes.c_float, P]
        for name in EXPORTS:
            getattr(L, name).restype = getattr(L, name).restype or ctypes.c_int
        L.vq_kivi_plane_bytes.restype = ctypes.c_size_t
        L.vq_kivi_launch_count.restype = ctypes.c_uint64
        L.vq_kivi_last_error.restype = ctypes.c_char_p
        _lib = L
        return L


def check(rc: int):
    if rc != VQ_OK:
        msg = load().vq_kivi_last_error().decode(errors="replace")
        raise VqError(rc, msg)


def launch_count() -> int:
    return int(load().vq_kivi_launch_count())
