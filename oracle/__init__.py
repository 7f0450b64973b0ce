"""CPU oracle for KIVI-style group-affine KV-cache quantization and decode
attention (plain C, single-threaded, in ``kivi_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the library's product
path never does.  The oracle shares no code with the CUDA library.

Sources (VeloxQuant-MLX pages): changelog v0.8.0 "New" (KIVI: per-channel
keys, per-token values, fp16 residual window, group size), changelog v0.42.0
"Added" (scalar_fused_decode_attend: codes plus a per-group (scale, zero) from
the group min/max; attention over rebuilt k_hat/v_hat), method overview
(AgeTieredKV entry: recency-gated residual window, shared min/max group
quantizer) and changelog v0.28.0 (chunk-flush residual; prefill and decode
give identical state).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(invariants, closed forms, hand-worked golden values, brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kivi_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkivi_oracle.so")
_lock = threading.Lock()
_lib = None

PLANES = ("Kc", "Ks", "Kz", "Vc", "Vs", "Vz", "Kr", "Vr",
          "sink_pos", "sink_k", "sink_v", "Kmask", "Vf", "tier")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-frounding-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_long, ctypes.c_double
        lib.orc_new.restype = P
        lib.orc_new.argtypes = [i32] * 8
        lib.orc_free.argtypes = [P]
        lib.orc_set_sinks.argtypes = [P, i32]
        lib.orc_set_kitty.argtypes = [P, i32]
        lib.orc_set_age.argtypes = [P, i32, i32, i32, i32, i32]
        lib.orc_quantize.argtypes = [P, P, P, i64, P]
        lib.orc_append.argtypes = [P, P, P, i64, P]
        lib.orc_attend.argtypes = [P, P, f64, P]
        lib.orc_attend_one.argtypes = [P, i32, i32, P, f64, P]
        lib.orc_attend_multi.argtypes = [P, P, i32, f64, P]
        lib.orc_attend_prefix.argtypes = [P, i32, i32, P, i32, f64, P]
        lib.orc_lengths.argtypes = [P, P, P, P]
        lib.orc_dims.argtypes = [P, P, P]
        lib.orc_plane_bytes.restype = ctypes.c_size_t
        lib.orc_plane_bytes.argtypes = [P, i32]
        lib.orc_get_plane.argtypes = [P, i32, P]
        lib.orc_quant_group_f32.argtypes = [P, i32, i32, P, P, P, P]
        lib.orc_pack_codes.argtypes = [P, i32, i32, P]
        lib.orc_unpack_codes.argtypes = [P, i32, i32, P]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _f16bits(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a))
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype == np.uint16:
        return a
    raise TypeError(f"expected float16 or uint16 bit patterns, got {a.dtype}")


# --------------------------------------------------------------------------
# Primitives
# --------------------------------------------------------------------------

def quant_group(x, bits: int):
    """Quantize one group.  x: fp32 values (exact copies of fp16 inputs).
    Returns (codes uint8[n], scale32 float, scale16 bits, zero16 bits)."""
    lib = _load()
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    codes = np.zeros(x.size, np.uint8)
    s32 = np.zeros(1, np.float32)
    s16 = np.zeros(1, np.uint16)
    z16 = np.zeros(1, np.uint16)
    lib.orc_quant_group_f32(_ptr(x), x.size, bits, _ptr(codes), _ptr(s32),
                            _ptr(s16), _ptr(z16))
    return codes, float(s32[0]), int(s16[0]), int(z16[0])


def pack_codes(codes, bits: int) -> np.ndarray:
    lib = _load()
    codes = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.zeros((codes.size * bits + 7) // 8, np.uint8)
    lib.orc_pack_codes(_ptr(codes), codes.size, bits, _ptr(out))
    return out


def unpack_codes(packed, n: int, bits: int) -> np.ndarray:
    lib = _load()
    packed = np.ascontiguousarray(np.asarray(packed, dtype=np.uint8))
    out = np.zeros(n, np.uint8)
    lib.orc_unpack_codes(_ptr(packed), n, bits, _ptr(out))
    return out


# --------------------------------------------------------------------------
# Cache
# --------------------------------------------------------------------------

class OracleCache:
    """The oracle's KIVI cache for B sequences x H_kv heads.

    Canonical planes (row-major):
      Kc, Vc  uint8  [B][H_kv][Tcap][D*bits/8]   (LSB-first packing)
      sink_pos int32 [B][H_kv][n_sink]           (KIVI-Sink: ascending, -1 unused)
      sink_k, sink_v fp16 [B][H_kv][n_sink][D]
      Ks, Kz  fp16   [B][H_kv][Tcap/g][D]        (per channel, per key group)
      Vs, Vz  fp16   [B][H_kv][Tcap][D/g]        (per token, per channel group)
      Kr, Vr  fp16   [B][H_kv][R+g][D]           (slot i holds token Tq+i)
    """

    def __init__(self, B, H_q, H_kv, D, bits, group, residual, max_seq,
                 n_sink=0, kitty_hi=None, age=None):
        self.B, self.H_q, self.H_kv, self.D = B, H_q, H_kv, D
        self.bits, self.group, self.residual, self.max_seq = (
            bits, group, residual, max_seq)
        self.n_sink = n_sink
        self._lib = _load()
        self._c = self._lib.orc_new(B, H_q, H_kv, D, bits, group, residual,
                                    max_seq)
        if not self._c:
            raise ValueError("oracle: unsupported cache parameters")
        if self._lib.orc_set_sinks(self._c, n_sink) != 0:
            raise ValueError("oracle: bad sink count")
        self.kitty_hi = kitty_hi
        if kitty_hi is not None and self._lib.orc_set_kitty(self._c, kitty_hi) != 0:
            raise ValueError("oracle: bad Kitty parameters")
        # AgeTieredKV: (boundary 1, boundary 2, bits of the three tiers)
        self.age = age
        if age is not None and self._lib.orc_set_age(self._c, *age) != 0:
            raise ValueError("oracle: bad AgeTieredKV parameters")
        tcap = np.zeros(1, np.int32)
        rcap = np.zeros(1, np.int32)
        self._lib.orc_dims(self._c, _ptr(tcap), _ptr(rcap))
        self.Tcap, self.Rcap = int(tcap[0]), int(rcap[0])

    def __del__(self):
        c = getattr(self, "_c", None)
        if c:
            self._lib.orc_free(c)
            self._c = None

    def quantize(self, K, V, seq_lens):
        K, V = _f16bits(K), _f16bits(V)
        assert K.shape == V.shape and K.ndim == 4
        assert K.shape[:2] == (self.B, self.H_kv) and K.shape[3] == self.D
        lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
        rc = self._lib.orc_quantize(self._c, _ptr(K), _ptr(V), K.shape[2],
                                    _ptr(lens))
        if rc != 0:
            raise ValueError("oracle: bad sequence length")

    def append(self, K_new, V_new, n_new):
        K, V = _f16bits(K_new), _f16bits(V_new)
        assert K.shape == V.shape and K.ndim == 4
        n = np.ascontiguousarray(np.asarray(n_new, dtype=np.int32))
        rc = self._lib.orc_append(self._c, _ptr(K), _ptr(V), K.shape[2],
                                  _ptr(n))
        if rc != 0:
            raise ValueError("oracle: bad append length")

    def attend(self, q, scale=None) -> np.ndarray:
        q = _f16bits(q)
        assert q.shape == (self.B, self.H_q, self.D)
        out = np.zeros((self.B, self.H_q, self.D), np.float32)
        sc = (1.0 / np.sqrt(self.D)) if scale is None else float(scale)
        self._lib.orc_attend(self._c, _ptr(q), sc, _ptr(out))
        return out

    def attend_multi(self, q, scale=None) -> np.ndarray:
        """q: fp16 [B][H_q][S_q][D], the queries of each sequence's newest
        S_q tokens (query i at position S - S_q + i, causal).  Returns fp32
        [B][H_q][S_q][D]."""
        q = _f16bits(q)
        assert q.ndim == 4 and q.shape[:2] == (self.B, self.H_q)
        assert q.shape[3] == self.D
        out = np.zeros(q.shape, np.float32)
        sc = (1.0 / np.sqrt(self.D)) if scale is None else float(scale)
        rc = self._lib.orc_attend_multi(self._c, _ptr(q), q.shape[2], sc,
                                        _ptr(out))
        if rc != 0:
            raise ValueError("oracle: a sequence is shorter than S_q")
        return out

    def attend_prefix(self, b: int, hq: int, q_row, last: int,
                      scale=None) -> np.ndarray:
        """One query of head hq attending tokens 0 ... last of sequence b
        (the causal prefix of the query at position last)."""
        q_row = _f16bits(q_row).reshape(-1)
        assert q_row.size == self.D
        out = np.zeros(self.D, np.float64)
        sc = (1.0 / np.sqrt(self.D)) if scale is None else float(scale)
        if self._lib.orc_attend_prefix(self._c, b, hq, _ptr(q_row), last, sc,
                                       _ptr(out)) != 0:
            raise ValueError("oracle: position outside the sequence")
        return out

    def attend_one(self, b: int, hq: int, q_row, scale=None) -> np.ndarray:
        q_row = _f16bits(q_row).reshape(-1)
        assert q_row.size == self.D
        out = np.zeros(self.D, np.float64)
        sc = (1.0 / np.sqrt(self.D)) if scale is None else float(scale)
        self._lib.orc_attend_one(self._c, b, hq, _ptr(q_row), sc, _ptr(out))
        return out

    def lengths(self):
        S = np.zeros(self.B, np.int32)
        Tq = np.zeros(self.B, np.int32)
        nres = np.zeros(self.B, np.int32)
        self._lib.orc_lengths(self._c, _ptr(S), _ptr(Tq), _ptr(nres))
        return S, Tq, nres

    def plane(self, name: str) -> np.ndarray:
        which = PLANES.index(name)
        nbytes = self._lib.orc_plane_bytes(self._c, which)
        raw = np.zeros(nbytes, np.uint8)
        self._lib.orc_get_plane(self._c, which, _ptr(raw))
        B, H, D, g = self.B, self.H_kv, self.D, self.group
        row = D * self.bits // 8
        if name == "Kc" and self.kitty_hi is not None:
            krow = (self.kitty_hi * 4 + (D - self.kitty_hi) * 2) // 8
            return raw.reshape(B, H, self.Tcap, krow)
        if name == "Kmask":
            return raw.view(np.uint32).reshape(B, H, self.Tcap // g, D // 32)
        if name == "Vf":
            return raw.view(np.float16).reshape(B, H, self.Tcap, D)
        if name == "tier":
            return raw.view(np.int8).reshape(B, H, self.Tcap // g)
        if name in ("Kc", "Vc"):
            return raw.reshape(B, H, self.Tcap, row)
        if name in ("Ks", "Kz"):
            return raw.view(np.float16).reshape(B, H, self.Tcap // g, D)
        if name in ("Vs", "Vz"):
            return raw.view(np.float16).reshape(B, H, self.Tcap, D // g)
        if name == "sink_pos":
            return raw.view(np.int32).reshape(B, H, self.n_sink)
        if name in ("sink_k", "sink_v"):
            return raw.view(np.float16).reshape(B, H, self.n_sink, D)
        return raw.view(np.float16).reshape(B, H, self.Rcap, D)
