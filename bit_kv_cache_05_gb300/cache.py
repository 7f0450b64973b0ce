"""Python handle over the C ABI (include/vq_kivi.h): passes torch tensor
pointers, sizes and the current CUDA stream; holds no arithmetic.

Method: VeloxQuant-MLX changelog v0.8.0 "New" (KIVI cache with an fp16
residual window) and v0.42.0 "Added" (fused decode-attend over the
group-affine cache).
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _lib

PLANES = ("Kc", "Ks", "Kz", "Vc", "Vs", "Vz", "Kr", "Vr",
          "sink_pos", "sink_k", "sink_v", "Kmask", "Vf", "tier")


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream: Optional[torch.cuda.Stream],
                   device: Optional[int] = None) -> ctypes.c_void_p:
    """The stream to launch on: `stream`, else torch's current stream of
    `device` (the current device when None).  torch's raw lookup skips the
    Stream object that torch.cuda.current_stream() builds (~3 us a call)."""
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    if _raw_stream is not None:
        dev = torch.cuda.current_device() if device is None else device
        return ctypes.c_void_p(_raw_stream(dev))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _host_ptr(t: torch.Tensor, dtype: torch.dtype, name: str) -> ctypes.c_void_p:
    if t.is_cuda or not t.is_pinned():
        raise ValueError(f"{name} must be a pinned host tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dev_ptr(t: torch.Tensor, dtype: torch.dtype, name: str) -> ctypes.c_void_p:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _i32_array(xs: Sequence[int]):
    arr = (ctypes.c_int32 * len(xs))(*[int(x) for x in xs])
    return arr


class KiviCache:
    """A KIVI cache on the current CUDA device.

    K, V: fp16 CUDA tensors [B][H_kv][S_stride][D]; seq_lens: B ints.
    """

    def __init__(self, K: torch.Tensor, V: torch.Tensor, seq_lens, *, H_q: int,
                 bits: int, group: int, residual: int,
                 max_seq: Optional[int] = None, n_sink: int = 0,
                 kitty_hi: Optional[int] = None, age=None,
                 stream: Optional[torch.cuda.Stream] = None):
        L = _lib.load()
        if K.shape != V.shape or K.dim() != 4:
            raise ValueError("K and V must both be [B][H_kv][S][D]")
        B, H_kv, S_stride, D = K.shape
        lens = [int(x) for x in seq_lens]
        if len(lens) != B:
            raise ValueError("seq_lens must have B entries")
        self.params = _lib.Params(B, H_q, H_kv, D, bits, group, residual,
                                  max(lens + [0]) if max_seq is None else max_seq)
        self.B, self.H_q, self.H_kv, self.D = B, H_q, H_kv, D
        self.bits, self.group, self.residual = bits, group, residual
        self.max_seq = self.params.max_seq
        self._h = ctypes.c_void_p()
        kp = _dev_ptr(K, torch.float16, "K")
        vp = _dev_ptr(V, torch.float16, "V")
        self.n_sink = int(n_sink)
        self.kitty_hi = kitty_hi
        # age: (recent boundary, mid boundary, bits recent, mid, old)
        self.age = tuple(age) if age is not None else None
        opts = _lib.Options(self.n_sink, 0 if kitty_hi is None else 1,
                            0 if kitty_hi is None else int(kitty_hi),
                            *(self.age if self.age else (0, 0, 0, 0, 0)))
        _lib.check(L.vq_kivi_quantize_ex(ctypes.byref(self.params),
                                         ctypes.byref(opts), kp, vp,
                                         S_stride, _i32_array(lens),
                                         _stream_handle(stream),
                                         ctypes.byref(self._h)))
        self.device = K.device

    # -- steps ---------------------------------------------------------------

    def append(self, K_new: torch.Tensor, V_new: torch.Tensor, n_new,
               stream: Optional[torch.cuda.Stream] = None):
        n = [int(x) for x in n_new]
        if len(n) != self.B:
            raise ValueError("n_new must have B entries")
        if K_new.shape != V_new.shape or K_new.dim() != 4:
            raise ValueError("K_new and V_new must both be [B][H_kv][N][D]")
        _lib.check(_lib.load().vq_kivi_append(
            self._h, _dev_ptr(K_new, torch.float16, "K_new"),
            _dev_ptr(V_new, torch.float16, "V_new"), K_new.shape[2],
            _i32_array(n), _stream_handle(stream, self.device.index)))

    def decode_attend(self, q: torch.Tensor, out: Optional[torch.Tensor] = None,
                      scale: float = 0.0,
                      stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        if tuple(q.shape) != (self.B, self.H_q, self.D):
            raise ValueError(f"q must be [{self.B}][{self.H_q}][{self.D}]")
        if out is None:
            out = torch.empty((self.B, self.H_q, self.D), dtype=torch.float32,
                              device=q.device)
        _lib.check(_lib.load().vq_kivi_decode_attend(
            self._h, _dev_ptr(q, torch.float16, "q"),
            _dev_ptr(out, torch.float32, "out"), float(scale),
            _stream_handle(stream, self.device.index)))
        return out

    def step_host(self, K_new: torch.Tensor, V_new: torch.Tensor, q: torch.Tensor,
                  out: torch.Tensor, scale: float = 0.0,
                  stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """One serving step from pinned host memory (vq_kivi_step_host):
        append one token per sequence (K_new, V_new fp16 [B][H_kv][D]) and
        decode q (fp16 [B][H_q][D]) into out (fp32 [B][H_q][D]), all pinned
        host tensors.  Asynchronous: out holds the result once the stream
        has reached the end of the step."""
        if tuple(K_new.shape) != (self.B, self.H_kv, self.D) or K_new.shape != V_new.shape:
            raise ValueError(f"K_new and V_new must be [{self.B}][{self.H_kv}][{self.D}]")
        if tuple(q.shape) != (self.B, self.H_q, self.D) or q.shape != out.shape:
            raise ValueError(f"q and out must be [{self.B}][{self.H_q}][{self.D}]")
        _lib.check(_lib.load().vq_kivi_step_host(
            self._h, _host_ptr(K_new, torch.float16, "K_new"),
            _host_ptr(V_new, torch.float16, "V_new"),
            _host_ptr(q, torch.float16, "q"), _host_ptr(out, torch.float32, "out"),
            float(scale), _stream_handle(stream, self.device.index)))
        return out

    def attend_multi(self, q: torch.Tensor, out: Optional[torch.Tensor] = None,
                     scale: float = 0.0,
                     stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """Causal attention of each sequence's newest S_q tokens (already
        appended): q fp16 [B][H_q][S_q][D] -> fp32 [B][H_q][S_q][D]."""
        if q.dim() != 4 or (q.shape[0], q.shape[1], q.shape[3]) != (
                self.B, self.H_q, self.D):
            raise ValueError(f"q must be [{self.B}][{self.H_q}][S_q][{self.D}]")
        if out is None:
            out = torch.empty(tuple(q.shape), dtype=torch.float32, device=q.device)
        _lib.check(_lib.load().vq_kivi_attend_multi(
            self._h, _dev_ptr(q, torch.float16, "q"), int(q.shape[2]),
            _dev_ptr(out, torch.float32, "out"), float(scale),
            _stream_handle(stream)))
        return out

    # -- inspection ------------------------------------------------------------

    def lengths(self):
        S = (ctypes.c_int32 * self.B)()
        Tq = (ctypes.c_int32 * self.B)()
        nres = (ctypes.c_int32 * self.B)()
        _lib.check(_lib.load().vq_kivi_lengths(self._h, S, Tq, nres))
        return list(S), list(Tq), list(nres)

    def plane_bytes(self, name: str) -> int:
        return int(_lib.load().vq_kivi_plane_bytes(self._h, PLANES.index(name)))

    def export(self, name: str, stream: Optional[torch.cuda.Stream] = None):
        """Canonical plane as a CUDA tensor (layouts in include/vq_kivi.h)."""
        which = PLANES.index(name)
        nbytes = self.plane_bytes(name)
        raw = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        _lib.check(_lib.load().vq_kivi_export(
            self._h, which, ctypes.c_void_p(raw.data_ptr()), nbytes,
            _stream_handle(stream)))
        B, H, D, g = self.B, self.H_kv, self.D, self.group
        row = D * self.bits // 8
        if name == "Kc" and self.kitty_hi is not None:
            return raw.view(B, H, -1, (D + self.kitty_hi) // 4)
        if name == "Kmask":
            return raw.view(torch.int32).view(B, H, -1, D // 32)
        if name == "Vf":
            return raw.view(torch.float16).view(B, H, -1, D)
        if name == "tier":
            return raw.view(torch.int8).view(B, H, -1)
        if name == "sink_pos":
            return raw.view(torch.int32).view(B, H, self.n_sink)
        if name in ("sink_k", "sink_v"):
            return raw.view(torch.float16).view(B, H, self.n_sink, D)
        if name in ("Kc", "Vc"):
            return raw.view(B, H, -1, row)
        raw = raw.view(torch.float16)
        if name in ("Ks", "Kz"):
            return raw.view(B, H, -1, D)
        if name in ("Vs", "Vz"):
            return raw.view(B, H, -1, D // g)
        return raw.view(B, H, -1, D)

    def dequantize(self, out=None, stream: Optional[torch.cuda.Stream] = None):
        """fp16 K_hat, V_hat [B][H_kv][S_max][D] rebuilt from the cache (rows
        past a sequence's length are left as allocated)."""
        S, _, _ = self.lengths()
        smax = max(max(S), 1)
        if out is None:
            shape = (self.B, self.H_kv, smax, self.D)
            out = (torch.empty(shape, dtype=torch.float16, device=self.device),
                   torch.empty(shape, dtype=torch.float16, device=self.device))
        Kh, Vh = out
        _lib.check(_lib.load().vq_kivi_dequantize(
            self._h, _dev_ptr(Kh, torch.float16, "K_hat"),
            _dev_ptr(Vh, torch.float16, "V_hat"), Kh.shape[2],
            _stream_handle(stream)))
        return Kh, Vh

    def cache_bytes(self) -> dict:
        b = _lib.Bytes()
        _lib.check(_lib.load().vq_kivi_cache_bytes(self._h, ctypes.byref(b)))
        return {n: int(getattr(b, n)) for n, _ in _lib.Bytes._fields_}

    def device_status(self):
        """Raise if a decode kernel gave up a bounded pipeline wait."""
        _lib.check(_lib.load().vq_kivi_device_status(self._h))

    def decode_kernel(self) -> str:
        k = _lib.load().vq_kivi_decode_kernel(self._h)
        if k < 0:
            _lib.check(k)
        return "tensor-core" if k == 1 else "cuda-core"

    def set_split_tokens(self, n: int):
        _lib.check(_lib.load().vq_kivi_set_split_tokens(self._h, int(n)))

    # -- lifetime ------------------------------------------------------------

    def close(self):
        if self._h:
            rc = _lib.load().vq_kivi_free(self._h)
            self._h = ctypes.c_void_p()
            _lib.check(rc)

    def __del__(self):
        try:
            if getattr(self, "_h", None):
                self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
