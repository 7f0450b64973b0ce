"""The allocation-free decode entry point, vq_kivi_decode_attend_static.

It serves callers that may not allocate device memory while they run, for
example engines that reserve all device memory at start-up and serve only
from their own pool, plugins whose host forbids allocations, and
latency-critical loops where cudaMalloc would synchronize the device.  Such
a caller keeps the cache planes in memory it owns; here that memory is a
set of torch tensors filled from a regular cache's exported planes.  Two calls
in a row must each match vq_kivi_decode_attend on the same inputs: the
second call reuses the fixed scratch array that still holds the first
call's partial results.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from bit_kv_cache_05_gb300 import synth

pytestmark = pytest.mark.gpu

ATOL = 1e-3
RTOL = 1e-3


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_kv_cache_05_gb300 import _lib, build
    build.build()
    return _lib.load()


def caller_planes(c):
    """The cache's planes copied into caller-owned device tensors, with the
    residual rearranged into the ring layout the entry point documents
    (token at position p in slot p mod (R+g))."""
    S, Tq, nres = c.lengths()
    planes = {n: c.export(n).clone() for n in ("Kc", "Ks", "Kz", "Vc", "Vs", "Vz")}
    rcap = c.residual + c.group
    for name in ("Kr", "Vr"):
        lin = c.export(name)
        ring = torch.zeros_like(lin)
        for b in range(c.B):
            for i in range(nres[b]):
                ring[b, :, (Tq[b] + i) % rcap] = lin[b, :, i]
        planes[name] = ring
    torch.cuda.synchronize()
    return planes


def call_static(lib, c, planes, q, out):
    from bit_kv_cache_05_gb300 import _lib
    p = _lib.Params(c.B, c.H_q, c.H_kv, c.D, c.bits, c.group, c.residual,
                    c.max_seq)
    view = _lib.Planes(*[ctypes.c_void_p(planes[n].data_ptr()) for n in
                         ("Kc", "Ks", "Kz", "Vc", "Vs", "Vz", "Kr", "Vr")])
    S = c.lengths()[0]
    lens = (ctypes.c_int32 * c.B)(*S)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    _lib.check(lib.vq_kivi_decode_attend_static(
        ctypes.byref(p), ctypes.byref(view), lens,
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        0.0, stream))


def close_enough(a, b):
    a = a.cpu().numpy().astype(np.float64)
    b = b.cpu().numpy().astype(np.float64)
    d = np.abs(a - b)
    assert np.isfinite(a).all()
    assert (d <= ATOL + RTOL * np.abs(b)).all(), f"max abs diff {d.max():.3e}"


@pytest.mark.parametrize("w", [
    synth.workload("tiny"),
    synth.shrink(synth.workload("gqa_serving"), [3000, 517, 40]),
    synth.shrink(synth.workload("int4_append"), [1500, 64], n_append=0),
], ids=["tiny", "gqa", "int4"])
def test_static_decode_matches_regular_decode_twice(lib, w):
    from bit_kv_cache_05_gb300.cache import KiviCache
    inp = synth.make_inputs(w, seed=31, device="cuda")
    c = KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=w.bits,
                  group=w.group, residual=w.residual, max_seq=w.max_seq)
    planes = caller_planes(c)
    q1 = inp["q"]
    q2 = (inp["q"].float() * -0.7 + 0.1).half().contiguous()
    ref1 = c.decode_attend(q1).clone()
    ref2 = c.decode_attend(q2).clone()
    out1 = torch.empty_like(ref1)
    out2 = torch.empty_like(ref2)
    call_static(lib, c, planes, q1, out1)
    torch.cuda.synchronize()
    # after the first call (which may load the library's device code and the
    # scratch array), a call changes neither the device's free memory nor
    # torch's pool
    free0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
    call_static(lib, c, planes, q2, out2)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_reserved() == reserved0
    close_enough(out1, ref1)
    close_enough(out2, ref2)
    c.close()


def test_static_decode_rejects_sizes_beyond_the_scratch(lib):
    from bit_kv_cache_05_gb300 import _lib
    # B*H_q*(D+2)*4 bytes for two work items exceed the fixed scratch
    p = _lib.Params(256, 64, 8, 256, 2, 32, 32, 1024)
    dummy = ctypes.c_void_p(256)
    view = _lib.Planes(*([dummy] * 8))
    lens = (ctypes.c_int32 * 256)(*([100] * 256))
    rc = lib.vq_kivi_decode_attend_static(ctypes.byref(p), ctypes.byref(view),
                                          lens, dummy, dummy, 0.0, None)
    assert rc == _lib.VQ_ERR_CAPACITY
    assert b"scratch" in lib.vq_kivi_last_error()
