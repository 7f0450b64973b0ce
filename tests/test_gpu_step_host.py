"""The serving step from pinned host memory (vq_kivi_step_host) against the
same step through device buffers (vq_kivi_append + vq_kivi_decode_attend):
the same kernels run, so every step's output is equal bit for bit, and the
device path is checked against the oracle by the parity tests.  Also the
rejection of buffers that are not pinned host memory."""
import ctypes

import pytest
import torch

from bit_kv_cache_05_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_kv_cache_05_gb300 import _lib, build
    build.build()
    return _lib.load()


@pytest.mark.parametrize("name,kw", [
    ("pages_S512", {}),                                  # tensor-core decode
    ("gqa_serving", {}),                                 # GQA, B = 16
    ("pages_S512", {"kitty_hi": 32}),                    # CUDA-core decode
])
def test_step_host_equals_device_steps(lib, name, kw):
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.workload(name)
    w = synth.shrink(w, [min(s, 700) for s in w.seq_lens[:3]], n_append=0)
    inp = synth.make_inputs(w, seed=81, device="cuda")
    n = 40                                               # crosses a flush
    mk = lambda: KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=2,
                           group=w.group, residual=w.residual,
                           max_seq=w.max_seq + n, **kw)
    a, d = mk(), mk()
    g = torch.Generator().manual_seed(3)
    hK = torch.randn(n, w.B, w.H_kv, w.D, generator=g).half().pin_memory()
    hV = torch.randn(n, w.B, w.H_kv, w.D, generator=g).half().pin_memory()
    hq = torch.randn(n, w.B, w.H_q, w.D, generator=g).half().pin_memory()
    hout = torch.zeros(n, w.B, w.H_q, w.D).pin_memory()
    ones = [1] * w.B
    for i in range(n):
        a.step_host(hK[i], hV[i], hq[i], hout[i])
    torch.cuda.synchronize()
    for i in range(n):
        d.append(hK[i].cuda().unsqueeze(2).contiguous(),
                 hV[i].cuda().unsqueeze(2).contiguous(), ones)
        ref = d.decode_attend(hq[i].cuda()).cpu()
        assert torch.equal(hout[i], ref), f"step {i}"
    assert list(a.lengths()[0]) == list(d.lengths()[0])
    a.device_status()
    a.close()
    d.close()


def test_step_host_rejects_device_and_pageable_buffers(lib):
    from bit_kv_cache_05_gb300 import _lib
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.shrink(synth.workload("tiny"), [100], n_append=0)
    inp = synth.make_inputs(w, seed=82, device="cuda")
    c = KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=2, group=32,
                  residual=32, max_seq=200)
    kv = torch.zeros(w.B, w.H_kv, w.D, dtype=torch.float16)          # pageable
    q = torch.zeros(w.B, w.H_q, w.D, dtype=torch.float16).pin_memory()
    out = torch.zeros(w.B, w.H_q, w.D).pin_memory()
    with pytest.raises(ValueError):
        c.step_host(kv, kv, q, out)
    # the C entry point itself: pageable host memory and device memory
    dq = torch.zeros(w.B, w.H_q, w.D, dtype=torch.float16, device="cuda")
    P = ctypes.c_void_p
    for args in ((kv.data_ptr(), kv.data_ptr(), q.data_ptr(), out.data_ptr()),
                 (q.data_ptr(), q.data_ptr(), dq.data_ptr(), out.data_ptr())):
        rc = lib.vq_kivi_step_host(c._h, *[P(x) for x in args], 0.0, None)
        assert rc == _lib.VQ_ERR_ARG
    assert c.lengths()[0][0] == 100          # the rejected calls changed nothing
    c.close()
