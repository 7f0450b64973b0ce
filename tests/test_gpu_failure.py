"""Failure detection of the tensor-core decode, without a GPU fault.

Every pipeline wait in the decode kernel is bounded.  The testing hook
vq_kivi_debug_fail_chunk makes one warp wait for shared-memory copies that
are never issued; its wait gives up after about half a second, the kernel
records the failure and returns, and the host reads the status with
vq_kivi_device_status.  The context stays usable: the next decode on the
same cache is correct again.
"""
import ctypes

import numpy as np
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


def test_bounded_wait_reports_and_recovers(lib):
    from bit_kv_cache_05_gb300 import _lib
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.workload("pages_S2048")
    inp = synth.make_inputs(w, device="cuda")
    c = KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=w.bits,
                  group=w.group, residual=w.residual)
    assert c.decode_kernel() == "tensor-core"
    good = c.decode_attend(inp["q"]).clone()
    c.device_status()
    _lib.check(lib.vq_kivi_debug_fail_chunk(c._h, 5))
    c.decode_attend(inp["q"])
    with pytest.raises(_lib.VqError) as e:
        c.device_status()
    assert e.value.code == _lib.VQ_ERR_CUDA
    assert b"gave up" in lib.vq_kivi_last_error()
    # the hook is one-shot; the next decode is right again
    again = c.decode_attend(inp["q"])
    c.device_status()
    assert torch.equal(again, good)
    c.close()
