"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/vq_kivi.h declares, and rejects bad arguments with
the documented status codes before touching the device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT, cuda_ok


def declared_functions():
    src = open(os.path.join(ROOT, "include", "vq_kivi.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(vq_kivi_\w+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("vq_kivi_quantize", "vq_kivi_append",
                 "vq_kivi_decode_attend", "vq_kivi_free"):
        assert must in names


def test_library_exports_every_declared_symbol(vqlib):
    from bit_kv_cache_05_gb300 import _lib
    names = declared_functions()
    for n in names:
        assert hasattr(vqlib, n), n
    assert set(names) <= set(_lib.EXPORTS) | set(names)
    assert set(_lib.EXPORTS) == set(names)


def _params(**kw):
    from bit_kv_cache_05_gb300._lib import Params
    d = dict(B=1, H_q=4, H_kv=4, D=64, bits=2, group=32, residual=32,
             max_seq=256)
    d.update(kw)
    return Params(**d)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), -1), (dict(D=-1), -1), (dict(max_seq=-5), -1),
    (dict(B=257), -2), (dict(H_q=6, H_kv=4), -2), (dict(H_q=32, H_kv=2), -2),
    (dict(D=96), -2), (dict(bits=3), -2), (dict(group=48), -2),
    (dict(D=64, group=128), -2), (dict(residual=5000), -2),
])
def test_bad_params_rejected_without_device(vqlib, kw, code):
    p = _params(**kw)
    h = ctypes.c_void_p()
    lens = (ctypes.c_int32 * max(p.B, 1))(*([1] * max(p.B, 1)))
    rc = vqlib.vq_kivi_quantize(ctypes.byref(p), None, None, 1, lens, None,
                                ctypes.byref(h))
    assert rc == code
    assert not h.value
    assert len(vqlib.vq_kivi_last_error()) > 0


def test_length_checks(vqlib):
    p = _params()
    h = ctypes.c_void_p()
    rc = vqlib.vq_kivi_quantize(ctypes.byref(p), None, None, 1, None, None,
                                ctypes.byref(h))
    assert rc == -1                       # seq_lens NULL
    lens = (ctypes.c_int32 * 1)(300)      # > max_seq
    rc = vqlib.vq_kivi_quantize(ctypes.byref(p), None, None, 300, lens, None,
                                ctypes.byref(h))
    assert rc == -3
    lens = (ctypes.c_int32 * 1)(-1)
    rc = vqlib.vq_kivi_quantize(ctypes.byref(p), None, None, 1, lens, None,
                                ctypes.byref(h))
    assert rc == -1
    lens = (ctypes.c_int32 * 1)(10)
    rc = vqlib.vq_kivi_quantize(ctypes.byref(p), None, None, 10, lens, None,
                                ctypes.byref(h))
    assert rc == -1                       # K, V NULL with a non-empty sequence
    assert b"NULL" in vqlib.vq_kivi_last_error()


def test_null_handles(vqlib):
    assert vqlib.vq_kivi_free(None) == 0
    assert vqlib.vq_kivi_lengths(None, None, None, None) == -1
    assert vqlib.vq_kivi_plane_bytes(None, 0) == 0
    assert vqlib.vq_kivi_set_split_tokens(None, 0) == -1
    assert vqlib.vq_kivi_decode_attend(None, None, None, 0.0, None) == -1
    assert vqlib.vq_kivi_append(None, None, None, 0, None, None) == -1
    assert vqlib.vq_kivi_step_host(None, None, None, None, None, 0.0, None) == -1
    assert vqlib.vq_kivi_export(None, 0, None, 0, None) == -1
    assert isinstance(vqlib.vq_kivi_launch_count(), int)


@pytest.mark.skipif(cuda_ok(), reason="checks the no-device error path")
def test_no_device_gives_cuda_error(vqlib):
    p = _params()
    h = ctypes.c_void_p()
    lens = (ctypes.c_int32 * 1)(0)
    rc = vqlib.vq_kivi_quantize(ctypes.byref(p), None, None, 1, lens, None,
                                ctypes.byref(h))
    assert rc == -5
    assert not h.value
