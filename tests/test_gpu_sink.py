"""KIVI-Sink on the GPU against the oracle: sink choice, planes and sink
rows bit for bit, attention (one query and causal multi-query) within
1e-3 + 1e-3 |oracle|.

Readings (changelog v0.9.0 "New", KIVI-Sink): per (sequence, kv head) the
n_sink prefill tokens with the largest key L2 norms (fp32, channel order;
equal norms: the earlier token) are kept in fp16 and left out of their
groups' min/max; appended tokens never become sinks; n_sink = 0 is plain
KIVI bit for bit.
"""
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


def _inputs(w, seed, n_big=6, gain=25.0):
    """The workload's K, V with n_big seeded tokens per (b, h) whose keys
    are scaled up (candidate sinks), two of them with equal norms."""
    inp = synth.make_inputs(w, seed=seed, device="cpu")
    K = inp["K"].float()
    g = torch.Generator().manual_seed(seed + 1)
    for b in range(w.B):
        S = w.seq_lens[b]
        if S < 4:
            continue
        for h in range(w.H_kv):
            idx = torch.randperm(S, generator=g)[:n_big]
            K[b, h, idx] *= gain
            # an exact tie: the same row at two positions
            K[b, h, idx[1]] = K[b, h, idx[0]]
    return K.half(), inp["V"], inp["q"]


def _pair(w, n_sink, seed):
    import oracle
    from bit_kv_cache_05_gb300.cache import KiviCache
    K, V, q = _inputs(w, seed)
    c = KiviCache(K.cuda(), V.cuda(), w.seq_lens, H_q=w.H_q, bits=w.bits,
                  group=w.group, residual=w.residual, max_seq=w.max_seq,
                  n_sink=n_sink)
    oc = oracle.OracleCache(w.B, w.H_q, w.H_kv, w.D, w.bits, w.group,
                            w.residual, w.max_seq, n_sink=n_sink)
    oc.quantize(K.numpy(), V.numpy(), w.seq_lens)
    return c, oc, K, V, q


def _planes_equal(c, oc, w):
    S, Tq, _ = c.lengths()
    assert list(Tq) == list(oc.lengths()[1])
    for name in ("sink_pos", "sink_k", "sink_v"):
        a = c.export(name).cpu().numpy()
        o = oc.plane(name)
        assert a.shape == o.shape, name
        assert np.array_equal(a.view(np.uint8), o.view(np.uint8)), name
    for b in range(w.B):
        T = Tq[b]
        for name, n in (("Kc", T), ("Vc", T), ("Ks", T // w.group),
                        ("Kz", T // w.group), ("Vs", T), ("Vz", T)):
            a = c.export(name).cpu().numpy()[b, :, :n]
            o = oc.plane(name)[b, :, :n]
            assert np.array_equal(a.view(np.uint8), o.view(np.uint8)), (name, b)


def _close(got, ref, what):
    d = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    assert np.isfinite(got).all(), what
    bad = d > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: max abs diff {d.max():.3e}"


CASES = [
    ("gqa_serving", [700, 1000, 96], 5),    # tensor-core decode, GQA 4:1
    ("pages_S512", [900], 16),              # one head per kv head, 16 sinks
    ("int4_append", [1200, 333], 3),        # 4-bit, g = 64
    ("tiny", [256, 40, 0], 5),              # D = 64, an empty sequence
]


@pytest.mark.parametrize("name,lens,n_sink", CASES, ids=[c[0] for c in CASES])
def test_sink_planes_and_attention(lib, name, lens, n_sink):
    w = synth.shrink(synth.workload(name), lens, n_append=0)
    c, oc, K, V, q = _pair(w, n_sink, seed=50)
    torch.cuda.synchronize()
    _planes_equal(c, oc, w)
    out = c.decode_attend(q.cuda())
    torch.cuda.synchronize()
    _close(out.cpu().numpy(), oc.attend(q.numpy()), f"{name} decode")
    c.device_status()
    if min(lens) >= 7:
        qm = torch.randn(w.B, w.H_q, 7, w.D, generator=torch.Generator().manual_seed(9)).half()
        outm = c.attend_multi(qm.cuda())
        torch.cuda.synchronize()
        _close(outm.cpu().numpy(), oc.attend_multi(qm.numpy()), f"{name} multi")
    c.close()


def test_sink_cuda_core_kernel(lib):
    """Eight query heads per kv head run on the CUDA-core decode."""
    w = synth.Workload("gq8", 2, 16, 2, 128, 2, 32, 32, [800, 301])
    c, oc, K, V, q = _pair(w, 4, seed=51)
    assert c.decode_kernel() == "cuda-core"
    _planes_equal(c, oc, w)
    out = c.decode_attend(q.cuda())
    torch.cuda.synchronize()
    _close(out.cpu().numpy(), oc.attend(q.numpy()), "cuda-core decode")
    c.close()


def test_sinks_in_the_window_survive_appends(lib):
    """Sinks chosen at prefill while still in the fp16 window are left out
    of their groups when appends flush them; appended tokens never become
    sinks (a larger appended key included)."""
    import oracle
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.Workload("win", 2, 8, 2, 128, 2, 32, 32, [60, 45])
    K, V, q = _inputs(w, seed=52, n_big=3)
    n = 200
    g = torch.Generator().manual_seed(3)
    Kn = torch.randn(w.B, w.H_kv, n, w.D, generator=g)
    Kn[:, :, 17] *= 100.0
    Kn = Kn.half()
    Vn = torch.randn(w.B, w.H_kv, n, w.D, generator=g).half()
    c = KiviCache(K.cuda(), V.cuda(), w.seq_lens, H_q=w.H_q, bits=2, group=32,
                  residual=32, max_seq=max(w.seq_lens) + n, n_sink=3)
    oc = oracle.OracleCache(w.B, w.H_q, w.H_kv, w.D, 2, 32, 32,
                            max(w.seq_lens) + n, n_sink=3)
    oc.quantize(K.numpy(), V.numpy(), w.seq_lens)
    for chunk in (1, 30, 169):
        c.append(Kn[:, :, :chunk].contiguous().cuda(), Vn[:, :, :chunk].contiguous().cuda(),
                 [chunk] * w.B)
        oc.append(Kn[:, :, :chunk].numpy(), Vn[:, :, :chunk].numpy(), [chunk] * w.B)
        Kn, Vn = Kn[:, :, chunk:], Vn[:, :, chunk:]
    w.seq_lens = c.lengths()[0]
    torch.cuda.synchronize()
    _planes_equal(c, oc, w)
    out = c.decode_attend(q.cuda())
    torch.cuda.synchronize()
    _close(out.cpu().numpy(), oc.attend(q.numpy()), "after appends")
    c.close()


def test_zero_sinks_is_plain_kivi_on_the_gpu(lib):
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.shrink(synth.workload("gqa_serving"), [500, 77], n_append=0)
    K, V, q = _inputs(w, seed=53)
    a = KiviCache(K.cuda(), V.cuda(), w.seq_lens, H_q=w.H_q, bits=2, group=32,
                  residual=32, n_sink=0)
    oa = a.decode_attend(q.cuda())
    from bit_kv_cache_05_gb300 import _lib
    import ctypes
    L = _lib.load()
    h = ctypes.c_void_p()
    Kd, Vd = K.cuda(), V.cuda()
    _lib.check(L.vq_kivi_quantize(ctypes.byref(a.params), ctypes.c_void_p(Kd.data_ptr()),
                                  ctypes.c_void_p(Vd.data_ptr()), K.shape[2],
                                  (ctypes.c_int32 * w.B)(*w.seq_lens),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                  ctypes.byref(h)))
    ob = torch.empty_like(oa)
    qd = q.cuda()
    _lib.check(L.vq_kivi_decode_attend(h, ctypes.c_void_p(qd.data_ptr()),
                                       ctypes.c_void_p(ob.data_ptr()), 0.0,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
    torch.cuda.synchronize()
    assert torch.equal(oa, ob)
    for name in ("Kc", "Ks", "Kz", "Vc", "Vs", "Vz"):
        raw = torch.empty(a.plane_bytes(name), dtype=torch.uint8, device="cuda")
        _lib.check(L.vq_kivi_export(h, ("Kc", "Ks", "Kz", "Vc", "Vs", "Vz").index(name),
                                    ctypes.c_void_p(raw.data_ptr()), raw.numel(), None))
        torch.cuda.synchronize()
        assert torch.equal(a.export(name).reshape(-1).view(torch.uint8), raw), name
    L.vq_kivi_free(h)
    a.close()


def test_sink_dequantize_and_bytes(lib):
    """The unfused dequantize reads sinks from their fp16 rows; the byte
    accounting counts the sinks of the quantized region once."""
    w = synth.shrink(synth.workload("gqa_serving"), [600, 130], n_append=0)
    c, oc, K, V, q = _pair(w, 4, seed=54)
    Kh, Vh = c.dequantize()
    torch.cuda.synchronize()
    pos = oc.plane("sink_pos")
    _, Tq, _ = oc.lengths()
    n_in = 0
    for b in range(w.B):
        for h in range(w.H_kv):
            for t in pos[b, h]:
                if 0 <= t < Tq[b]:
                    n_in += 1
                    assert torch.equal(Kh[b, h, t].cpu(), K[b, h, t])
                    assert torch.equal(Vh[b, h, t].cpu(), V[b, h, t])
    assert n_in > 0
    assert c.cache_bytes()["sink_bytes"] == n_in * w.D * 4
    c.close()
