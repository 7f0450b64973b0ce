"""The rows beyond the plain cache at the sizes the benchmark times: KIVI-Sink,
Kitty and AgeTieredKV caches of the pages' decode shape at S_kv = 32768
(B = 1, 32 heads, D = 128; the pages' defaults: 5 sinks, 32 of 128 key
channels in 4 bits, tiers 8 / 4 / 2 bits at 128 / 1024 tokens of age), and
the multi-query attend of the 4-bit workload's 512-token chunk (B = 8,
32 heads, S_kv = 33280).  For sampled heads a one-sequence oracle is built
from the same input rows: its planes equal the GPU planes of that head and
its outputs match the GPU outputs (|d| <= 1e-3 + 1e-3 |oracle|); for the
multi-query attend, sampled queries of the chunk (first, middle, last).
"""
import numpy as np
import pytest
import torch

import oracle
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


def _close(got, ref, what):
    d = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    assert np.isfinite(got).all(), what
    bad = d > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: max abs diff {d.max():.3e}"


def _head_planes_equal(c, oc, b, h, names, Tq, g):
    for name in names:
        a = c.export(name).cpu().numpy()[b, h]
        o = oc.plane(name)[0, 0]
        if name in ("Ks", "Kz", "Kmask", "tier"):
            n = Tq // g
        elif name.startswith("sink"):
            n = a.shape[0]
        else:
            n = Tq
        assert np.array_equal(a[:n].view(np.uint8), o[:n].view(np.uint8)), (name, b, h)


ROWS = [
    ("sink", dict(n_sink=5), dict(n_sink=5), 2, 32,
     ("Kc", "Ks", "Kz", "Vc", "Vs", "Vz", "sink_pos", "sink_k", "sink_v")),
    ("kitty", dict(kitty_hi=32), dict(kitty_hi=32), 2, 32,
     ("Kc", "Ks", "Kz", "Kmask", "Vf")),
    ("age", dict(age=(128, 1024, 8, 4, 2)), dict(age=(128, 1024, 8, 4, 2)), 8, 0,
     ("Kc", "Ks", "Kz", "Vc", "Vs", "Vz", "tier")),
]


@pytest.mark.parametrize("row,gpu_kw,orc_kw,bits,R,names", ROWS,
                         ids=[r[0] for r in ROWS])
def test_row_full_size_sampled_heads(lib, row, gpu_kw, orc_kw, bits, R, names):
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.dataclasses.replace(synth.workload("pages_S32768"), bits=bits, residual=R)
    inp = synth.make_inputs(w, device="cuda")
    c = KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=bits,
                  group=w.group, residual=R, max_seq=w.max_seq, **gpu_kw)
    out = c.decode_attend(inp["q"]).cpu().numpy()
    S = w.seq_lens[0]
    Tq = c.lengths()[1][0]
    for h in (0, 13, 31):
        K1 = inp["K"][0:1, h:h + 1].cpu().numpy()
        V1 = inp["V"][0:1, h:h + 1].cpu().numpy()
        oc = oracle.OracleCache(1, 1, 1, w.D, bits, w.group, R, w.max_seq, **orc_kw)
        oc.quantize(K1, V1, [S])
        assert oc.lengths()[1][0] == Tq
        _head_planes_equal(c, oc, 0, h, names, Tq, w.group)
        ref = oc.attend(inp["q"][0:1, h:h + 1].cpu().numpy())
        _close(out[0, h], ref[0, 0], f"{row} h={h}")
    c.device_status()
    c.close()
    del inp
    torch.cuda.empty_cache()


def test_multi_query_full_size_sampled(lib):
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.workload("int4_append")
    inp = synth.make_inputs(w, device="cuda")
    n = w.n_append
    c = KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=w.bits,
                  group=w.group, residual=w.residual, max_seq=w.max_seq)
    c.append(inp["K_new"], inp["V_new"], [n] * w.B)
    g = torch.Generator(device="cuda").manual_seed(17)
    q = torch.randn(w.B, w.H_q, n, w.D, generator=g, device="cuda").half()
    out = c.attend_multi(q).cpu().numpy()
    S = w.seq_lens[0] + n
    for b, h in ((0, 0), (5, 17), (7, 31)):
        K1 = inp["K"][b:b + 1, h:h + 1].cpu().numpy()
        V1 = inp["V"][b:b + 1, h:h + 1].cpu().numpy()
        oc = oracle.OracleCache(1, 1, 1, w.D, w.bits, w.group, w.residual, w.max_seq)
        oc.quantize(K1, V1, [w.seq_lens[b]])
        oc.append(inp["K_new"][b:b + 1, h:h + 1].cpu().numpy(),
                  inp["V_new"][b:b + 1, h:h + 1].cpu().numpy(), [n])
        for i in (0, 255, n - 1):
            ref = oc.attend_prefix(0, 0, q[b, h, i].cpu().numpy(), S - n + i)
            _close(out[b, h, i], ref, f"b={b} h={h} i={i}")
    c.device_status()
    c.close()
    del inp
    torch.cuda.empty_cache()
