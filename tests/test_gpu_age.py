"""AgeTieredKV on the GPU against the oracle: codes at each group's tier
width, scales, zeros and tiers bit for bit after a prefill and after appends
that age groups across both boundaries; the fused decode within
1e-3 + 1e-3 |oracle|.

Readings (method overview, AgeTieredKV entry): a group's age counts from
its newest token; tiers 8 / 4 / 2 bits below / between / above the two
boundaries; a group moves down one tier at a time, re-quantized from its
values rebuilt in fp32.
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


def _close(got, ref, what):
    d = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    assert np.isfinite(got).all(), what
    bad = d > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: max abs diff {d.max():.3e}"


def _planes_equal(c, oc, g):
    _, Tq, _ = c.lengths()
    assert list(Tq) == list(oc.lengths()[1])
    for b in range(c.B):
        for name, n in (("Kc", Tq[b]), ("Vc", Tq[b]), ("Ks", Tq[b] // g),
                        ("Kz", Tq[b] // g), ("Vs", Tq[b]), ("Vz", Tq[b]),
                        ("tier", Tq[b] // g)):
            a = c.export(name).cpu().numpy()[b, :, :n]
            o = oc.plane(name)[b, :, :n]
            assert np.array_equal(a.view(np.uint8), o.view(np.uint8)), (name, b)


CASES = [
    # recipe, lengths, residual, (recent, mid, bits), group (None: the recipe's)
    ("pages_S512", [1500, 700], 0, (128, 1024, 8, 4, 2), None),
    ("gqa_serving", [1300, 260, 40], 32, (128, 1024, 8, 4, 2), None),
    ("tiny", [400, 333], 0, (64, 192, 8, 4, 2), None),
    ("pages_S512", [900], 0, (96, 512, 4, 4, 2), None),
    # groups of 64 (two or four staged blocks per group), of 16 (blocks of
    # one group), of 128; every tier at 8 bits (16-token blocks throughout)
    ("pages_S512", [1100, 600], 0, (128, 512, 8, 4, 2), 64),
    ("tiny", [300, 170], 16, (32, 96, 8, 4, 2), 16),
    ("gqa_serving", [900, 300], 32, (128, 256, 4, 2, 2), 128),
    ("pages_S512", [700], 0, (64, 256, 8, 8, 8), None),
]


@pytest.mark.parametrize("name,lens,R,age,group", CASES,
                         ids=[f"{c[0]}-{c[3][0]}-{c[3][2]}{c[3][3]}{c[3][4]}-g{c[4]}"
                              for c in CASES])
def test_age_planes_and_decode(lib, name, lens, R, age, group):
    import oracle
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.shrink(synth.workload(name), lens, n_append=0)
    if group is not None:
        w = synth.dataclasses.replace(w, group=group)
    inp = synth.make_inputs(w, seed=70, device="cpu")
    c = KiviCache(inp["K"].cuda(), inp["V"].cuda(), w.seq_lens, H_q=w.H_q,
                  bits=8, group=w.group, residual=R, max_seq=w.max_seq, age=age)
    oc = oracle.OracleCache(w.B, w.H_q, w.H_kv, w.D, 8, w.group, R, w.max_seq,
                            age=age)
    oc.quantize(inp["K"].numpy(), inp["V"].numpy(), w.seq_lens)
    torch.cuda.synchronize()
    _planes_equal(c, oc, w.group)
    out = c.decode_attend(inp["q"].cuda())
    torch.cuda.synchronize()
    _close(out.cpu().numpy(), oc.attend(inp["q"].numpy()), name)
    c.close()


def test_age_appends_cross_both_boundaries(lib):
    import oracle
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.shrink(synth.workload("gqa_serving"), [90, 33], n_append=0)
    age = (64, 256, 8, 4, 2)
    inp = synth.make_inputs(w, seed=71, device="cpu")
    n_tot = 400
    g = torch.Generator().manual_seed(5)
    Kn = torch.randn(w.B, w.H_kv, n_tot, w.D, generator=g).half()
    Vn = torch.randn(w.B, w.H_kv, n_tot, w.D, generator=g).half()
    cap = max(w.seq_lens) + n_tot
    c = KiviCache(inp["K"].cuda(), inp["V"].cuda(), w.seq_lens, H_q=w.H_q,
                  bits=8, group=32, residual=0, max_seq=cap, age=age)
    oc = oracle.OracleCache(w.B, w.H_q, w.H_kv, w.D, 8, 32, 0, cap, age=age)
    oc.quantize(inp["K"].numpy(), inp["V"].numpy(), w.seq_lens)
    at = 0
    for chunk in (1, 31, 2, 96, 170, 100):
        c.append(Kn[:, :, at:at + chunk].contiguous().cuda(),
                 Vn[:, :, at:at + chunk].contiguous().cuda(), [chunk] * w.B)
        oc.append(Kn[:, :, at:at + chunk].numpy(), Vn[:, :, at:at + chunk].numpy(),
                  [chunk] * w.B)
        at += chunk
        torch.cuda.synchronize()
        _planes_equal(c, oc, 32)
    out = c.decode_attend(inp["q"].cuda())
    torch.cuda.synchronize()
    _close(out.cpu().numpy(), oc.attend(inp["q"].numpy()), "after appends")
    assert {0, 1, 2} <= set(c.export("tier").cpu().numpy()[0, 0, : c.lengths()[1][0] // 32].tolist())
    c.close()


def test_age_rejects_what_it_does_not_serve(lib):
    from bit_kv_cache_05_gb300 import _lib
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.shrink(synth.workload("tiny"), [200], n_append=0)
    inp = synth.make_inputs(w, seed=72, device="cuda")
    with pytest.raises(_lib.VqError) as ei:        # row capacity must be 8 bits
        KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=2, group=32,
                  residual=0, age=(64, 128, 8, 4, 2))
    assert ei.value.code == _lib.VQ_ERR_UNSUPPORTED
    with pytest.raises(_lib.VqError) as ei:        # widths must not grow
        KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=8, group=32,
                  residual=0, age=(64, 128, 2, 4, 8))
    assert ei.value.code == _lib.VQ_ERR_ARG
    c = KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=8, group=32,
                  residual=0, age=(64, 128, 8, 4, 2))
    with pytest.raises(_lib.VqError) as ei:
        c.attend_multi(torch.zeros(1, 4, 2, 64, dtype=torch.float16, device="cuda"))
    assert ei.value.code == _lib.VQ_ERR_UNSUPPORTED
    # 200 tokens, g = 32, R = 0: groups 0..5; ages 168, 136, 104, 72, 40, 8
    # -> tiers 2, 2, 1, 1, 0, 0 -> widths 2, 2, 4, 4, 8, 8 bits
    assert c.export("tier").cpu().numpy()[0, 0, :6].tolist() == [2, 2, 1, 1, 0, 0]
    per_bit = 4 * 32 * 64 // 8 * 2                 # heads x tokens x channels, K and V
    assert c.cache_bytes()["code_bytes"] == per_bit * (2 + 2 + 4 + 4 + 8 + 8)
    c.close()
