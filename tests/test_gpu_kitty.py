"""Kitty on the GPU against the oracle: the per-group 4-bit channel masks,
mixed-width key rows, key scales / zeros and fp16 values bit for bit, the
fused decode within 1e-3 + 1e-3 |oracle|.

Readings (changelog v0.11.0 "New", Kitty): per key group the kitty_hi
channels of largest running variance (exact integer sums over the tokens up
to the group's last one; the smaller channel on ties) get 4-bit codes, the
rest 2-bit; values stay fp16.
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
        for name, n in (("Kc", Tq[b]), ("Ks", Tq[b] // g), ("Kz", Tq[b] // g),
                        ("Kmask", Tq[b] // g), ("Vf", Tq[b])):
            a = c.export(name).cpu().numpy()[b, :, :n]
            o = oc.plane(name)[b, :, :n]
            assert np.array_equal(a.view(np.uint8), o.view(np.uint8)), (name, b)


CASES = [
    # recipe, lengths, 4-bit channels, group (None: the recipe's)
    ("gqa_serving", [700, 1000, 96], 32, None),   # 8 outlier key channels x10, GQA
    ("pages_S512", [900], 32, None),
    ("pages_S512", [300, 64], 0, None),           # every channel 2-bit
    ("ragged_long", [1500, 200], 128, None),      # every channel 4-bit
    ("tiny", [256, 50], 16, None),                # D = 64
    # groups of 64 (two staged blocks per group), 16 (a block is a group;
    # D = 64: 8-byte channel masks), 128
    ("pages_S512", [1100, 333], 32, 64),
    ("tiny", [300, 170], 16, 16),
    ("gqa_serving", [900, 300], 48, 128),
]


@pytest.mark.parametrize("name,lens,hi,group", CASES,
                         ids=[f"{c[0]}-hi{c[2]}-g{c[3]}" for c in CASES])
def test_kitty_planes_and_decode(lib, name, lens, hi, group):
    import oracle
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.shrink(synth.workload(name), lens, n_append=0)
    w = synth.dataclasses.replace(w, bits=2)
    if group is not None:
        w = synth.dataclasses.replace(w, group=group)
    inp = synth.make_inputs(w, seed=60, device="cpu")
    c = KiviCache(inp["K"].cuda(), inp["V"].cuda(), w.seq_lens, H_q=w.H_q,
                  bits=2, group=w.group, residual=w.residual, max_seq=w.max_seq,
                  kitty_hi=hi)
    oc = oracle.OracleCache(w.B, w.H_q, w.H_kv, w.D, 2, w.group, w.residual,
                            w.max_seq, kitty_hi=hi)
    oc.quantize(inp["K"].numpy(), inp["V"].numpy(), w.seq_lens)
    torch.cuda.synchronize()
    assert c.decode_kernel() == "cuda-core"
    _planes_equal(c, oc, w.group)
    out = c.decode_attend(inp["q"].cuda())
    torch.cuda.synchronize()
    _close(out.cpu().numpy(), oc.attend(inp["q"].numpy()), name)
    c.close()


APPEND_CASES = [
    ("gqa_serving", [100, 37], (1, 7, 64, 100, 128)),
    # one query head per kv head and a short cache: the decode's partial
    # buffer, which a flush borrows for its ranking totals, is small; single
    # tokens up to a flush, then a few more
    ("pages_S512", [500], (1,) * 40 + (3,)),
]


@pytest.mark.parametrize("name,lens,chunks", APPEND_CASES,
                         ids=[c[0] for c in APPEND_CASES])
def test_kitty_appends_match_the_oracle(lib, name, lens, chunks):
    """Appends in several chunk sizes: the running sums carry over between
    flushes exactly as in the oracle's incremental procedure."""
    import oracle
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.shrink(synth.workload(name), lens, n_append=0)
    inp = synth.make_inputs(w, seed=61, device="cpu")
    n_tot = sum(chunks)
    g = torch.Generator().manual_seed(4)
    Kn = (torch.randn(w.B, w.H_kv, n_tot, w.D, generator=g) *
          torch.linspace(0.2, 6, w.D)).half()
    Vn = torch.randn(w.B, w.H_kv, n_tot, w.D, generator=g).half()
    c = KiviCache(inp["K"].cuda(), inp["V"].cuda(), w.seq_lens, H_q=w.H_q,
                  bits=2, group=32, residual=32, max_seq=max(w.seq_lens) + n_tot,
                  kitty_hi=32)
    oc = oracle.OracleCache(w.B, w.H_q, w.H_kv, w.D, 2, 32, 32,
                            max(w.seq_lens) + n_tot, kitty_hi=32)
    oc.quantize(inp["K"].numpy(), inp["V"].numpy(), w.seq_lens)
    at = 0
    for chunk in chunks:
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
    c.close()


def test_kitty_rejects_what_it_does_not_serve(lib):
    from bit_kv_cache_05_gb300 import _lib
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.shrink(synth.workload("tiny"), [200], n_append=0)
    inp = synth.make_inputs(w, seed=62, device="cuda")
    with pytest.raises(_lib.VqError) as ei:
        KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=4, group=32,
                  residual=32, kitty_hi=16)
    assert ei.value.code == _lib.VQ_ERR_UNSUPPORTED
    c = KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=2, group=32,
                  residual=32, kitty_hi=16)
    with pytest.raises(_lib.VqError) as ei:
        c.attend_multi(torch.zeros(1, 4, 2, 64, dtype=torch.float16, device="cuda"))
    assert ei.value.code == _lib.VQ_ERR_UNSUPPORTED
    b = c.cache_bytes()
    # 200 tokens, R = g = 32: 160 quantized per head
    assert b["value_fp16_bytes"] == 4 * 160 * 64 * 2
    assert b["code_bytes"] == 4 * 160 * (64 + 16) // 4
    c.close()
