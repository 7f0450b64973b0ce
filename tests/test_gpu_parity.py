"""CUDA path vs the CPU oracle, through the C ABI.

Codes, scales, zeros and the residual are compared bit for bit (the
quantizer is integer output decided in fp32 on both sides); attention
outputs must satisfy |gpu - oracle| <= 1e-3 + 1e-3 * |oracle| element-wise
(fp32 accumulation against a double-precision oracle).

Method: VeloxQuant-MLX changelog v0.8.0 "New" (KIVI) and v0.42.0 "Added"
(fused decode-attend over the group-affine cache).
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_05_gb300 import synth

pytestmark = pytest.mark.gpu

ATOL = 1e-3
RTOL = 1e-3


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.fixture(scope="module")
def lib():
    _need_gpu()
    from bit_kv_cache_05_gb300 import _lib, build
    build.build()
    return _lib.load()


def gpu_cache(w, inp, max_seq=None):
    from bit_kv_cache_05_gb300.cache import KiviCache
    return KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=w.bits,
                     group=w.group, residual=w.residual,
                     max_seq=w.max_seq if max_seq is None else max_seq)


def oracle_cache(w, K, V, seq_lens, max_seq=None, B=None, H_kv=None, H_q=None):
    from oracle import OracleCache
    B = w.B if B is None else B
    H_kv = w.H_kv if H_kv is None else H_kv
    H_q = w.H_q if H_q is None else H_q
    oc = OracleCache(B, H_q, H_kv, w.D, w.bits, w.group, w.residual,
                     w.max_seq if max_seq is None else max_seq)
    oc.quantize(K, V, seq_lens)
    return oc


def export_all(c):
    torch.cuda.synchronize()
    out = {n: c.export(n) for n in ("Kc", "Ks", "Kz", "Vc", "Vs", "Vz", "Kr", "Vr")}
    torch.cuda.synchronize()
    return {n: t.cpu().numpy() for n, t in out.items()}


def bits16(a):
    return np.ascontiguousarray(a).view(np.uint16)


def assert_planes_equal(gp, lens_gpu, oc, b_gpu, b_orc, h_gpu=None, h_orc=None):
    """Valid rows of sequence b (all heads, or one head) bit-identical."""
    S, Tq, nres = lens_gpu
    oS, oTq, onres = oc.lengths()
    assert (S[b_gpu], Tq[b_gpu], nres[b_gpu]) == (oS[b_orc], oTq[b_orc], onres[b_orc])
    t, r, g = Tq[b_gpu], nres[b_gpu], oc.group
    hs = slice(None) if h_gpu is None else slice(h_gpu, h_gpu + 1)
    ho = slice(None) if h_orc is None else slice(h_orc, h_orc + 1)
    for name, n in (("Kc", t), ("Vc", t), ("Vs", t), ("Vz", t),
                    ("Ks", t // g), ("Kz", t // g), ("Kr", r), ("Vr", r)):
        a = gp[name][b_gpu, hs, :n]
        o = oc.plane(name)[b_orc, ho, :n]
        if a.dtype == np.float16:
            a, o = bits16(a), bits16(o)
        if not np.array_equal(a, o):
            bad = np.argwhere(a != o)
            raise AssertionError(f"{name} differs at {len(bad)} places, first "
                                 f"{bad[:3].tolist()}: gpu {a[tuple(bad[0])]} "
                                 f"oracle {o[tuple(bad[0])]}")


def assert_attn_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(got - ref)
    ok = d <= ATOL + RTOL * np.abs(ref)
    assert np.isfinite(got).all(), what
    assert ok.all(), (f"{what}: {np.count_nonzero(~ok)} elements outside "
                      f"tolerance; max abs {d.max():.3e}, rel-l2 "
                      f"{np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30):.3e}")
    return float(d.max())


# ---------------------------------------------------------------------------
# oracle-sized cases: whole batches, every plane and every output compared
# ---------------------------------------------------------------------------

SMALL = {
    "tiny": synth.workload("tiny"),
    "pages_S512": synth.workload("pages_S512"),
    "pages_S2048": synth.workload("pages_S2048"),
    "pages_S8192": synth.workload("pages_S8192"),
    "gqa_small": synth.shrink(synth.workload("gqa_serving"), [8192, 1000, 37]),
    "int4_small": synth.shrink(synth.workload("int4_append"), [2000, 333],
                               n_append=0),
    "ragged_small": synth.shrink(synth.workload("ragged_long"),
                                 [16384, 5000, 777, 129]),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_quantize_and_decode_parity(lib, name):
    w = SMALL[name]
    inp = synth.make_inputs(w, device="cuda")
    K, V, q = inp["K"], inp["V"], inp["q"]
    c = gpu_cache(w, inp)
    out = c.decode_attend(q)
    gp = export_all(c)
    lens = c.lengths()
    oc = oracle_cache(w, K.cpu().numpy(), V.cpu().numpy(), w.seq_lens)
    for b in range(w.B):
        assert_planes_equal(gp, lens, oc, b, b)
    ref = oc.attend(q.cpu().numpy())
    assert_attn_close(out.cpu().numpy(), ref, name)
    c.device_status()
    c.close()


@pytest.mark.parametrize("D,bits,g,R,Hq,Hkv,lens", [
    (64, 2, 16, 0, 2, 2, [300, 17, 0]),
    (64, 4, 64, 5, 8, 1, [129, 64, 3]),
    (64, 8, 32, 32, 4, 2, [200, 31]),
    (128, 2, 128, 128, 16, 2, [1000, 255, 256]),
    (128, 4, 32, 7, 2, 1, [777]),
    (128, 8, 64, 64, 32, 4, [513, 64, 1]),
    (256, 2, 32, 32, 4, 4, [1100, 40]),
    (256, 4, 128, 16, 8, 8, [640, 200]),
    (256, 8, 16, 0, 3, 1, [97]),
])
def test_shape_sweep(lib, D, bits, g, R, Hq, Hkv, lens):
    w = synth.Workload("sweep", len(lens), Hq, Hkv, D, bits, g, R, lens,
                       key_kind="chscale", chscale_lo=0.5, chscale_hi=4.0)
    inp = synth.make_inputs(w, seed=7, device="cuda")
    c = gpu_cache(w, inp)
    out = c.decode_attend(inp["q"])
    gp = export_all(c)
    lens_g = c.lengths()
    oc = oracle_cache(w, inp["K"].cpu().numpy(), inp["V"].cpu().numpy(), lens)
    for b in range(w.B):
        assert_planes_equal(gp, lens_g, oc, b, b)
    assert_attn_close(out.cpu().numpy(), oc.attend(inp["q"].cpu().numpy()),
                      f"D={D} b={bits} g={g}")
    c.device_status()
    want = "tensor-core" if D <= 128 and Hq // Hkv <= 4 else "cuda-core"
    assert c.decode_kernel() == want
    c.close()


def test_empty_and_short_sequences(lib):
    """S = 0 (zero output), S < R (all residual), S = R, S = R + g - 1,
    S = R + g in one batch."""
    w = synth.Workload("edge", 6, 8, 2, 128, 2, 32, 32, [0, 1, 31, 32, 63, 64])
    inp = synth.make_inputs(w, seed=3, device="cuda")
    c = gpu_cache(w, inp)
    assert c.lengths()[1] == [0, 0, 0, 0, 0, 32]
    out = c.decode_attend(inp["q"]).cpu().numpy()
    assert (out[0] == 0).all()
    oc = oracle_cache(w, inp["K"].cpu().numpy(), inp["V"].cpu().numpy(),
                      w.seq_lens)
    assert_attn_close(out, oc.attend(inp["q"].cpu().numpy()), "edge")
    c.close()


def test_softmax_scale_argument(lib):
    w = SMALL["tiny"]
    inp = synth.make_inputs(w, seed=5, device="cuda")
    c = gpu_cache(w, inp)
    oc = oracle_cache(w, inp["K"].cpu().numpy(), inp["V"].cpu().numpy(),
                      w.seq_lens)
    for s in (0.05, 0.6):
        out = c.decode_attend(inp["q"], scale=s)
        assert_attn_close(out.cpu().numpy(),
                          oc.attend(inp["q"].cpu().numpy(), scale=s), f"scale {s}")
    c.close()


@pytest.mark.parametrize("bits,g,Hq,Hkv,klo,khi,qmul", [
    (2, 32, 8, 8, 1e-3, 1e-2, 1.0),     # tiny key scales
    (2, 32, 8, 2, 50.0, 300.0, 1.0),    # large key scales (products near the bound)
    (4, 64, 8, 8, 1e-3, 1e2, 1.0),      # five decades across channels
    (2, 32, 4, 4, 0.5, 2.0, 1e-3),      # a nearly flat softmax
    (2, 32, 8, 2, 0.5, 2.0, 20.0),      # a sharp softmax
])
def test_operand_scaling_extremes(lib, bits, g, Hq, Hkv, klo, khi, qmul):
    """The score operand is q' * s_K carried as fp16 hi + lo, scaled per
    head by a power of two from the largest key scale: key scales over
    several decades and query magnitudes from 1e-3 to 20x stay within the
    parity tolerance."""
    lens = [1000, 333]
    w = synth.Workload("extremes", len(lens), Hq, Hkv, 128, bits, g, g, lens,
                       key_kind="chscale", chscale_lo=klo, chscale_hi=khi)
    inp = synth.make_inputs(w, seed=13, device="cuda")
    q = (inp["q"].float() * qmul).half()
    c = gpu_cache(w, inp)
    assert c.decode_kernel() == "tensor-core"
    out = c.decode_attend(q)
    oc = oracle_cache(w, inp["K"].cpu().numpy(), inp["V"].cpu().numpy(), lens)
    assert_attn_close(out.cpu().numpy(), oc.attend(q.cpu().numpy()),
                      f"b={bits} keys x[{klo}, {khi}] q x{qmul}")
    c.close()


# ---------------------------------------------------------------------------
# append: prefill-vs-decode path independence, against the oracle's own
# incremental procedure
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits,g,R", [(2, 32, 32), (4, 64, 64), (2, 16, 0),
                                      (8, 32, 5)])
def test_append_matches_prefill_and_oracle(lib, bits, g, R):
    from bit_kv_cache_05_gb300.cache import KiviCache
    B, Hq, Hkv, D = 3, 8, 2, 128
    S_final = [700, 95, 64 + R]
    w = synth.Workload("app", B, Hq, Hkv, D, bits, g, R, S_final)
    inp = synth.make_inputs(w, seed=11, device="cuda")
    K, V = inp["K"], inp["V"]
    ref = gpu_cache(w, inp)
    S0 = [min(s, 40) for s in S_final]
    c = KiviCache(K, V, S0, H_q=Hq, bits=bits, group=g, residual=R,
                  max_seq=max(S_final))
    oc = oracle_cache(w, K.cpu().numpy(), V.cpu().numpy(), S0,
                      max_seq=max(S_final))
    cur = list(S0)
    step = 0
    Kh, Vh = K.cpu().numpy(), V.cpu().numpy()
    while cur != S_final:
        n = [min([1, 5, 64, 33, 250][(step + b) % 5], S_final[b] - cur[b])
             for b in range(B)]
        nmax = max(max(n), 1)
        Kn = torch.zeros(B, Hkv, nmax, D, dtype=torch.float16, device="cuda")
        Vn = torch.zeros_like(Kn)
        for b in range(B):
            Kn[b, :, : n[b]] = K[b, :, cur[b]: cur[b] + n[b]]
            Vn[b, :, : n[b]] = V[b, :, cur[b]: cur[b] + n[b]]
        c.append(Kn, Vn, n)
        oc.append(Kn.cpu().numpy(), Vn.cpu().numpy(), n)
        cur = [a + x for a, x in zip(cur, n)]
        step += 1
    assert c.lengths() == ref.lengths()
    ga, gr = export_all(c), export_all(ref)
    lens = c.lengths()
    for b in range(B):
        assert_planes_equal(ga, lens, oc, b, b)
        assert_planes_equal(gr, lens, oc, b, b)
    q = inp["q"]
    assert_attn_close(c.decode_attend(q).cpu().numpy(),
                      oc.attend(q.cpu().numpy()), "after appends")
    c.close()
    ref.close()


def test_capacity_error_leaves_cache_unchanged(lib):
    from bit_kv_cache_05_gb300 import _lib
    w = SMALL["tiny"]
    inp = synth.make_inputs(w, device="cuda")
    c = gpu_cache(w, inp, max_seq=260)
    before = c.lengths()
    Kn = torch.zeros(1, 4, 8, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(_lib.VqError) as e:
        c.append(Kn, Kn, [8])
    assert e.value.code == _lib.VQ_ERR_CAPACITY
    assert c.lengths() == before
    c.append(Kn, Kn, [4])
    assert c.lengths()[0] == [260]
    c.close()


# ---------------------------------------------------------------------------
# split-KV partition invariance
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["pages_S8192", "gqa_small"])
def test_split_count_invariance(lib, name):
    w = SMALL[name]
    inp = synth.make_inputs(w, seed=21, device="cuda")
    c = gpu_cache(w, inp)
    assert c.decode_kernel() == "tensor-core"
    outs = []
    for tps in (0, 256, 512, 1024, 4096, 8192):
        c.set_split_tokens(tps)
        outs.append(c.decode_attend(inp["q"]).cpu().numpy())
    # Partitions change only the fp32 summation order: each warp accumulates
    # its segment (up to a whole head here) in fp32, and on the value side
    # the code sum and the zero-point sum, each of the size of the values,
    # cancel to the output, which amplifies the rounding.  Measured spreads
    # against the finest partition: up to 3e-5 (pages shape, outputs ~0.08)
    # and 1e-4 (grouped-query case with outlier keys, outputs up to ~3).
    # The bound is ten times below the parity tolerance, in the same form.
    ref = outs[0]
    for o in outs[1:]:
        assert (np.abs(o - ref) <= 1e-4 + 1e-4 * np.abs(ref)).all()
    c.device_status()
    c.close()


# ---------------------------------------------------------------------------
# full-size workloads (the sizes the benchmark times): sampled heads
# ---------------------------------------------------------------------------

def _sampled_parity(w, inp, c, samples, after_append=None):
    """For each sampled (b, h_kv): a one-sequence oracle built from the same
    input rows; its planes equal the GPU planes of that head, and its outputs
    match the GPU outputs of the query heads that read it."""
    gq = w.H_q // w.H_kv
    out = c.decode_attend(inp["q"]).cpu().numpy()
    gp = export_all(c)
    lens = c.lengths()
    worst = 0.0
    for b, h in samples:
        S0 = w.seq_lens[b]
        K1 = inp["K"][b: b + 1, h: h + 1, :S0].cpu().numpy()
        V1 = inp["V"][b: b + 1, h: h + 1, :S0].cpu().numpy()
        oc = oracle_cache(w, K1, V1, [S0], max_seq=w.max_seq, B=1, H_kv=1,
                          H_q=gq)
        if after_append is not None:
            Kn, Vn, n = after_append
            oc.append(Kn[b: b + 1, h: h + 1].cpu().numpy(),
                      Vn[b: b + 1, h: h + 1].cpu().numpy(), [n[b]])
        assert_planes_equal(gp, lens, oc, b, 0, h, 0)
        q1 = inp["q"][b: b + 1, h * gq: (h + 1) * gq].cpu().numpy()
        ref = oc.attend(q1)
        worst = max(worst, assert_attn_close(out[b, h * gq: (h + 1) * gq],
                                             ref[0], f"{w.name} b={b} h={h}"))
    return worst


@pytest.mark.parametrize("name,samples", [
    ("pages_S65536", [(0, 0), (0, 17), (0, 31)]),
    ("pages_S32768", [(0, 5)]),
    ("gqa_serving", [(0, 0), (7, 3), (15, 7)]),
    ("ragged_long", [(0, 0), (1, 5), (2, 2), (3, 7)]),
])
def test_full_size_sampled(lib, name, samples):
    w = synth.workload(name)
    inp = synth.make_inputs(w, device="cuda")
    c = gpu_cache(w, inp)
    assert c.decode_kernel() == "tensor-core"
    _sampled_parity(w, inp, c, samples)
    c.device_status()
    c.close()
    del inp
    torch.cuda.empty_cache()


def test_full_size_int4_append(lib):
    """The 4-bit workload end to end: prefill 32768 tokens per sequence,
    append the 512-token chunk, decode; sampled heads vs the oracle's own
    prefill + incremental append."""
    w = synth.workload("int4_append")
    inp = synth.make_inputs(w, device="cuda")
    c = gpu_cache(w, inp)
    n = [w.n_append] * w.B
    c.append(inp["K_new"], inp["V_new"], n)
    _sampled_parity(w, inp, c, [(0, 0), (5, 17), (7, 31)],
                    after_append=(inp["K_new"], inp["V_new"], n))
    c.close()
    del inp
    torch.cuda.empty_cache()
