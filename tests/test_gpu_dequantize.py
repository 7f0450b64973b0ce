"""Dequantized copy of the cache (the unfused baseline the pages compare the
fused decode against: VeloxQuant-MLX changelog v0.42.0, a dequantize to
fp16 K_hat / V_hat in memory followed by a separate attention).

Quantized tokens must equal fp16_rn(fp32(code * scale + zero)) with code,
scale and zero taken from the oracle's planes (the product and sum are
exact in double; the kernel's fp32 fma rounds that exact value once, then to
fp16), bit for bit; residual tokens equal the oracle's fp16 residual rows.
"""
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


def expected_hat(oc, b, h, S):
    """(K_hat, V_hat) fp16 [S][D] from the oracle's planes."""
    import oracle
    _, Tq_all, _ = oc.lengths()
    Tq = Tq_all[b]
    D, g, bits = oc.D, oc.group, oc.bits
    Kc, Vc = oc.plane("Kc")[b, h], oc.plane("Vc")[b, h]
    Ks = oc.plane("Ks")[b, h].astype(np.float64)
    Kz = oc.plane("Kz")[b, h].astype(np.float64)
    Vs = oc.plane("Vs")[b, h].astype(np.float64)
    Vz = oc.plane("Vz")[b, h].astype(np.float64)
    Kr, Vr = oc.plane("Kr")[b, h], oc.plane("Vr")[b, h]
    K = np.zeros((S, D), np.float16)
    V = np.zeros((S, D), np.float16)
    for t in range(Tq):
        kc = oracle.unpack_codes(Kc[t], D, bits).astype(np.float64)
        vc = oracle.unpack_codes(Vc[t], D, bits).astype(np.float64)
        k = kc * Ks[t // g] + Kz[t // g]
        v = vc * np.repeat(Vs[t], g) + np.repeat(Vz[t], g)
        K[t] = k.astype(np.float32).astype(np.float16)
        V[t] = v.astype(np.float32).astype(np.float16)
    K[Tq:S] = Kr[: S - Tq]
    V[Tq:S] = Vr[: S - Tq]
    return K, V


@pytest.mark.parametrize("D,bits,g,R,Hq,Hkv,lens", [
    (128, 2, 32, 32, 4, 4, [700, 0, 31, 64]),     # 2-bit, MMA-fragment order
    (128, 4, 64, 64, 8, 2, [1000, 129]),          # 4-bit, MMA-fragment order
    (64, 8, 32, 16, 2, 2, [333, 48]),             # 8-bit, packed order
    (256, 2, 32, 32, 4, 4, [400, 70]),            # CUDA-core cache, packed order
])
def test_dequantize_matches_oracle_planes(lib, D, bits, g, R, Hq, Hkv, lens):
    from oracle import OracleCache
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.Workload("dq", len(lens), Hq, Hkv, D, bits, g, R, lens,
                       key_kind="chscale", chscale_lo=0.5, chscale_hi=4.0)
    inp = synth.make_inputs(w, seed=11, device="cuda")
    c = KiviCache(inp["K"], inp["V"], lens, H_q=Hq, bits=bits, group=g,
                  residual=R, max_seq=w.max_seq)
    Kh, Vh = c.dequantize()
    torch.cuda.synchronize()
    Kh, Vh = Kh.cpu().numpy(), Vh.cpu().numpy()
    oc = OracleCache(w.B, Hq, Hkv, D, bits, g, R, w.max_seq)
    oc.quantize(inp["K"].cpu().numpy(), inp["V"].cpu().numpy(), lens)
    for b, S in enumerate(lens):
        for h in range(Hkv):
            ek, ev = expected_hat(oc, b, h, S)
            assert np.array_equal(Kh[b, h, :S].view(np.uint16), ek.view(np.uint16)), (b, h)
            assert np.array_equal(Vh[b, h, :S].view(np.uint16), ev.view(np.uint16)), (b, h)
    c.close()


def test_dequantize_rejects_bad_arguments(lib):
    from bit_kv_cache_05_gb300 import _lib
    from bit_kv_cache_05_gb300.cache import KiviCache
    w = synth.workload("tiny")
    inp = synth.make_inputs(w, device="cuda")
    c = KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=w.bits,
                  group=w.group, residual=w.residual, max_seq=w.max_seq)
    short = torch.empty(w.B, w.H_kv, w.seq_lens[0] - 1, w.D, dtype=torch.float16,
                        device="cuda")
    with pytest.raises(_lib.VqError):
        c.dequantize(out=(short, short.clone()))
    c.close()
