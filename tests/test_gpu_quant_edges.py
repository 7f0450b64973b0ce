"""Quantizer edge cases on the GPU, bit for bit against the oracle: the
hand-worked groups of tests/golden/group_quant_worked.json (ties to even, a
code decided by fp32 rounding, constant groups) and groups built from small
integer grids, whose quotients (x - min) / scale fall exactly on, or within
one rounding of, half-integers -- the cases where the kernel's reciprocal
shortcut must defer to the exact quotient.

Method: VeloxQuant-MLX changelog v0.8.0 "New" (KIVI) and v0.42.0 "Added"
(codes plus a per-group (scale, zero) from the group min/max).
"""
import json
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "group_quant_worked.json")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_kv_cache_05_gb300 import _lib, build
    build.build()
    return _lib.load()


def _compare(K, V, bits, g, R):
    """Quantize fp16 K, V [1][1][S][D] on the GPU and in the oracle; all
    planes of the quantized region must match bit for bit."""
    import oracle
    from bit_kv_cache_05_gb300.cache import KiviCache
    S, D = K.shape[2], K.shape[3]
    c = KiviCache(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda(), [S],
                  H_q=1, bits=bits, group=g, residual=R)
    torch.cuda.synchronize()
    oc = oracle.OracleCache(1, 1, 1, D, bits, g, R, S)
    oc.quantize(K, V, [S])
    Tq = c.lengths()[1][0]
    assert Tq == oc.lengths()[1][0] and Tq > 0
    for name, n in (("Kc", Tq), ("Vc", Tq), ("Ks", Tq // g), ("Kz", Tq // g),
                    ("Vs", Tq), ("Vz", Tq)):
        a = c.export(name).cpu().numpy()[0, 0, :n]
        o = oc.plane(name)[0, 0, :n]
        if a.dtype == np.float16:
            a, o = a.view(np.uint16), o.view(np.uint16)
        assert np.array_equal(a, o), name
    c.close()


def test_golden_groups_through_the_kernel(lib):
    cases = json.load(open(GOLDEN))["cases"]
    rng = np.random.default_rng(0)
    for case in cases:
        bits = case["bits"]
        g, D, R = 16, 64, 16
        x = np.array(case["x"], np.float16)
        col = np.resize(x, g)              # the case's values, repeated
        S = 2 * g + R
        K = rng.standard_normal((1, 1, S, D)).astype(np.float16)
        V = rng.standard_normal((1, 1, S, D)).astype(np.float16)
        K[0, 0, :g, 5] = col               # one key channel group
        K[0, 0, g:2 * g, 9] = col[::-1]
        V[0, 0, 3, 16:32] = col            # one value group of token 3
        V[0, 0, 20, 0:16] = col[::-1]
        _compare(K, V, bits, g, R)


@pytest.mark.parametrize("bits,g", [(2, 16), (2, 32), (4, 32), (4, 64),
                                    (8, 16), (8, 64)])
def test_half_integer_quotients(lib, bits, g):
    """Values on integer grids m * 2^e: (x - min) / scale = P (m - m0) / span
    hits half-integers exactly for many groups."""
    rng = np.random.default_rng(100 + bits + g)
    D, R = 128, 8
    S = 64 * g + R
    P = (1 << bits) - 1
    span = rng.choice([2 * P, 2, 4, 6, 10, 2 * P + 2], size=(S, D))
    m = rng.integers(0, 1 << 10, size=(S, D))
    m = m % (span + 1)
    # keys share an exponent per channel, values per token, so every group
    # is one integer grid
    e_ch = rng.integers(-10, 4, size=(1, D)).astype(np.float64)
    e_tok = rng.integers(-10, 4, size=(S, 1)).astype(np.float64)
    K = (m * 2.0 ** e_ch).astype(np.float16)[None, None]
    V = (m * 2.0 ** e_tok).astype(np.float16)[None, None]
    _compare(K, V, bits, g, R)


@pytest.mark.parametrize("bits,g", [(2, 16), (4, 32), (8, 16)])
def test_signed_zero_groups(lib, bits, g):
    """Groups made only of +0.0 and -0.0, in both orders (a -0.0 first and a
    +0.0 first), on key channels and on value groups: the stored scale and
    zero are +0.0 and the codes 0, bit for bit as in the oracle, whatever the
    order in which the kernel's min/max reduction meets the two zeros."""
    rng = np.random.default_rng(200 + bits + g)
    D, R = 64, 16
    S = 4 * g + R
    K = rng.standard_normal((1, 1, S, D)).astype(np.float16)
    V = rng.standard_normal((1, 1, S, D)).astype(np.float16)
    nf = np.resize(np.array([-0.0, 0.0], np.float16), g)   # -0 first
    pf = np.resize(np.array([0.0, -0.0], np.float16), g)   # +0 first
    allneg = np.full(g, -0.0, np.float16)
    for G, col in enumerate((nf, pf, allneg, pf[::-1])):
        K[0, 0, G * g:(G + 1) * g, 7 + G] = col
        K[0, 0, G * g:(G + 1) * g, 40] = col if G % 2 else col[::-1]
    for t, col in ((1, nf), (2, pf), (g + 3, allneg), (2 * g, nf[::-1])):
        j = t % (D // g)
        V[0, 0, t, j * g:(j + 1) * g] = col
    _compare(K, V, bits, g, R)
