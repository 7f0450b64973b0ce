"""Pins of the CPU oracle against facts fixed by the pages and by arithmetic,
not against the oracle itself.

Sources: VeloxQuant-MLX changelog v0.8.0 "New" (KIVI: per-channel keys,
per-token values, fp16 residual window, group size), changelog v0.42.0
"Added" (codes plus a per-group (scale, zero) from the group min/max;
attention over rebuilt k_hat / v_hat), changelog v0.28.0 (chunk-flush
residual; prefill and decode give identical state), method overview
(AgeTieredKV entry: recency-gated window, shared min/max group quantizer).

Each pin is chosen so that a plausible slip in the oracle (a dropped zero
point, a transposed key/value axis, a wrong residual rule, an off-by-one in
packing, a wrong GQA head map, a missing max-subtraction) fails one of them.
"""
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "group_quant_worked.json")


# ---------------------------------------------------------------------------
# independent helpers (numpy, written separately from the C oracle)
# ---------------------------------------------------------------------------

def np_unpack_rows(packed: np.ndarray, D: int, bits: int) -> np.ndarray:
    """[..., D*bits/8] uint8 -> [..., D] codes, LSB-first within each byte."""
    per = 8 // bits
    mask = (1 << bits) - 1
    shifts = (np.arange(per, dtype=np.uint8) * bits)
    x = (packed[..., :, None] >> shifts) & mask
    return x.reshape(*packed.shape[:-1], packed.shape[-1] * per)[..., :D]


def np_dequant_sequence(oc, b, h):
    """k_hat, v_hat [S][D] in long double for sequence (b, h) from the
    oracle's exported canonical planes."""
    S, Tq, nres = (x[b] for x in oc.lengths())
    D, g, bits = oc.D, oc.group, oc.bits
    L = np.longdouble
    kc = np_unpack_rows(oc.plane("Kc")[b, h, :Tq], D, bits).astype(L)
    vc = np_unpack_rows(oc.plane("Vc")[b, h, :Tq], D, bits).astype(L)
    Ks = oc.plane("Ks")[b, h, : Tq // g].astype(L)      # [G][D]
    Kz = oc.plane("Kz")[b, h, : Tq // g].astype(L)
    Vs = oc.plane("Vs")[b, h, :Tq].astype(L)            # [Tq][D/g]
    Vz = oc.plane("Vz")[b, h, :Tq].astype(L)
    tok_group = np.arange(Tq) // g
    kq = kc * Ks[tok_group] + Kz[tok_group]
    ch_group = np.arange(D) // g
    vq = vc * Vs[:, ch_group] + Vz[:, ch_group]
    kr = oc.plane("Kr")[b, h, :nres].astype(L)
    vr = oc.plane("Vr")[b, h, :nres].astype(L)
    return np.concatenate([kq, kr]), np.concatenate([vq, vr])


def np_dense_attention(q, K, V, scale):
    s = (K @ q) * scale
    p = np.exp(s - s.max())
    return (p[:, None] * V).sum(0) / p.sum()


def rand_f16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


# ---------------------------------------------------------------------------
# group quantizer
# ---------------------------------------------------------------------------

def test_golden_worked_examples(oracle_mod):
    cases = json.load(open(GOLDEN))["cases"]
    assert len(cases) >= 6
    for c in cases:
        codes, _, s16, z16 = oracle_mod.quant_group(
            np.array(c["x"], np.float32), c["bits"])
        assert codes.tolist() == c["codes"], c["name"]
        assert s16 == int(c["scale_f16_bits"], 16), c["name"]
        assert z16 == int(c["zero_f16_bits"], 16), c["name"]
        packed = oracle_mod.pack_codes(codes, c["bits"])
        assert packed.tolist() == c["packed"], c["name"]
        back = oracle_mod.unpack_codes(packed, len(c["x"]), c["bits"])
        assert back.tolist() == c["codes"], c["name"]


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_extremes_get_end_codes(oracle_mod, bits):
    """Every non-constant group holds code 0 at its min and 2^b-1 at its max."""
    rng = np.random.default_rng(1)
    P = (1 << bits) - 1
    for n in (2, 3, 32, 64, 128):
        for _ in range(50):
            x = rand_f16(rng, n, scale=rng.uniform(0.01, 100)).astype(np.float32)
            if x.max() == x.min():
                continue
            codes, _, _, _ = oracle_mod.quant_group(x, bits)
            assert codes[np.argmin(x)] == 0
            assert codes[np.argmax(x)] == P
            assert codes.max() <= P


@pytest.mark.parametrize("bits", [2, 4])
def test_reconstruction_within_half_scale(oracle_mod, bits):
    """|x - (code*scale + min)| <= scale/2 (fp32 scale), and with the stored
    fp16 scale <= scale/2 + (2^b-1)*|scale32 - scale16| (the pages' "per
    element error at most half a quantization step")."""
    rng = np.random.default_rng(2)
    P = (1 << bits) - 1
    for _ in range(300):
        n = int(rng.choice([4, 32, 64, 128]))
        x = rand_f16(rng, n, scale=rng.uniform(0.05, 20)).astype(np.float32)
        codes, s32, s16, z16 = oracle_mod.quant_group(x, bits)
        mn = np.float64(x.min())
        assert np.float16(np.uint16(z16).view(np.float16)) == np.float16(mn)
        err32 = np.abs(x.astype(np.float64) - (codes * np.float64(s32) + mn))
        assert err32.max() <= np.float64(s32) * (0.5 + 2.0 ** -20) + 1e-30
        sc16 = np.float64(np.uint16(s16).view(np.float16))
        err16 = np.abs(x - (codes * sc16 + mn))
        bound = np.float64(s32) * (0.5 + 2.0 ** -20) + P * abs(np.float64(s32) - sc16)
        assert err16.max() <= bound


def test_eight_bit_near_lossless(oracle_mod):
    rng = np.random.default_rng(3)
    for _ in range(200):
        x = rand_f16(rng, 64, scale=3.0).astype(np.float32)
        codes, s32, s16, z16 = oracle_mod.quant_group(x, 8)
        sc16 = np.float64(np.uint16(s16).view(np.float16))
        rng_x = float(x.max() - x.min())
        rec = codes * sc16 + np.float64(x.min())
        # half a step (range/510) plus the fp16 rounding of the scale
        assert np.abs(rec - x).max() <= rng_x / 510 * (1 + 1e-6) + 255 * abs(s32 - sc16) + 1e-12


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_constant_group(oracle_mod, bits):
    for v in (0.0, 1.0, -3.25, 65504.0, 6e-8):
        x = np.full(32, np.float16(v), np.float16).astype(np.float32)
        codes, s32, s16, z16 = oracle_mod.quant_group(x, bits)
        assert s32 == 0.0 and s16 == 0
        assert (codes == 0).all()
        assert np.uint16(z16).view(np.float16) == np.float16(v)


@pytest.mark.parametrize("bits", [2, 4])
def test_power_of_two_scaling(oracle_mod, bits):
    """Scaling the inputs by 2^k leaves every code unchanged and scales the
    stored scale and zero exactly (while fp16 stays normal)."""
    rng = np.random.default_rng(4)
    for _ in range(100):
        x = rand_f16(rng, 32).astype(np.float32)
        c0, s0, h0, z0 = oracle_mod.quant_group(x, bits)
        for k in (-3, -1, 1, 4):
            xs = (x * np.float32(2.0 ** k))
            c1, s1, h1, z1 = oracle_mod.quant_group(xs, bits)
            assert (c0 == c1).all()
            assert s1 == np.float32(s0 * 2.0 ** k)
            f0 = np.float64(np.uint16(h0).view(np.float16))
            f1 = np.float64(np.uint16(h1).view(np.float16))
            if f0 > 2 ** -13 and f1 > 2 ** -13:
                assert f1 == f0 * 2.0 ** k
            assert np.float64(np.uint16(z1).view(np.float16)) == \
                np.float64(np.uint16(z0).view(np.float16)) * 2.0 ** k


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_pack_matches_numpy_unpacker(oracle_mod, bits):
    rng = np.random.default_rng(5)
    for n in (8, 64, 128):
        codes = rng.integers(0, 1 << bits, n).astype(np.uint8)
        packed = oracle_mod.pack_codes(codes, bits)
        assert packed.size == n * bits // 8
        assert (np_unpack_rows(packed[None], n, bits)[0] == codes).all()


# ---------------------------------------------------------------------------
# the cache: axes, residual rule, append path independence
# ---------------------------------------------------------------------------

def test_key_axis_is_per_channel_value_axis_per_token(oracle_mod):
    """Keys: one (scale, zero) per (token group, channel); values: one per
    (token, channel group).  Build K whose channel c is constant over tokens
    (so every key group is constant) and V whose token t is constant over
    channels (so every value group is constant)."""
    from oracle import OracleCache
    B, H, D, g, R, S = 1, 1, 16, 4, 4, 20
    ch = (np.arange(D) - 7.0).astype(np.float16)
    K = np.broadcast_to(ch, (B, H, S, D)).copy()
    tv = (np.arange(S) * 0.5 - 3.0).astype(np.float16)
    V = np.broadcast_to(tv[:, None], (B, H, S, D)).copy()
    oc = OracleCache(B, H, H, D, 2, g, R, S)
    oc.quantize(K, V, [S])
    _, Tq, _ = oc.lengths()
    assert Tq[0] == 16
    assert (oc.plane("Ks")[0, 0, :4] == 0).all()
    assert (oc.plane("Kz")[0, 0, :4] == ch[None, :]).all()
    assert (oc.plane("Vs")[0, 0, :16] == 0).all()
    assert (oc.plane("Vz")[0, 0, :16] == tv[:16, None]).all()
    assert (oc.plane("Kc")[0, 0, :16] == 0).all()


@pytest.mark.parametrize("R,g", [(32, 32), (0, 32), (4, 8), (64, 64), (5, 4)])
def test_residual_window_rule(oracle_mod, R, g):
    """Whole groups are quantized; between R and R+g-1 newest tokens (all of
    them when S < R) stay fp16, stored exactly."""
    from oracle import OracleCache
    rng = np.random.default_rng(6)
    D = 8 if g <= 8 else g
    lens = [0, 1, R - 1 if R else 0, R, R + g - 1, R + g, R + 3 * g + 1, 200]
    lens = [max(0, x) for x in lens]
    S_max = max(lens)
    K = rand_f16(rng, (len(lens), 1, S_max, D))
    V = rand_f16(rng, (len(lens), 1, S_max, D))
    oc = OracleCache(len(lens), 1, 1, D, 2, g, R, S_max)
    oc.quantize(K, V, lens)
    S, Tq, nres = oc.lengths()
    for b, L in enumerate(lens):
        assert S[b] == L and Tq[b] + nres[b] == L and Tq[b] % g == 0
        if L < R:
            assert Tq[b] == 0
        else:
            assert R <= nres[b] < R + g
        assert (oc.plane("Kr")[b, 0, : nres[b]] == K[b, 0, Tq[b]:L]).all()
        assert (oc.plane("Vr")[b, 0, : nres[b]] == V[b, 0, Tq[b]:L]).all()


@pytest.mark.parametrize("bits,g,R", [(2, 8, 8), (4, 4, 0), (2, 4, 7), (8, 8, 16)])
def test_append_path_independence(oracle_mod, bits, g, R):
    """quantize(S) == quantize(S0) followed by appends of any chunking, bit
    for bit (the prefill-vs-decode identity the pages pin for chunk-flush
    residual caches)."""
    from oracle import OracleCache
    rng = np.random.default_rng(7)
    B, Hq, H, D = 3, 4, 2, 16
    S_final = [57, 13, 96]
    S_max = max(S_final)
    K = rand_f16(rng, (B, H, S_max, D), 2.0)
    V = rand_f16(rng, (B, H, S_max, D))
    ref = OracleCache(B, Hq, H, D, bits, g, R, S_max)
    ref.quantize(K, V, S_final)
    for chunking in ("ones", "mixed"):
        oc = OracleCache(B, Hq, H, D, bits, g, R, S_max)
        S0 = [min(s, 5) for s in S_final]
        oc.quantize(K, V, S0)
        cur = list(S0)
        step = 0
        while cur != S_final:
            n = []
            for b in range(B):
                want = 1 if chunking == "ones" else [1, 7, 3, 19][(step + b) % 4]
                n.append(min(want, S_final[b] - cur[b]))
            nmax = max(n)
            Kn = np.zeros((B, H, nmax, D), np.float16)
            Vn = np.zeros((B, H, nmax, D), np.float16)
            for b in range(B):
                Kn[b, :, : n[b]] = K[b, :, cur[b]: cur[b] + n[b]]
                Vn[b, :, : n[b]] = V[b, :, cur[b]: cur[b] + n[b]]
            oc.append(Kn, Vn, n)
            cur = [c + x for c, x in zip(cur, n)]
            step += 1
        for a, b_ in zip(oc.lengths(), ref.lengths()):
            assert (a == b_).all()
        S, Tq, nres = ref.lengths()
        for b in range(B):
            for name in ("Kc", "Vc", "Vs", "Vz"):
                assert (oc.plane(name)[b, :, : Tq[b]] == ref.plane(name)[b, :, : Tq[b]]).all(), name
            for name in ("Ks", "Kz"):
                G = Tq[b] // g
                assert (oc.plane(name)[b, :, :G].view(np.uint16) ==
                        ref.plane(name)[b, :, :G].view(np.uint16)).all(), name
            for name in ("Kr", "Vr"):
                assert (oc.plane(name)[b, :, : nres[b]] == ref.plane(name)[b, :, : nres[b]]).all()


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def _cache(oracle_mod, B, Hq, H, D, bits, g, R, lens, seed=8, kscale=1.0):
    from oracle import OracleCache
    rng = np.random.default_rng(seed)
    S_max = max(lens)
    K = rand_f16(rng, (B, H, S_max, D), kscale)
    V = rand_f16(rng, (B, H, S_max, D))
    oc = OracleCache(B, Hq, H, D, bits, g, R, S_max)
    oc.quantize(K, V, lens)
    return oc, K, V


def test_zero_query_gives_mean_of_v_hat(oracle_mod):
    oc, K, V = _cache(oracle_mod, 2, 4, 2, 16, 2, 4, 4, [37, 9])
    q = np.zeros((2, 4, 16), np.float16)
    out = oc.attend(q)
    for b in range(2):
        for hq in range(4):
            _, v = np_dequant_sequence(oc, b, hq // 2)
            assert np.allclose(out[b, hq], v.mean(0).astype(np.float64), rtol=0, atol=1e-6)


def test_equal_keys_uniform_and_dominant_key(oracle_mod):
    from oracle import OracleCache
    rng = np.random.default_rng(9)
    B, H, D, g, R, S = 1, 1, 8, 4, 4, 30
    row = rand_f16(rng, D)
    K = np.broadcast_to(row, (B, H, S, D)).copy()
    V = rand_f16(rng, (B, H, S, D))
    oc = OracleCache(B, H, H, D, 4, g, R, S)
    oc.quantize(K, V, [S])
    q = rand_f16(rng, (B, H, D))
    _, v = np_dequant_sequence(oc, 0, 0)
    assert np.allclose(oc.attend(q)[0, 0], v.mean(0).astype(np.float64), atol=1e-6)
    # one residual key whose score exceeds every other by > 40
    K2 = rand_f16(rng, (B, H, S, D), 0.1)
    K2[0, 0, S - 2] = 0
    K2[0, 0, S - 2, 0] = 64.0
    oc2 = OracleCache(B, H, H, D, 2, g, R, S)
    oc2.quantize(K2, V, [S])
    q2 = np.zeros((B, H, D), np.float16)
    q2[0, 0, 0] = 8.0
    out = oc2.attend(q2, scale=1.0)
    assert np.allclose(out[0, 0], V[0, 0, S - 2].astype(np.float64), atol=1e-6)


@pytest.mark.parametrize("bits", [2, 4])
def test_brute_force_tiny(oracle_mod, bits):
    """Tiny inputs: dense softmax attention in long double over k_hat / v_hat
    rebuilt by an independent numpy unpacker equals the oracle to 1e-12."""
    for seed, lens in ((10, [64, 23, 5]), (11, [40, 41, 8])):
        B, Hq, H, D, g, R = 3, 4, 2, 8, 4, 8
        oc, K, V = _cache(oracle_mod, B, Hq, H, D, bits, g, R, lens, seed)
        rng = np.random.default_rng(seed + 100)
        q = rand_f16(rng, (B, Hq, D))
        scale = 0.37
        for b in range(B):
            for hq in range(Hq):
                k, v = np_dequant_sequence(oc, b, hq // 2)
                ref = np_dense_attention(q[b, hq].astype(np.longdouble), k, v,
                                         np.longdouble(scale))
                got = oc.attend_one(b, hq, q[b, hq], scale)
                assert np.abs(got - ref.astype(np.float64)).max() <= 1e-12


def test_gqa_head_mapping(oracle_mod):
    """Query head hq reads kv head hq // (H_q / H_kv) (contiguous groups)."""
    from oracle import OracleCache
    rng = np.random.default_rng(12)
    B, Hq, H, D, g, R, S = 1, 6, 3, 8, 4, 4, 12
    K = rand_f16(rng, (B, H, S, D))
    V = np.zeros((B, H, S, D), np.float16)
    for h in range(H):
        V[0, h] = np.float16(10 * (h + 1))       # kv head h -> constant 10(h+1)
    oc = OracleCache(B, Hq, H, D, 2, g, R, S)
    oc.quantize(K, V, [S])
    out = oc.attend(rand_f16(rng, (B, Hq, D)))
    for hq in range(Hq):
        assert np.allclose(out[0, hq], 10 * (hq // 2 + 1), atol=1e-5)


def test_empty_sequence(oracle_mod):
    oc, _, _ = _cache(oracle_mod, 2, 2, 2, 8, 2, 4, 4, [0, 9])
    out = oc.attend(np.ones((2, 2, 8), np.float16))
    assert (out[0] == 0).all()


def test_lse_combine_equals_one_pass():
    """The split-KV merge (max, rescaled sums) over any partition of the
    tokens equals a one-pass softmax to 1e-12 (pure arithmetic check of the
    combine step the kernels use)."""
    rng = np.random.default_rng(13)
    S, D = 300, 16
    s = rng.standard_normal(S) * 5
    V = rng.standard_normal((S, D))
    p = np.exp(s - s.max())
    ref = (p[:, None] * V).sum(0) / p.sum()
    for cuts in ([0, 300], [0, 1, 299, 300], [0, 77, 150, 151, 300]):
        parts = []
        for a, b in zip(cuts[:-1], cuts[1:]):
            m = s[a:b].max()
            e = np.exp(s[a:b] - m)
            parts.append((m, e.sum(), (e[:, None] * V[a:b]).sum(0)))
        M = max(m for m, _, _ in parts)
        L = sum(np.exp(m - M) * l for m, l, _ in parts)
        O = sum(np.exp(m - M) * o for m, _, o in parts)
        assert np.abs(O / L - ref).max() <= 1e-12


def test_large_scores_stay_finite(oracle_mod):
    """Scores near 1000 (exp overflows in double without the max shift):
    the result is still the exact softmax, here dominated by two residual
    tokens with equal scores, so out = the mean of their values."""
    from oracle import OracleCache
    rng = np.random.default_rng(14)
    B, H, D, g, R, S = 1, 1, 8, 4, 8, 20
    K = rand_f16(rng, (B, H, S, D), 0.1)
    V = rand_f16(rng, (B, H, S, D))
    for t in (S - 1, S - 3):
        K[0, 0, t] = 0
        K[0, 0, t, 0] = 31.25
    oc = OracleCache(B, H, H, D, 2, g, R, S)
    oc.quantize(K, V, [S])
    q = np.zeros((B, H, D), np.float16)
    q[0, 0, 0] = 32.0
    out = oc.attend(q, scale=1.0)                # top scores = 1000
    want = (V[0, 0, S - 1].astype(np.float64) + V[0, 0, S - 3]) / 2
    assert np.isfinite(out).all()
    assert np.allclose(out[0, 0], want, atol=1e-6)


def test_negative_zero_minimum_stored_as_positive_zero(oracle_mod):
    """A group whose minimum is -0.0 stores zero = +0.0 (bit pattern 0x0000);
    the codes are those of the same group with +0.0."""
    x = np.array([-0.0, 1.0, 2.0, 3.0], np.float32)
    codes, s32, s16, z16 = oracle_mod.quant_group(x, 2)
    assert z16 == 0x0000
    assert codes.tolist() == [0, 1, 2, 3]
    x2 = np.array([0.0, -0.0, 0.0, -0.0], np.float32)
    codes, s32, s16, z16 = oracle_mod.quant_group(x2, 2)
    assert z16 == 0x0000 and s16 == 0 and (codes == 0).all()


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_signed_zero_groups_in_either_order(oracle_mod, bits):
    """A group of zeros of mixed sign is a constant group: whatever the order
    of its elements, the stored scale and zero are both +0.0 (bit pattern
    0x0000) and every code is 0 -- the constant-group clause (scale 0, exact
    reconstruction) with signed zeros read as one value."""
    groups = [[-0.0, 0.0, 0.0, 0.0], [0.0, -0.0, 0.0, 0.0],
              [-0.0, -0.0, -0.0, -0.0], [0.0, 0.0, -0.0, -0.0],
              [-0.0, 0.0, -0.0, 0.0]]
    for x in groups:
        x = np.array(x, np.float32)
        assert np.signbit(x).any() or not np.signbit(x).any()
        codes, s32, s16, z16 = oracle_mod.quant_group(x, bits)
        assert (s16, z16) == (0x0000, 0x0000), x
        assert not np.signbit(np.float32(s32)), x
        assert (codes == 0).all()


def test_signed_zero_groups_through_the_cache(oracle_mod):
    """The same through the cache, on both axes: a key channel group (g
    tokens of one channel) and a value group (g channels of one token) made
    of +-0 in both orders store scale and zero 0x0000 with all-zero codes;
    the neighbouring groups are untouched by it."""
    from oracle import OracleCache
    rng = np.random.default_rng(15)
    B, H, D, g, R = 1, 1, 16, 4, 4
    S = 3 * g + R
    K = rand_f16(rng, (B, H, S, D))
    V = rand_f16(rng, (B, H, S, D))
    nz = np.array([-0.0, 0.0, 0.0, -0.0], np.float16)
    pz = np.array([0.0, -0.0, -0.0, 0.0], np.float16)
    K[0, 0, 0:g, 3] = nz            # key group 0, channel 3: -0 first
    K[0, 0, g:2 * g, 3] = pz        # key group 1, channel 3: +0 first
    V[0, 0, 5, 4:8] = nz            # token 5, value group 1
    V[0, 0, 6, 8:12] = pz           # token 6, value group 2
    oc = OracleCache(B, H, H, D, 2, g, R, S)
    oc.quantize(K, V, [S])
    assert oc.lengths()[1][0] == 3 * g
    ks, kz = oc.plane("Ks").view(np.uint16), oc.plane("Kz").view(np.uint16)
    vs, vz = oc.plane("Vs").view(np.uint16), oc.plane("Vz").view(np.uint16)
    for G in (0, 1):
        assert ks[0, 0, G, 3] == 0 and kz[0, 0, G, 3] == 0
        assert ks[0, 0, G, 2] != 0 and ks[0, 0, G, 4] != 0
    assert vs[0, 0, 5, 1] == 0 and vz[0, 0, 5, 1] == 0
    assert vs[0, 0, 6, 2] == 0 and vz[0, 0, 6, 2] == 0
    assert vs[0, 0, 5, 0] != 0 and vs[0, 0, 6, 1] != 0
    kc = np_unpack_rows(oc.plane("Kc")[0, 0, :3 * g], D, 2)
    vc = np_unpack_rows(oc.plane("Vc")[0, 0, :3 * g], D, 2)
    assert (kc[0:2 * g, 3] == 0).all()
    assert (vc[5, 4:8] == 0).all() and (vc[6, 8:12] == 0).all()


@pytest.mark.parametrize("bits,g", [(2, 4), (4, 8), (8, 4)])
def test_whole_cache_reconstruction_bound(oracle_mod, bits, g):
    """Every quantized element of a multi-sequence, multi-head ragged cache
    is within half a step of the input it came from, on the axes the method
    fixes: the key at (b, h, t, c) against the key group (t // g, c), the
    value at (b, h, t, c) against the value group (t, c // g).  With only the
    stored fp16 scale s16 at hand, the fp32 scale s32 it rounds from is
    within half an fp16 unit of it, so the bound is
    s16/2 + (2^b - 1 + 1/2) * u(s16), u = max(2^-11 s16, 2^-25) (the fp16
    subnormal spacing is 2^-24).  Positions are indexed here independently
    of the oracle, so a stride slip in the cache (wrong batch, head, token
    or channel offset) breaks the bound."""
    from oracle import OracleCache
    rng = np.random.default_rng(16 + bits)
    B, Hq, H, D, R = 3, 4, 2, 16, 5
    lens = [3 * g + R + 2, R + 1, 7 * g + R]
    S_max = max(lens) + 3
    K = rand_f16(rng, (B, H, S_max, D), 3.0)
    V = rand_f16(rng, (B, H, S_max, D), 0.5)
    K += (np.arange(B)[:, None, None, None] * 10 +
          np.arange(H)[None, :, None, None] * 4).astype(np.float16)
    oc = OracleCache(B, Hq, H, D, bits, g, R, S_max)
    oc.quantize(K, V, lens)
    _, Tq, _ = oc.lengths()
    P = (1 << bits) - 1
    checked = 0
    for b in range(B):
        for h in range(H):
            T = Tq[b]
            if T == 0:
                continue
            kc = np_unpack_rows(oc.plane("Kc")[b, h, :T], D, bits).astype(np.float64)
            vc = np_unpack_rows(oc.plane("Vc")[b, h, :T], D, bits).astype(np.float64)
            ks = oc.plane("Ks")[b, h, :T // g].astype(np.float64)[np.arange(T) // g]
            kz = oc.plane("Kz")[b, h, :T // g].astype(np.float64)[np.arange(T) // g]
            vs = oc.plane("Vs")[b, h, :T].astype(np.float64)[:, np.arange(D) // g]
            vz = oc.plane("Vz")[b, h, :T].astype(np.float64)[:, np.arange(D) // g]
            for code, s, z, x in ((kc, ks, kz, K[b, h, :T]), (vc, vs, vz, V[b, h, :T])):
                u = np.maximum(s * 2.0 ** -11, 2.0 ** -25)
                bound = s / 2 + (P + 0.5) * u + 1e-12
                err = np.abs(x.astype(np.float64) - (code * s + z))
                assert (err <= bound).all(), (b, h, err.max())
                checked += x.size
    assert checked > 0


# ---------------------------------------------------------------------------
# several query tokens per sequence (multi-query decode, chunked prefill)
# ---------------------------------------------------------------------------

def np_causal_attention(qs, K, V, scale, S):
    """Dense causal softmax attention in long double: query i of the newest
    S_q tokens sits at position S - S_q + i and sees tokens 0 ... that
    position."""
    S_q = qs.shape[0]
    out = []
    for i in range(S_q):
        pos = S - S_q + i
        out.append(np_dense_attention(qs[i], K[: pos + 1], V[: pos + 1], scale))
    return np.stack(out)


@pytest.mark.parametrize("bits", [2, 4])
def test_multi_query_brute_force_tiny(oracle_mod, bits):
    """Causal multi-query attention over k_hat / v_hat rebuilt by the
    independent numpy unpacker, in long double, equals the oracle to 1e-12;
    S_q spans the residual window and reaches into the quantized region."""
    B, Hq, H, D, g, R = 3, 4, 2, 8, 4, 6
    lens = [45, 17, 30]
    oc, K, V = _cache(oracle_mod, B, Hq, H, D, bits, g, R, lens, seed=20)
    rng = np.random.default_rng(120)
    for S_q in (1, 3, 12, 17):
        q = rand_f16(rng, (B, Hq, S_q, D))
        scale = 0.29
        got = oc.attend_multi(q, scale)
        for b in range(B):
            for hq in range(Hq):
                k, v = np_dequant_sequence(oc, b, hq // 2)
                ref = np_causal_attention(q[b, hq].astype(np.longdouble), k, v,
                                          np.longdouble(scale), lens[b])
                assert np.abs(got[b, hq] - ref.astype(np.float64)).max() <= 1e-6
                # the fp32 output is the double result rounded once
                assert np.abs(got[b, hq].astype(np.float64) -
                              ref.astype(np.float64)).max() <= \
                    1e-12 + 2.0 ** -24 * np.abs(ref.astype(np.float64)).max() * 2


def test_multi_query_reduces_to_decode_and_to_single_tokens(oracle_mod):
    """The last of S_q queries sees the whole sequence, as the one-query
    decode does; with S_q = S the first query sees token 0 alone, so its
    output is v_hat of token 0; S_q = 1 is the decode itself."""
    B, Hq, H, D, g, R = 2, 2, 1, 8, 4, 4
    lens = [23, 9]
    oc, K, V = _cache(oracle_mod, B, Hq, H, D, 2, g, R, lens, seed=21)
    rng = np.random.default_rng(121)
    q = rand_f16(rng, (B, Hq, 5, D))
    multi = oc.attend_multi(q)
    dec = oc.attend(np.ascontiguousarray(q[:, :, -1]))
    assert np.array_equal(multi[:, :, -1], dec)
    assert np.array_equal(oc.attend_multi(q[:, :, -1:])[:, :, 0], dec)
    qa = rand_f16(rng, (B, Hq, 9, D))
    oc9, _, _ = _cache(oracle_mod, B, Hq, H, D, 2, g, R, [9, 9], seed=22)
    out9 = oc9.attend_multi(qa)
    for b in range(B):
        _, v = np_dequant_sequence(oc9, b, 0)
        assert np.allclose(out9[b, :, 0], v[0].astype(np.float64), rtol=0, atol=1e-7)


def test_multi_query_rejects_more_queries_than_tokens(oracle_mod):
    oc, _, _ = _cache(oracle_mod, 2, 2, 2, 8, 2, 4, 4, [10, 3])
    with pytest.raises(ValueError):
        oc.attend_multi(np.zeros((2, 2, 4, 8), np.float16))


# ---------------------------------------------------------------------------
# KIVI-Sink: top key-norm tokens kept fp16, out of the groups' min/max
# (changelog v0.9.0 "New")
# ---------------------------------------------------------------------------

def _sink_cache(oracle_mod, n_sink, K, V, lens, Hq, bits=2, g=4, R=4):
    from oracle import OracleCache
    B, H, S_max, D = K.shape
    oc = OracleCache(B, Hq, H, D, bits, g, R, S_max, n_sink=n_sink)
    oc.quantize(K, V, lens)
    return oc


def test_sink_zero_is_plain_kivi_bit_for_bit(oracle_mod):
    """n_sink = 0 reproduces plain KIVI bit for bit (the pages' own
    invariant): every plane and the attention are identical."""
    from oracle import OracleCache
    rng = np.random.default_rng(30)
    B, Hq, H, D, g, R = 2, 4, 2, 16, 4, 6
    lens = [37, 22]
    K = rand_f16(rng, (B, H, 40, D), 3.0)
    V = rand_f16(rng, (B, H, 40, D))
    a = OracleCache(B, Hq, H, D, 2, g, R, 40)
    a.quantize(K, V, lens)
    b = _sink_cache(oracle_mod, 0, K, V, lens, Hq, 2, g, R)
    for name in ("Kc", "Ks", "Kz", "Vc", "Vs", "Vz", "Kr", "Vr"):
        assert np.array_equal(a.plane(name).view(np.uint8), b.plane(name).view(np.uint8)), name
    q = rand_f16(rng, (B, Hq, D))
    assert np.array_equal(a.attend(q), b.attend(q))


def test_sink_selection_by_key_norm(oracle_mod):
    """Sinks are the n_sink tokens with the largest key L2 norms, the
    earlier position first among equal norms, stored by ascending position
    with their exact fp16 rows."""
    rng = np.random.default_rng(31)
    B, H, D, S = 1, 2, 8, 30
    K = rand_f16(rng, (B, H, S, D), 0.1)
    V = rand_f16(rng, (B, H, S, D))
    # head 0: norms 4 at t = 20, 3 at t = 3 and t = 11 (a tie), 2 at t = 25
    for t, a in ((20, 4.0), (3, 3.0), (11, 3.0), (25, 2.0)):
        K[0, 0, t] = 0
        K[0, 0, t, 5] = a
    # head 1: one big key at t = 0
    K[0, 1, 0] = 10.0
    oc = _sink_cache(oracle_mod, 3, K, V, [S], Hq=2)
    pos = oc.plane("sink_pos")
    assert pos[0, 0].tolist() == [3, 11, 20]
    assert pos[0, 1][0] == 0 and len(set(pos[0, 1].tolist())) == 3
    for k, t in enumerate(pos[0, 0]):
        assert np.array_equal(oc.plane("sink_k")[0, 0, k], K[0, 0, t])
        assert np.array_equal(oc.plane("sink_v")[0, 0, k], V[0, 0, t])
    # fewer tokens than sinks: every token is a sink
    oc2 = _sink_cache(oracle_mod, 3, K[:, :, :2].copy(), V[:, :, :2].copy(), [2], Hq=2)
    assert oc2.plane("sink_pos")[0, 0].tolist() == [0, 1, -1]


def test_sink_is_left_out_of_its_groups(oracle_mod):
    """The sink's key group is quantized from the other g - 1 tokens alone
    (the group quantizer on the reduced group gives the same scale, zero and
    codes), the sink's code is 0, and its own value groups are empty
    (scale and zero +0, codes 0)."""
    rng = np.random.default_rng(32)
    B, H, D, g, R, S = 1, 1, 8, 4, 4, 20
    K = rand_f16(rng, (B, H, S, D))
    V = rand_f16(rng, (B, H, S, D))
    K[0, 0, 6] = 50.0                     # token 6 (key group 1) is the sink
    oc = _sink_cache(oracle_mod, 1, K, V, [S], Hq=1, bits=2, g=g, R=R)
    assert oc.plane("sink_pos")[0, 0].tolist() == [6]
    Ks = oc.plane("Ks")[0, 0].view(np.uint16)
    Kz = oc.plane("Kz")[0, 0].view(np.uint16)
    kc = np_unpack_rows(oc.plane("Kc")[0, 0], D, 2)
    others = [4, 5, 7]
    for ch in range(D):
        codes, _, s16, z16 = oracle_mod.quant_group(
            K[0, 0, others, ch].astype(np.float32), 2)
        assert (Ks[1, ch], Kz[1, ch]) == (s16, z16)
        assert kc[others, ch].tolist() == codes.tolist()
        assert kc[6, ch] == 0
    assert (oc.plane("Vs")[0, 0, 6].view(np.uint16) == 0).all()
    assert (oc.plane("Vz")[0, 0, 6].view(np.uint16) == 0).all()
    assert (np_unpack_rows(oc.plane("Vc")[0, 0], D, 2)[6] == 0).all()


def np_dequant_sinks(oc, b, h):
    """k_hat, v_hat [S][D] in long double, sink tokens of the quantized
    region from the sink rows."""
    k, v = np_dequant_sequence(oc, b, h)
    _, Tq, _ = oc.lengths()
    for slot, t in enumerate(oc.plane("sink_pos")[b, h]):
        if 0 <= t < Tq[b]:
            k[t] = oc.plane("sink_k")[b, h, slot].astype(np.longdouble)
            v[t] = oc.plane("sink_v")[b, h, slot].astype(np.longdouble)
    return k, v


@pytest.mark.parametrize("bits", [2, 4])
def test_sink_attention_brute_force(oracle_mod, bits):
    """Attention with sinks: long-double dense softmax over k_hat / v_hat
    rebuilt independently (sink rows exact) equals the oracle to 1e-12, for
    one query and for causal multi-query attention."""
    rng = np.random.default_rng(33 + bits)
    B, Hq, H, D, g, R = 2, 4, 2, 8, 4, 5
    lens = [41, 19]
    K = rand_f16(rng, (B, H, 45, D))
    V = rand_f16(rng, (B, H, 45, D))
    K[0, 0, 2] *= 20
    K[0, 1, 30] *= 15
    K[1, 0, 9] *= 30
    oc = _sink_cache(oracle_mod, 3, K, V, lens, Hq, bits=bits, g=g, R=R)
    q = rand_f16(rng, (B, Hq, D))
    out = oc.attend(q, 0.4)
    q4 = rand_f16(rng, (B, Hq, 6, D))
    outm = oc.attend_multi(q4, 0.4)
    for b in range(B):
        for hq in range(Hq):
            k, v = np_dequant_sinks(oc, b, hq // 2)
            ref = np_dense_attention(q[b, hq].astype(np.longdouble), k, v, np.longdouble(0.4))
            assert np.abs(oc.attend_one(b, hq, q[b, hq], 0.4) - ref.astype(np.float64)).max() <= 1e-12
            assert np.abs(out[b, hq] - ref.astype(np.float64)).max() <= 1e-6
            refm = np_causal_attention(q4[b, hq].astype(np.longdouble), k, v,
                                       np.longdouble(0.4), lens[b])
            assert np.abs(outm[b, hq] - refm.astype(np.float64)).max() <= 1e-6


def test_sink_protection_lowers_group_error(oracle_mod):
    """An outlier key inflates its group's scale under plain KIVI; with it
    kept as a sink, the other tokens of its groups reconstruct with a lower
    error (the pages' 'MSE improvement over plain KIVI')."""
    rng = np.random.default_rng(34)
    B, H, D, g, R, S = 1, 1, 16, 8, 8, 40
    K = rand_f16(rng, (B, H, S, D))
    V = rand_f16(rng, (B, H, S, D))
    K[0, 0, 3] = 40.0
    plain = _sink_cache(oracle_mod, 0, K, V, [S], Hq=1, g=g, R=R)
    sunk = _sink_cache(oracle_mod, 1, K, V, [S], Hq=1, g=g, R=R)
    kp, _ = np_dequant_sequence(plain, 0, 0)
    ks, _ = np_dequant_sinks(sunk, 0, 0)
    others = [t for t in range(g) if t != 3]
    x = K[0, 0, others].astype(np.float64)
    e_plain = ((kp[others].astype(np.float64) - x) ** 2).mean()
    e_sink = ((ks[others].astype(np.float64) - x) ** 2).mean()
    assert e_sink < 0.1 * e_plain
    assert np.array_equal(ks[3].astype(np.float64), K[0, 0, 3].astype(np.float64))


def test_sink_in_the_window_is_left_out_when_flushed(oracle_mod):
    """Sinks are chosen at prefill; a sink still in the fp16 window is left
    out of its group's min/max when a later append flushes the group, and
    appended tokens never become sinks."""
    from oracle import OracleCache
    rng = np.random.default_rng(35)
    B, H, D, g, R = 1, 1, 8, 4, 4
    K = rand_f16(rng, (B, H, 30, D))
    V = rand_f16(rng, (B, H, 30, D))
    K[0, 0, 9] = 30.0                  # in the window after a 10-token prefill
    oc = OracleCache(B, 1, H, D, 2, g, R, 30, n_sink=1)
    oc.quantize(K, V, [10])
    assert oc.lengths()[1][0] == 4 and oc.plane("sink_pos")[0, 0].tolist() == [9]
    Kn = K[:, :, 10:].copy()
    Kn[0, 0, 5] = 99.0                 # a larger key among the appended ones
    oc.append(Kn, V[:, :, 10:].copy(), [20])
    assert oc.plane("sink_pos")[0, 0].tolist() == [9]
    # group 2 (tokens 8 ... 11) was quantized without token 9
    Ks = oc.plane("Ks")[0, 0].view(np.uint16)
    for ch in range(D):
        _, _, s16, _ = oracle_mod.quant_group(K[0, 0, [8, 10, 11], ch].astype(np.float32), 2)
        assert Ks[2, ch] == s16


# ---------------------------------------------------------------------------
# Kitty: per key group, the kitty_hi channels of largest running variance in
# 4 bits, the rest in 2 bits; values in fp16 (changelog v0.11.0 "New")
# ---------------------------------------------------------------------------

def np_kitty_keys(oc, b, h):
    """k_hat [Tq][D] in long double from the Kitty planes: per token row the
    4-bit channels' codes in ascending channel order, then the 2-bit ones,
    LSB first; the group's mask marks the 4-bit channels."""
    _, Tq, _ = oc.lengths()
    D, g = oc.D, oc.group
    kc = oc.plane("Kc")[b, h]
    masks = oc.plane("Kmask")[b, h]
    Ks = oc.plane("Ks")[b, h].astype(np.longdouble)
    Kz = oc.plane("Kz")[b, h].astype(np.longdouble)
    out = np.zeros((Tq[b], D), np.longdouble)
    for t in range(Tq[b]):
        G = t // g
        hi = [(int(masks[G, c // 32]) >> (c % 32)) & 1 for c in range(D)]
        bits = "".join(format(int(x), "08b")[::-1] for x in kc[t])   # LSB first
        pos = 0
        for want in (1, 0):
            for c in range(D):
                if hi[c] != want:
                    continue
                w = 4 if want else 2
                code = int(bits[pos:pos + w][::-1], 2)
                pos += w
                out[t, c] = code * Ks[G, c] + Kz[G, c]
    return out


def _kitty(oracle_mod, hi, K, V, lens, Hq=None, g=8, R=8):
    from oracle import OracleCache
    B, H, S_max, D = K.shape
    oc = OracleCache(B, Hq or H, H, D, 2, g, R, S_max, kitty_hi=hi)
    oc.quantize(K, V, lens)
    return oc


def test_kitty_ranks_channels_by_variance(oracle_mod):
    """Channel c alternates +a_c / -a_c inside every key group, so its
    running variance is a_c^2: the 4-bit channels are the hi largest a_c,
    the smaller channel index first among equal a_c."""
    B, H, D, g = 1, 1, 32, 8
    S = 5 * g + 8
    # the 8th place is a tie between channels 2 and 4 (a = 2): channel 2 wins
    a = np.array([1, 7, 2, 7, 2, 9, 4, 0.5, 6, 5, 8, 1.5] + [0.25] * 20, np.float64)
    sign = np.where(np.arange(S) % 2 == 0, 1.0, -1.0)
    K = (sign[:, None] * a[None, :]).astype(np.float16)[None, None]
    V = np.zeros_like(K)
    oc = _kitty(oracle_mod, 8, K, V, [S], g=g, R=8)
    want = sorted(range(D), key=lambda c: (-a[c], c))[:8]
    mask = oc.plane("Kmask")[0, 0]
    for G in range(oc.lengths()[1][0] // g):
        got = [c for c in range(D) if (int(mask[G, c // 32]) >> (c % 32)) & 1]
        assert got == sorted(want), G


def test_kitty_hi_zero_and_all_reduce_to_kivi_keys(oracle_mod):
    """kitty_hi = 0 quantizes every key channel in 2 bits and kitty_hi = D
    every one in 4 bits: the key codes, scales and zeros are then those of a
    plain KIVI cache of that width (same packing), and the values are the
    fp16 inputs unchanged."""
    from oracle import OracleCache
    rng = np.random.default_rng(40)
    B, H, D, g, R = 2, 2, 32, 8, 8
    lens = [60, 35]
    K = rand_f16(rng, (B, H, 64, D), 2.0)
    V = rand_f16(rng, (B, H, 64, D))
    for hi, bits in ((0, 2), (D, 4)):
        kt = _kitty(oracle_mod, hi, K, V, lens, g=g, R=R)
        kv = OracleCache(B, H, H, D, bits, g, R, 64)
        kv.quantize(K, V, lens)
        _, Tq, _ = kv.lengths()
        for b in range(B):
            for name in ("Kc", "Ks", "Kz"):
                assert np.array_equal(kt.plane(name)[b, :, :Tq[b] // (g if name != "Kc" else 1)].view(np.uint8),
                                      kv.plane(name)[b, :, :Tq[b] // (g if name != "Kc" else 1)].view(np.uint8)), (hi, name)
            assert np.array_equal(kt.plane("Vf")[b, :, :Tq[b]], V[b, :, :Tq[b]])


def test_kitty_hi_channels_err_less_and_beat_uniform_2bit(oracle_mod):
    """Each channel reconstructs within half its step: (max-min)/15 for the
    4-bit channels, /3 for the 2-bit ones; on keys whose variance sits in a
    quarter of the channels, Kitty's key error is well below uniform 2-bit
    KIVI's."""
    from oracle import OracleCache
    rng = np.random.default_rng(41)
    B, H, D, g, R, S = 1, 1, 64, 16, 16, 96
    scale = np.ones(D)
    scale[rng.permutation(D)[:16]] = 12.0
    K = (rng.standard_normal((B, H, S, D)) * scale).astype(np.float16)
    V = rand_f16(rng, (B, H, S, D))
    oc = _kitty(oracle_mod, 16, K, V, [S], g=g, R=R)
    k = np_kitty_keys(oc, 0, 0).astype(np.float64)
    Tq = oc.lengths()[1][0]
    x = K[0, 0, :Tq].astype(np.float64)
    mask = oc.plane("Kmask")[0, 0]
    for G in range(Tq // g):
        rows = slice(G * g, (G + 1) * g)
        rng_c = x[rows].max(0) - x[rows].min(0)
        for c in range(D):
            hi = (int(mask[G, c // 32]) >> (c % 32)) & 1
            step = rng_c[c] / (15 if hi else 3)
            assert np.abs(k[rows, c] - x[rows, c]).max() <= step / 2 * (1 + 1e-3) + 2.0 ** -20
    kv = OracleCache(B, H, H, D, 2, g, R, S)
    kv.quantize(K, V, [S])
    k2, _ = np_dequant_sequence(kv, 0, 0)
    e_kitty = ((k - x) ** 2).mean()
    e_kivi = ((k2[:Tq].astype(np.float64) - x) ** 2).mean()
    assert e_kitty < 0.3 * e_kivi


def test_kitty_prefill_equals_appends(oracle_mod):
    """The ranking of a group uses the running sums up to that group's last
    token, so prefill and any chunking of appends give the same cache, bit
    for bit."""
    from oracle import OracleCache
    rng = np.random.default_rng(42)
    B, H, D, g, R = 2, 1, 32, 8, 5
    S_final = [70, 41]
    K = rand_f16(rng, (B, H, 72, D), 3.0)
    V = rand_f16(rng, (B, H, 72, D))
    ref = _kitty(oracle_mod, 8, K, V, S_final, g=g, R=R)
    oc = OracleCache(B, H, H, D, 2, g, R, 72, kitty_hi=8)
    oc.quantize(K, V, [3, 3])
    cur = [3, 3]
    step = 0
    while cur != S_final:
        n = [min([1, 9, 4][(step + b) % 3], S_final[b] - cur[b]) for b in range(B)]
        Kn = np.zeros((B, H, max(n), D), np.float16)
        Vn = np.zeros_like(Kn)
        for b in range(B):
            Kn[b, :, :n[b]] = K[b, :, cur[b]:cur[b] + n[b]]
            Vn[b, :, :n[b]] = V[b, :, cur[b]:cur[b] + n[b]]
        oc.append(Kn, Vn, n)
        cur = [c + x for c, x in zip(cur, n)]
        step += 1
    _, Tq, _ = ref.lengths()
    for b in range(B):
        for name in ("Kc", "Ks", "Kz", "Kmask", "Vf"):
            n = Tq[b] // g if name in ("Ks", "Kz", "Kmask") else Tq[b]
            assert np.array_equal(oc.plane(name)[b, :, :n].view(np.uint8),
                                  ref.plane(name)[b, :, :n].view(np.uint8)), name


def test_kitty_attention_brute_force(oracle_mod):
    """Attention over Kitty keys (independent unpacker) and exact fp16
    values, long double, equals the oracle to 1e-12 (one query; causal
    multi-query to 1e-6)."""
    rng = np.random.default_rng(43)
    B, Hq, H, D, g, R = 2, 4, 2, 32, 8, 6
    lens = [53, 30]
    K = rand_f16(rng, (B, H, 56, D), 2.0)
    V = rand_f16(rng, (B, H, 56, D))
    oc = _kitty(oracle_mod, 8, K, V, lens, Hq=Hq, g=g, R=R)
    q = rand_f16(rng, (B, Hq, D))
    q3 = rand_f16(rng, (B, Hq, 3, D))
    outm = oc.attend_multi(q3, 0.3)
    _, Tq, nres = oc.lengths()
    for b in range(B):
        for hq in range(Hq):
            h = hq // 2
            kq = np_kitty_keys(oc, b, h)
            kr = oc.plane("Kr")[b, h, :nres[b]].astype(np.longdouble)
            vq = oc.plane("Vf")[b, h, :Tq[b]].astype(np.longdouble)
            vr = oc.plane("Vr")[b, h, :nres[b]].astype(np.longdouble)
            k = np.concatenate([kq, kr])
            v = np.concatenate([vq, vr])
            ref = np_dense_attention(q[b, hq].astype(np.longdouble), k, v, np.longdouble(0.3))
            assert np.abs(oc.attend_one(b, hq, q[b, hq], 0.3) - ref.astype(np.float64)).max() <= 1e-12
            refm = np_causal_attention(q3[b, hq].astype(np.longdouble), k, v,
                                       np.longdouble(0.3), lens[b])
            assert np.abs(outm[b, hq] - refm.astype(np.float64)).max() <= 1e-6


# ---------------------------------------------------------------------------
# AgeTieredKV: three widths by token age (method overview, AgeTieredKV)
# ---------------------------------------------------------------------------

def np_age_hat(oc, b, h):
    """k_hat, v_hat [Tq][D] in long double from the age-tiered planes: each
    group's codes at its tier's width in the leading bytes of a D-byte
    row."""
    _, Tq, _ = oc.lengths()
    D, g = oc.D, oc.group
    b1, b2, *widths = oc.age
    tiers = oc.plane("tier")[b, h]
    k = np.zeros((Tq[b], D), np.longdouble)
    v = np.zeros((Tq[b], D), np.longdouble)
    Ks = oc.plane("Ks")[b, h].astype(np.longdouble)
    Kz = oc.plane("Kz")[b, h].astype(np.longdouble)
    Vs = oc.plane("Vs")[b, h].astype(np.longdouble)
    Vz = oc.plane("Vz")[b, h].astype(np.longdouble)
    for G in range(Tq[b] // g):
        w = widths[tiers[G]]
        rows = slice(G * g, (G + 1) * g)
        kc = np_unpack_rows(oc.plane("Kc")[b, h, rows, : D * w // 8], D, w)
        vc = np_unpack_rows(oc.plane("Vc")[b, h, rows, : D * w // 8], D, w)
        k[rows] = kc * Ks[G] + Kz[G]
        v[rows] = vc * Vs[rows][:, np.arange(D) // g] + Vz[rows][:, np.arange(D) // g]
    return k, v


def _age(oracle_mod, age, K, V, lens, Hq=None, g=8, R=0):
    from oracle import OracleCache
    B, H, S_max, D = K.shape
    oc = OracleCache(B, Hq or H, H, D, 8, g, R, S_max, age=age)
    oc.quantize(K, V, lens)
    return oc


def test_age_tiers_follow_the_age_rule(oracle_mod):
    """A group's tier: 0 while fewer than b1 tokens are newer than its last
    token, 1 while fewer than b2, else 2."""
    rng = np.random.default_rng(50)
    B, H, D, g = 2, 1, 16, 8
    lens = [123, 60]
    K = rand_f16(rng, (B, H, 128, D))
    V = rand_f16(rng, (B, H, 128, D))
    oc = _age(oracle_mod, (16, 48, 8, 4, 2), K, V, lens, g=g)
    _, Tq, _ = oc.lengths()
    for b in range(B):
        for G in range(Tq[b] // g):
            age = lens[b] - (G + 1) * g
            want = 0 if age < 16 else (1 if age < 48 else 2)
            assert oc.plane("tier")[b, 0, G] == want, (b, G)


@pytest.mark.parametrize("w", [8, 4, 2])
def test_age_without_demotion_is_kivi(oracle_mod, w):
    """While no group is old enough to move (boundaries beyond the
    sequence), the age-tiered cache holds plain KIVI codes at the top
    tier's width, scales and zeros bit for bit."""
    from oracle import OracleCache
    rng = np.random.default_rng(51)
    B, H, D, g, R = 2, 2, 16, 8, 4
    lens = [70, 33]
    K = rand_f16(rng, (B, H, 72, D), 2.0)
    V = rand_f16(rng, (B, H, 72, D))
    oa = _age(oracle_mod, (1024, 2048, w, 2, 2), K, V, lens, g=g, R=R)
    ok = OracleCache(B, H, H, D, w, g, R, 72)
    ok.quantize(K, V, lens)
    _, Tq, _ = ok.lengths()
    for b in range(B):
        T = Tq[b]
        assert np.array_equal(oa.plane("Kc")[b, :, :T, : D * w // 8], ok.plane("Kc")[b, :, :T])
        assert np.array_equal(oa.plane("Vc")[b, :, :T, : D * w // 8], ok.plane("Vc")[b, :, :T])
        assert (oa.plane("Kc")[b, :, :T, D * w // 8:] == 0).all()
        for name in ("Ks", "Kz"):
            assert np.array_equal(oa.plane(name)[b, :, : T // g].view(np.uint16),
                                  ok.plane(name)[b, :, : T // g].view(np.uint16))
        for name in ("Vs", "Vz"):
            assert np.array_equal(oa.plane(name)[b, :, :T].view(np.uint16),
                                  ok.plane(name)[b, :, :T].view(np.uint16))


def test_age_demotion_requantizes_the_rebuilt_values(oracle_mod):
    """A group that moved 8 -> 4 bits holds the group quantizer's result on
    its 8-bit values rebuilt in fp32 (code * scale rounded, then + zero
    rounded), the keys per channel and the values per token: checked against
    an independent numpy rebuild and the (pinned) quantizer."""
    rng = np.random.default_rng(52)
    B, H, D, g = 1, 1, 16, 8
    S = 40
    K = rand_f16(rng, (B, H, S, D), 3.0)
    V = rand_f16(rng, (B, H, S, D))
    o8 = _age(oracle_mod, (1024, 2048, 8, 4, 2), K, V, [S], g=g)   # no demotion
    o4 = _age(oracle_mod, (8, 2048, 8, 4, 2), K, V, [S], g=g)      # groups 0..3 -> 4 bits
    assert o4.plane("tier")[0, 0].tolist()[:5] == [1, 1, 1, 1, 0]
    f32 = np.float32
    for G in range(4):
        rows = slice(G * g, (G + 1) * g)
        kc8 = np_unpack_rows(o8.plane("Kc")[0, 0, rows], D, 8).astype(f32)
        ks8 = o8.plane("Ks")[0, 0, G].astype(f32)
        kz8 = o8.plane("Kz")[0, 0, G].astype(f32)
        xk = (kc8 * ks8).astype(f32) + kz8                       # two roundings
        kc4 = np_unpack_rows(o4.plane("Kc")[0, 0, rows, : D // 2], D, 4)
        for ch in range(D):
            codes, _, s16, z16 = oracle_mod.quant_group(xk[:, ch].astype(f32), 4)
            assert kc4[:, ch].tolist() == codes.tolist()
            assert o4.plane("Ks")[0, 0, G, ch].view(np.uint16) == s16
            assert o4.plane("Kz")[0, 0, G, ch].view(np.uint16) == z16
        vc8 = np_unpack_rows(o8.plane("Vc")[0, 0, rows], D, 8).astype(f32)
        vs8 = o8.plane("Vs")[0, 0, rows].astype(f32)[:, np.arange(D) // g]
        vz8 = o8.plane("Vz")[0, 0, rows].astype(f32)[:, np.arange(D) // g]
        xv = (vc8 * vs8).astype(f32) + vz8
        vc4 = np_unpack_rows(o4.plane("Vc")[0, 0, rows, : D // 2], D, 4)
        for i in range(g):
            for j in range(D // g):
                codes, _, s16, _ = oracle_mod.quant_group(xv[i, j * g:(j + 1) * g], 4)
                assert vc4[i, j * g:(j + 1) * g].tolist() == codes.tolist()
                assert o4.plane("Vs")[0, 0, G * g + i, j].view(np.uint16) == s16


def test_age_prefill_equals_appends(oracle_mod):
    """A group always passes the tiers in order, one at a time, so a prefill
    and any chunking of appends reach the same cache, bit for bit."""
    from oracle import OracleCache
    rng = np.random.default_rng(53)
    B, H, D, g, R = 2, 1, 16, 8, 3
    S_final = [150, 61]
    K = rand_f16(rng, (B, H, 152, D), 2.0)
    V = rand_f16(rng, (B, H, 152, D))
    age = (16, 64, 8, 4, 2)
    ref = _age(oracle_mod, age, K, V, S_final, g=g, R=R)
    oc = OracleCache(B, H, H, D, 8, g, R, 152, age=age)
    oc.quantize(K, V, [2, 2])
    cur = [2, 2]
    step = 0
    while cur != S_final:
        n = [min([1, 13, 40, 5][(step + b) % 4], S_final[b] - cur[b]) for b in range(B)]
        Kn = np.zeros((B, H, max(n), D), np.float16)
        Vn = np.zeros_like(Kn)
        for b in range(B):
            Kn[b, :, :n[b]] = K[b, :, cur[b]:cur[b] + n[b]]
            Vn[b, :, :n[b]] = V[b, :, cur[b]:cur[b] + n[b]]
        oc.append(Kn, Vn, n)
        cur = [c + x for c, x in zip(cur, n)]
        step += 1
    _, Tq, _ = ref.lengths()
    for b in range(B):
        T = Tq[b]
        for name, n in (("Kc", T), ("Vc", T), ("Ks", T // g), ("Kz", T // g),
                        ("Vs", T), ("Vz", T), ("tier", T // g)):
            assert np.array_equal(oc.plane(name)[b, :, :n].view(np.uint8),
                                  ref.plane(name)[b, :, :n].view(np.uint8)), name


def test_age_attention_brute_force_and_error_grows_with_age(oracle_mod):
    """Attention over k_hat / v_hat rebuilt at each group's width (long
    double) equals the oracle to 1e-12; and old (2-bit) groups reconstruct
    the inputs with a larger error than recent (8-bit) ones."""
    rng = np.random.default_rng(54)
    B, Hq, H, D, g, R = 1, 2, 1, 16, 8, 0
    S = 200
    K = rand_f16(rng, (B, H, S, D))
    V = rand_f16(rng, (B, H, S, D))
    oc = _age(oracle_mod, (32, 96, 8, 4, 2), K, V, [S], Hq=Hq, g=g, R=R)
    q = rand_f16(rng, (B, Hq, D))
    k, v = np_age_hat(oc, 0, 0)
    _, Tq, nres = oc.lengths()
    kr = oc.plane("Kr")[0, 0, :nres[0]].astype(np.longdouble)
    vr = oc.plane("Vr")[0, 0, :nres[0]].astype(np.longdouble)
    kk = np.concatenate([k, kr])
    vv = np.concatenate([v, vr])
    for hq in range(Hq):
        ref = np_dense_attention(q[0, hq].astype(np.longdouble), kk, vv, np.longdouble(0.25))
        assert np.abs(oc.attend_one(0, hq, q[0, hq], 0.25) - ref.astype(np.float64)).max() <= 1e-12
    tiers = oc.plane("tier")[0, 0, : Tq[0] // g]
    err = np.abs(k.astype(np.float64) - K[0, 0, : Tq[0]].astype(np.float64))
    per_group = err.reshape(-1, g, D).mean(axis=(1, 2))
    assert per_group[tiers == 2].mean() > 4 * per_group[tiers == 0].mean()
    assert {0, 1, 2} <= set(tiers.tolist())


def test_prefix_attention_reduces_to_decode_and_multi(oracle_mod):
    """A query attending the prefix that ends at the last token is the
    one-query decode, bit for bit; prefixes ending earlier are the causal
    multi-query outputs of those positions."""
    B, Hq, H, D, g, R = 2, 4, 2, 8, 4, 5
    lens = [33, 12]
    oc, K, V = _cache(oracle_mod, B, Hq, H, D, 2, g, R, lens, seed=23)
    rng = np.random.default_rng(123)
    q = rand_f16(rng, (B, Hq, D))
    dec = oc.attend(q)
    q3 = np.ascontiguousarray(np.repeat(q[:, :, None], 3, axis=2))
    multi = oc.attend_multi(q3)
    for b in range(B):
        for hq in range(Hq):
            full = oc.attend_prefix(b, hq, q[b, hq], lens[b] - 1)
            assert np.array_equal(full.astype(np.float32), dec[b, hq])
            for i in range(3):
                pre = oc.attend_prefix(b, hq, q[b, hq], lens[b] - 3 + i)
                assert np.array_equal(pre.astype(np.float32), multi[b, hq, i])
    with pytest.raises(ValueError):
        oc.attend_prefix(1, 0, q[1, 0], lens[1])
