"""Several query tokens per sequence (multi-token decode, chunked prefill
attend) on the tensor cores, element by element against the oracle's causal
multi-query attention on the same seeded inputs: |gpu - oracle| <= 1e-3 +
1e-3 |oracle| for every output.

The queries of a sequence are its newest S_q tokens, already in the cache
(query i at position S - S_q + i, attending tokens up to its own position).
Cases span several 128-row query tiles, several 64-token key tiles with a
ragged tail, the quantized region, the fp16 residual window, GQA, 2/4/8-bit
caches (fragment-order and packed code planes) and a chunk appended just
before it is attended.

Method: attention over the group-affine cache of VeloxQuant-MLX changelog
v0.42.0 "Added"; the causal S_q > 1 form after the prefill companion of
changelog v0.40.0 "Added".
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
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    d = np.abs(got - ref)
    assert np.isfinite(got).all(), what
    bad = d > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {bad.sum()} outputs off, max abs diff "
                           f"{d.max():.3e}")


def _pair(w, seed):
    import oracle
    from bit_kv_cache_05_gb300.cache import KiviCache
    inp = synth.make_inputs(w, seed=seed, device="cpu")
    c = KiviCache(inp["K"].cuda(), inp["V"].cuda(), w.seq_lens, H_q=w.H_q,
                  bits=w.bits, group=w.group, residual=w.residual,
                  max_seq=w.max_seq)
    oc = oracle.OracleCache(w.B, w.H_q, w.H_kv, w.D, w.bits, w.group,
                            w.residual, w.max_seq)
    oc.quantize(inp["K"].numpy(), inp["V"].numpy(), w.seq_lens)
    return c, oc


CASES = [
    # (workload recipe, lengths, S_q values)
    ("tiny", [256], (1, 5, 40, 129)),
    ("pages_S512", [700, 333], (3, 64, 200)),
    ("gqa_serving", [900, 260, 517], (1, 7, 33, 70, 100)),   # 70: 3 tiles of 32
    ("int4_append", [1000, 450], (2, 65, 130)),
]


@pytest.mark.parametrize("name,lens,sqs", CASES, ids=[c[0] for c in CASES])
def test_multi_query_matches_oracle(lib, name, lens, sqs):
    w = synth.shrink(synth.workload(name), lens, n_append=0)
    c, oc = _pair(w, seed=41)
    g = torch.Generator().manual_seed(7)
    for S_q in sqs:
        q = (torch.randn(w.B, w.H_q, S_q, w.D, generator=g)).half()
        got = c.attend_multi(q.cuda())
        torch.cuda.synchronize()
        ref = oc.attend_multi(q.numpy())
        _close(got.cpu().numpy(), ref, f"{name} S_q={S_q}")
    c.device_status()
    c.close()


@pytest.mark.parametrize("bits,g", [(8, 32), (4, 32)])
def test_multi_query_other_code_orders(lib, bits, g):
    """8-bit caches keep packed code planes; 4-bit with g = 32 too."""
    w = synth.Workload("m", 2, 8, 4, 128, bits, g, 32, [300, 650])
    c, oc = _pair(w, seed=43)
    q = torch.randn(w.B, w.H_q, 37, w.D, generator=torch.Generator().manual_seed(3)).half()
    got = c.attend_multi(q.cuda())
    torch.cuda.synchronize()
    _close(got.cpu().numpy(), oc.attend_multi(q.numpy()), f"bits={bits}")
    c.close()


def test_chunk_appended_then_attended(lib):
    """Chunked prefill: append n tokens to every sequence (flushing groups),
    then attend them as S_q = n queries."""
    w = synth.shrink(synth.workload("gqa_serving"), [600, 211], n_append=0)
    w.seq_lens = [600, 211]
    import oracle
    from bit_kv_cache_05_gb300.cache import KiviCache
    inp = synth.make_inputs(w, seed=44, device="cpu")
    n = 150
    gk = torch.Generator().manual_seed(11)
    Kn = torch.randn(w.B, w.H_kv, n, w.D, generator=gk).half()
    Vn = torch.randn(w.B, w.H_kv, n, w.D, generator=gk).half()
    q = torch.randn(w.B, w.H_q, n, w.D, generator=gk).half()
    c = KiviCache(inp["K"].cuda(), inp["V"].cuda(), w.seq_lens, H_q=w.H_q,
                  bits=w.bits, group=w.group, residual=w.residual,
                  max_seq=max(w.seq_lens) + n)
    c.append(Kn.cuda(), Vn.cuda(), [n] * w.B)
    got = c.attend_multi(q.cuda())
    torch.cuda.synchronize()
    oc = oracle.OracleCache(w.B, w.H_q, w.H_kv, w.D, w.bits, w.group,
                            w.residual, max(w.seq_lens) + n)
    oc.quantize(inp["K"].numpy(), inp["V"].numpy(), w.seq_lens)
    oc.append(Kn.numpy(), Vn.numpy(), [n] * w.B)
    _close(got.cpu().numpy(), oc.attend_multi(q.numpy()), "appended chunk")
    c.close()


@pytest.mark.parametrize("split_tokens", [256, 640])
def test_key_ranges_match_the_oracle(lib, split_tokens):
    """Key ranges per query tile (forced through the split hook): partial
    rows merged by the combine kernel, the same result within tolerance;
    ranges that lie wholly past some rows' own tokens leave those rows
    empty partials."""
    from bit_kv_cache_05_gb300 import _lib
    w = synth.shrink(synth.workload("gqa_serving"), [900, 260, 517], n_append=0)
    c, oc = _pair(w, seed=46)
    _lib.check(lib.vq_kivi_set_split_tokens(c._h, split_tokens))
    g = torch.Generator().manual_seed(8)
    for S_q in (40, 200):
        q = (torch.randn(w.B, w.H_q, S_q, w.D, generator=g)).half()
        got = c.attend_multi(q.cuda())
        torch.cuda.synchronize()
        _close(got.cpu().numpy(), oc.attend_multi(q.numpy()),
               f"split_tokens={split_tokens} S_q={S_q}")
    c.device_status()
    c.close()


def test_one_query_equals_the_decode(lib):
    w = synth.shrink(synth.workload("pages_S512"), [512], n_append=0)
    c, _ = _pair(w, seed=45)
    q = torch.randn(1, 32, 128, generator=torch.Generator().manual_seed(5)).half().cuda()
    dec = c.decode_attend(q)
    mq = c.attend_multi(q.view(1, 32, 1, 128).contiguous())
    torch.cuda.synchronize()
    _close(mq.view(1, 32, 128).cpu().numpy(), dec.cpu().numpy(), "S_q=1")
    c.close()


def test_more_queries_than_tokens_is_an_argument_error(lib):
    from bit_kv_cache_05_gb300 import _lib
    w = synth.shrink(synth.workload("tiny"), [10, 3], n_append=0)
    c, _ = _pair(w, seed=46)
    with pytest.raises(_lib.VqError) as ei:
        c.attend_multi(torch.zeros(2, 4, 4, 64, dtype=torch.float16, device="cuda"))
    assert ei.value.code == _lib.VQ_ERR_ARG
    c.close()
