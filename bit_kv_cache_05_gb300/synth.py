"""Seeded synthetic workloads for the KIVI cache and its decode step.

This module only draws inputs: it holds none of the quantization or
attention arithmetic, and both the CUDA library's tests/benchmark and the CPU
oracle take their inputs from it.

The shapes follow the workloads of the VeloxQuant-MLX changelog v0.42.0
"Added" entry (B=1, H=32, D=128, b=2, g=32, S_q=1, S_kv from 512 to 65536),
the KIVI entry of v0.8.0 (fp16 residual window of 32 tokens in its numbers
table) and four derived serving shapes (GQA with outlier key channels, a 4-bit
variant with a prefill-chunk append, a long ragged batch).  Every stream
(K, V, q, outlier channels, per-channel key scales, lengths, appended tokens)
has its own seeded generator, so changing one size never changes another
stream's values.  Seed 42 is the pages' default seed (KVCacheConfig.seed).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

DEFAULT_SEED = 42

# stream offsets: one independent generator per drawn quantity
_S_K, _S_V, _S_Q, _S_OUTLIER, _S_CHSCALE, _S_LEN, _S_KNEW, _S_VNEW = range(8)


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    H_q: int
    H_kv: int
    D: int
    bits: int
    group: int
    residual: int
    seq_lens: List[int]           # tokens in the cache before the step
    n_append: int = 0             # tokens appended per sequence in the step
    key_kind: str = "normal"      # normal | outliers | chscale
    n_outlier: int = 0
    outlier_gain: float = 1.0
    chscale_lo: float = 1.0
    chscale_hi: float = 1.0
    note: str = ""

    @property
    def S_max(self) -> int:
        return max(self.seq_lens)

    @property
    def max_seq(self) -> int:
        return self.S_max + self.n_append

    def params(self) -> Dict[str, int]:
        return dict(B=self.B, H_q=self.H_q, H_kv=self.H_kv, D=self.D,
                    bits=self.bits, group=self.group, residual=self.residual,
                    max_seq=self.max_seq)


def _ragged_lens(B: int, lo: int, hi: int, seed: int) -> List[int]:
    g = torch.Generator().manual_seed(seed * 1000 + _S_LEN)
    return [int(x) for x in torch.randint(lo, hi + 1, (B,), generator=g)]


def workload(name: str, seed: int = DEFAULT_SEED) -> Workload:
    """The named workloads.

    tiny          B=1 H=4/4 D=64 S=256 (224 quantized + 32 residual) b=2 g=32
    pages_S<N>    B=1 H=32/32 D=128 b=2 g=32 R=32, S=N (512 ... 65536)
    gqa_serving   B=16 H=32/8 D=128 S=8192 b=2 g=32 R=32, 8 key outlier
                  channels per kv head scaled x10
    int4_append   B=8 H=32/32 D=128 S=32768 b=4 g=64 R=64, a 512-token fp16
                  chunk appended per sequence, then one decode; 4 key outlier
                  channels x8
    ragged_long   B=4 H=32/8 D=128 S_b ~ U[16384, 131072] b=2 g=32 R=32, per
                  (kv head, channel) key scale log-uniform in [0.1, 10]
    """
    if name == "tiny":
        return Workload(name, 1, 4, 4, 64, 2, 32, 32, [256])
    if name.startswith("pages_S"):
        S = int(name[len("pages_S"):])
        return Workload(name, 1, 32, 32, 128, 2, 32, 32, [S])
    if name == "gqa_serving":
        return Workload(name, 16, 32, 8, 128, 2, 32, 32, [8192] * 16,
                        key_kind="outliers", n_outlier=8, outlier_gain=10.0)
    if name == "int4_append":
        return Workload(name, 8, 32, 32, 128, 4, 64, 64, [32768] * 8,
                        n_append=512, key_kind="outliers", n_outlier=4,
                        outlier_gain=8.0)
    if name == "ragged_long":
        return Workload(name, 4, 32, 8, 128, 2, 32, 32,
                        _ragged_lens(4, 16384, 131072, seed),
                        key_kind="chscale", chscale_lo=0.1, chscale_hi=10.0)
    raise KeyError(name)


def shrink(w: Workload, seq_lens: List[int], B: Optional[int] = None,
           n_append: Optional[int] = None) -> Workload:
    """Same recipe (heads, D, bits, group, window, key distribution) with
    other lengths, for oracle-sized parity cases."""
    B = len(seq_lens) if B is None else B
    assert len(seq_lens) == B
    return dataclasses.replace(
        w, name=w.name + "_small", B=B, seq_lens=list(seq_lens),
        n_append=w.n_append if n_append is None else n_append)


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + stream)
    return g


def _key_channel_gain(w: Workload, seed: int) -> torch.Tensor:
    """Per (kv head, channel) multiplier of the key distribution, [H_kv][D]
    fp32 on the CPU (small, so always drawn on the CPU)."""
    gain = torch.ones(w.H_kv, w.D, dtype=torch.float32)
    if w.key_kind == "outliers":
        g = _gen("cpu", seed, _S_OUTLIER)
        for h in range(w.H_kv):
            idx = torch.randperm(w.D, generator=g)[: w.n_outlier]
            gain[h, idx] = w.outlier_gain
    elif w.key_kind == "chscale":
        g = _gen("cpu", seed, _S_CHSCALE)
        u = torch.rand(w.H_kv, w.D, generator=g, dtype=torch.float64)
        lo, hi = math.log(w.chscale_lo), math.log(w.chscale_hi)
        gain = torch.exp(lo + (hi - lo) * u).to(torch.float32)
    return gain


def _normal(shape, g: torch.Generator, device) -> torch.Tensor:
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)


def make_inputs(w: Workload, seed: int = DEFAULT_SEED, device="cpu"):
    """Draw the step's inputs.

    Returns a dict of fp16 tensors on `device`:
      K, V      [B][H_kv][S_max][D]   prefill keys / values (rows past a
                                      sequence's length are drawn but unused)
      q         [B][H_q][D]           the decode query (S_q = 1)
      K_new, V_new [B][H_kv][n_append][D]   (only when n_append > 0)
    and the int32 CPU tensor seq_lens [B].
    """
    dev = torch.device(device)
    gain = _key_channel_gain(w, seed).to(dev)
    shape = (w.B, w.H_kv, w.S_max, w.D)
    K = _normal(shape, _gen(dev, seed, _S_K), dev)
    K.mul_(gain.view(1, w.H_kv, 1, w.D))
    K = K.half()
    V = _normal(shape, _gen(dev, seed, _S_V), dev).half()
    q = _normal((w.B, w.H_q, w.D), _gen(dev, seed, _S_Q), dev).half()
    out = dict(K=K, V=V, q=q,
               seq_lens=torch.tensor(w.seq_lens, dtype=torch.int32))
    if w.n_append:
        nshape = (w.B, w.H_kv, w.n_append, w.D)
        Kn = _normal(nshape, _gen(dev, seed, _S_KNEW), dev)
        Kn.mul_(gain.view(1, w.H_kv, 1, w.D))
        out["K_new"] = Kn.half()
        out["V_new"] = _normal(nshape, _gen(dev, seed, _S_VNEW), dev).half()
    return out


def decode_tokens(w: Workload, n_steps: int, seed: int = DEFAULT_SEED,
                  device="cpu"):
    """Per-step single-token K/V and queries for a run of decode steps:
    K1, V1 [n_steps][B][H_kv][1][D], q [n_steps][B][H_q][D] (fp16)."""
    dev = torch.device(device)
    gain = _key_channel_gain(w, seed).to(dev)
    K1 = _normal((n_steps, w.B, w.H_kv, 1, w.D),
                 _gen(dev, seed, _S_KNEW + 10), dev)
    K1.mul_(gain.view(1, 1, w.H_kv, 1, w.D))
    V1 = _normal((n_steps, w.B, w.H_kv, 1, w.D),
                 _gen(dev, seed, _S_VNEW + 10), dev)
    q = _normal((n_steps, w.B, w.H_q, w.D), _gen(dev, seed, _S_Q + 10), dev)
    return K1.half(), V1.half(), q.half()
