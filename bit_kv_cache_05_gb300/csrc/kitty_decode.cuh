// Kitty fused decode (the kernel template; kitty_decode_d64.cu and
// kitty_decode_d128.cu instantiate it per query heads per kv head, kitty.cu
// plans and launches).
//
// Method: VeloxQuant-MLX changelog v0.11.0 "New" (Kitty: the key channels of
// high running variance in 4 bits, the rest in 2 bits, values left at fp16)
// and v0.42.0 "Added" (attention directly over the group-affine cache, k_hat
// never written to memory, online softmax in fp32).
#pragma once

#include <atomic>
#include <mutex>
#include <type_traits>

#include "bulk_pipe.cuh"
#include "vqk_internal.cuh"

namespace vqk {
namespace kitdec {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
// One stage per warp: a block's 8 KB of fp16 values make a stage 10.9 KB,
// so a single stage keeps four to five CTAs on an SM, whose warps hide one
// another's copy latency (two stages per warp allowed two CTAs: 87 against
// 74.7 us at the pages' shape)
constexpr int kStages = 1;
constexpr unsigned kFull = 0xffffffffu;
// Code fields enter the key products as fp32 subnormals (a field masked in
// place at bit pos of a 32-bit word, pos + width <= 16, reads as
// code * 2^(pos - 149)); each field's factor carries 2^(149 - kCarry - pos),
// so every product is the exact one times 2^-kCarry.  Needs IEEE subnormals
// on the FMA path (the library is built without flush-to-zero).
constexpr int kCarry = 64;

__device__ __forceinline__ float pow2(int e) {   // 2^e, -126 <= e <= 127
  return __int_as_float((127 + e) << 23);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ int find_seq(const int32_t *prefix, int B, int item) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// A warp's stage holds one block of up to 32 tokens of one key group: the
// tokens' key rows ((D + kitty_hi) / 4 bytes each, at most D / 2), their
// fp16 value rows, and with a group's first block the group's key scale and
// zero rows and the 16-byte-aligned window holding its channel mask.
template <int D> struct KitStage {
  static constexpr int KC = 0, VF = 16 * D, KS = VF + 64 * D, KZ = KS + 2 * D,
                       KM = KZ + 2 * D, BYTES = (KM + 16 + 127) / 128 * 128;
};

// Shared memory of a CTA: q' [GQ][D] (fp32), then per warp its mbarriers,
// a' [GQ][D] of its current group in field order (fp32) and kStages stages.
template <int D, int GQ> struct KitSmem {
  static constexpr int SQ = GQ * D * 4;
  static constexpr int OFF_W0 = (SQ + 127) / 128 * 128;
  static constexpr int W_BAR = 0;
  static constexpr int W_SA = 32;
  static constexpr int W_ST = (W_SA + GQ * D * 4 + 127) / 128 * 128;
  static constexpr int PER_WARP = W_ST + kStages * KitStage<D>::BYTES;
  static constexpr int BYTES = OFF_W0 + kWarps * PER_WARP;
  static_assert(PER_WARP % 128 == 0, "stages stay 128-byte aligned");
};

// bit position of field f of a key row within its 16-bit half: fields
// 0 ... HI-1 are 4 bits wide (8 per word), the rest 2 bits (16 per word)
__device__ __forceinline__ int kit_pos(int f, int HI) {
  return f < HI ? (4 * (f & 7)) & 15 : (2 * ((f - HI) & 15)) & 15;
}

// Fused decode over a Kitty cache.  One CTA of 4 warps per (work item, kv
// head); an item takes the key groups k, k + nq, k + 2 nq, ... of its
// sequence and the warps take those groups round robin, each copying its
// blocks (32 tokens, at most g) into its own stage by bulk copies.  Per
// group a' = q' s in field order (the field of channel c follows from the
// group's mask: the 4-bit channels first, ascending, then the 2-bit ones)
// and beta = q'.z; per block:
//  - scores, one token per lane: the lane's row words against a' (one
//    and-mask and one FMA per field, the fields as fp32 subnormals);
//  - online softmax per block and query head (sums kept per lane);
//  - values, lanes over channels (lane*CPL ...): the fp16 rows from the
//    stage, the block's weights by shuffles.
// A sequence's last item also folds in the fp16 residual window.  The CTA's
// warps are merged with a log-sum-exp into one partial per item.
template <int D, int GQ>
__global__ void __launch_bounds__(kThreads)
k_decode_kitty(Geometry geo, Planes pl, DecodeArgs args, DecodeTable tab) {
  using SG = KitStage<D>;
  using SM = KitSmem<D, GQ>;
  constexpr int CPL = D / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float red_m[kWarps][GQ], red_l[kWarps][GQ];
  float *sq = reinterpret_cast<float *>(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char *ws = smem + SM::OFF_W0 + warp * SM::PER_WARP;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ws + SM::W_BAR);
  float *sa = reinterpret_cast<float *>(ws + SM::W_SA);
  unsigned char *stage0 = ws + SM::W_ST;

  const int item = blockIdx.x, h = blockIdx.y;
  const int b = find_seq(tab.prefix, geo.B, item);
  const int k = item - tab.prefix[b];
  const int g = geo.g, HI = geo.kitty_hi;
  const int krow = (D + HI) / 4;                 // key row bytes
  const size_t bh = (size_t)b * geo.H_kv + h;
  const int Tq = tab.Tq[b];
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = threadIdx.x; i < GQ * D; i += kThreads) {
    const int hh = i / D, c = i % D;
    sq[i] = __half2float(args.q[((size_t)b * geo.H_q + h * GQ + hh) * D + c]) *
            args.scale_log2;
  }
  __syncthreads();
  // the combine kernel behind this one waits for its completion
  // (griddepcontrol.wait); releasing it now only lets it be scheduled
  asm volatile("griddepcontrol.launch_dependents;");

  float m[GQ], l[GQ], o[GQ][CPL];
#pragma unroll
  for (int hh = 0; hh < GQ; ++hh) {
    m[hh] = -INFINITY; l[hh] = 0.f;
#pragma unroll
    for (int u = 0; u < CPL; ++u) o[hh][u] = 0.f;
  }
  // online softmax of one score per lane (-inf where absent): updates the
  // running maximum (rescaling o and the lane's sum), returns the weights
  auto fold = [&](const float (&sc)[GQ], float (&p)[GQ]) {
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
      if (__any_sync(kFull, sc[hh] > m[hh])) {
        float mb = sc[hh];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
          mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, off));
        const float mn = fmaxf(m[hh], mb);
        const float alpha = m[hh] == -INFINITY ? 0.f : exp2f(m[hh] - mn);
        l[hh] *= alpha;
#pragma unroll
        for (int u = 0; u < CPL; ++u) o[hh][u] *= alpha;
        m[hh] = mn;
      }
      p[hh] = sc[hh] == -INFINITY ? 0.f : exp2f(sc[hh] - m[hh]);
      l[hh] += p[hh];
    }
  };
  // the weights p of the block (one per lane) applied to its fp16 value
  // rows: lane owns channels lane*CPL ...
  auto values = [&](const __half *vrow0, int nt, const float (&p)[GQ], int rstride) {
#pragma unroll 8
    for (int jj = 0; jj < nt; ++jj) {
      const __half *vr = vrow0 + (size_t)jj * rstride + lane * CPL;
      float v[CPL];
      if constexpr (CPL == 4) {
        const uint2 r = *reinterpret_cast<const uint2 *>(vr);
        const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
        const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
        v[0] = v01.x; v[1] = v01.y; v[2] = v23.x; v[3] = v23.y;
      } else {
        const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(vr));
        v[0] = v01.x; v[1] = v01.y;
      }
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) {
        const float pj = __shfl_sync(kFull, p[hh], jj);
        // two channels per packed (f32x2) FMA
#pragma unroll
        for (int u = 0; u < CPL; u += 2) {
          const float2 r = __ffma2_rn(make_float2(pj, pj), make_float2(v[u], v[u + 1]),
                                      make_float2(o[hh][u], o[hh][u + 1]));
          o[hh][u] = r.x;
          o[hh][u + 1] = r.y;
        }
      }
    }
  };

  bool failed = false;
  uint32_t phase = 0, pending = 0;
  {
    // the item's key groups: k, k + nq, ... of the sequence's Tq / g
    const int nq = tab.nq[b];
    const int Gend = Tq / g;
    const int bt = g < 32 ? g : 32;             // tokens per block
    const int nb = g / bt;                      // blocks per group
    const uint8_t *kc0 = pl.Kc + bh * geo.Tcap * krow;
    const __half *vf0 = pl.Vf + bh * geo.Tcap * D;
    const __half *ks0 = pl.Ks + bh * (geo.Tcap / g) * D;
    const __half *kz0 = pl.Kz + bh * (geo.Tcap / g) * D;
    const uint32_t *km0 = pl.kmask + bh * (geo.Tcap / g) * (D / 32);
    struct Cur { int G, blk; };
    auto advance = [&](Cur &c) {
      if (++c.blk == nb) { c.blk = 0; c.G += kWarps * nq; }
    };
    auto issue = [&](const Cur &c, int s) {
      if (lane == 0) {
        unsigned char *st = stage0 + s * SG::BYTES;
        const int r0 = c.G * g + c.blk * bt;     // first token of the block
        const uint32_t kb = bt * krow, vb = bt * D * 2;
        // the group's mask: the aligned 16 bytes holding its D / 32 words
        // (the plane is padded to 256 bytes, so the window stays inside it)
        const uint32_t *mk = km0 + (size_t)c.G * (D / 32);
        const uint32_t *mka = reinterpret_cast<const uint32_t *>(
            reinterpret_cast<uintptr_t>(mk) & ~uintptr_t(15));
        mbar_expect_tx(&bars[s], kb + vb + (c.blk == 0 ? 4 * D + 16 : 0));
        bulk_g2s(st + SG::KC, kc0 + (size_t)r0 * krow, kb, &bars[s]);
        bulk_g2s(st + SG::VF, vf0 + (size_t)r0 * D, vb, &bars[s]);
        if (c.blk == 0) {
          bulk_g2s(st + SG::KS, ks0 + (size_t)c.G * D, 2 * D, &bars[s]);
          bulk_g2s(st + SG::KZ, kz0 + (size_t)c.G * D, 2 * D, &bars[s]);
          bulk_g2s(st + SG::KM, mka, 16, &bars[s]);
        }
      }
    };
    Cur pc{k + warp * nq, 0};   // next block to copy
    Cur cc = pc;                // next block to compute
    for (int s = 0; s < kStages && pc.G < Gend; ++s) {
      issue(pc, s);
      pending |= 1u << s;
      advance(pc);
    }
    {
      // (run before the first stage lands: its loads overlap the pipeline's
      // first copies)
      // the fp16 residual window, folded into the running states of the
      // sequence's last items: block j of kWinT tokens goes to item
      // nq - 1 - (j mod nq), warp j mod kWarps of it (lanes 0 ... kWinT - 1
      // score a token each, lanes over channels sum the values), so that no
      // CTA carries much more than its share and every warp's loads are few
      // rounds
      constexpr int kWinT = 8;
      const int nblk = (tab.nres[b] + kWinT - 1) / kWinT;
      for (int j = tab.nq[b] - 1 - k; j < nblk; j += tab.nq[b]) {
        if (j % kWarps != warp) continue;
        const int i0 = j * kWinT;
        const int i = i0 + lane;
        const bool ok = lane < kWinT && i < tab.nres[b];
        // ring slots: the block's first token's, then one wrap at most (the
        // window holds fewer than Rcap tokens)
        const int s0 = (Tq + i0) % geo.Rcap;
        int sl = s0 + lane;
        if (sl >= geo.Rcap) sl -= geo.Rcap;
        // this lane's key row in 16-byte loads, half of them in flight at a
        // time (two rounds; the loop keeps q' in shared memory)
        const uint4 *kr = reinterpret_cast<const uint4 *>(
            pl.Kr + (bh * geo.Rcap + (ok ? sl : s0)) * D);
        constexpr int KB = D / 16;
        float acc[GQ];
  #pragma unroll
        for (int hh = 0; hh < GQ; ++hh) acc[hh] = 0.f;
  #pragma unroll 1
        for (int j0 = 0; j0 < D / 8; j0 += KB) {
          uint4 kx[KB];
  #pragma unroll
          for (int j = 0; j < KB; ++j) kx[j] = kr[j0 + j];
  #pragma unroll
          for (int j = 0; j < KB; ++j) {
            const __half2 *k2 = reinterpret_cast<const __half2 *>(&kx[j]);
  #pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 kv = __half22float2(k2[e]);
              const int c = 8 * (j0 + j) + 2 * e;
  #pragma unroll
              for (int hh = 0; hh < GQ; ++hh)
                acc[hh] = fmaf(sq[hh * D + c], kv.x, fmaf(sq[hh * D + c + 1], kv.y, acc[hh]));
            }
          }
        }
        float sc[GQ], p[GQ];
  #pragma unroll
        for (int hh = 0; hh < GQ; ++hh) sc[hh] = ok ? acc[hh] : -INFINITY;
        fold(sc, p);
        const int nb = min(kWinT, tab.nres[b] - i0);
  #pragma unroll 4
        for (int jj = 0; jj < nb; ++jj) {
          int sj = s0 + jj;
          if (sj >= geo.Rcap) sj -= geo.Rcap;
          const __half *vr = pl.Vr + (bh * geo.Rcap + sj) * D + lane * CPL;
          float v[CPL];
  #pragma unroll
          for (int u = 0; u < CPL; ++u) v[u] = __half2float(vr[u]);
  #pragma unroll
          for (int hh = 0; hh < GQ; ++hh) {
            const float pj = __shfl_sync(kFull, p[hh], jj);
  #pragma unroll
            for (int u = 0; u < CPL; ++u) o[hh][u] = fmaf(pj, v[u], o[hh][u]);
          }
        }
      }
    }
    float beta[GQ];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) beta[hh] = 0.f;
    int s = 0;
    while (cc.G < Gend) {
      const bool ok = __all_sync(kFull, mbar_wait(&bars[s], (phase >> s) & 1u));
      if (!ok) { failed = true; break; }
      phase ^= 1u << s;
      pending &= ~(1u << s);
      const unsigned char *st = stage0 + s * SG::BYTES;
      if (cc.blk == 0) {
        // a' of the group in field order and beta = q'.z, lanes over channels
        const __half *ks = reinterpret_cast<const __half *>(st + SG::KS);
        const __half *kz = reinterpret_cast<const __half *>(st + SG::KZ);
        const uint32_t *mk = reinterpret_cast<const uint32_t *>(st + SG::KM) +
                             (((bh * (geo.Tcap / g) + cc.G) * (D / 32)) & 3);
        int below0 = 0;                          // 4-bit channels below word c/32
        const int cw = (lane * CPL) >> 5;
        for (int w = 0; w < cw; ++w) below0 += __popc(mk[w]);
        const uint32_t mw = mk[cw];
        float part[GQ];
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) part[hh] = 0.f;
#pragma unroll
        for (int u = 0; u < CPL; ++u) {
          const int c = lane * CPL + u;
          const int below = below0 + __popc(mw & ((1u << (c & 31)) - 1u));
          const int f = ((mw >> (c & 31)) & 1u) ? below : HI + (c - below);
          const float sf = __half2float(ks[c]) * pow2(149 - kCarry - kit_pos(f, HI));
          const float zf = __half2float(kz[c]);
#pragma unroll
          for (int hh = 0; hh < GQ; ++hh) {
            const float qc = sq[hh * D + c];
            sa[hh * D + f] = qc * sf;
            part[hh] = fmaf(qc, zf, part[hh]);
          }
        }
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) beta[hh] = warp_sum(part[hh]);
        __syncwarp();
      }
      // scores: lane = token; its row's 4-bit words, then its 2-bit words,
      // two fields per packed (f32x2) FMA
      float sc[GQ];
      {
        float2 acc[GQ][2];
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) acc[hh][0] = acc[hh][1] = make_float2(0.f, 0.f);
        if (lane < bt) {
          const uint32_t *row = reinterpret_cast<const uint32_t *>(st + SG::KC + lane * krow);
#pragma unroll 2
          for (int w = 0; w < HI / 8; ++w) {
            const uint32_t x = row[w], y = x >> 16;
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) {
              const float4 a0 = *reinterpret_cast<const float4 *>(sa + hh * D + 8 * w);
              const float4 a1 = *reinterpret_cast<const float4 *>(sa + hh * D + 8 * w + 4);
              float2 r0 = acc[hh][0], r1 = acc[hh][1];
              r0 = __ffma2_rn(make_float2(a0.x, a0.y),
                              make_float2(__uint_as_float(x & 0xFu), __uint_as_float(x & 0xF0u)), r0);
              r0 = __ffma2_rn(make_float2(a0.z, a0.w),
                              make_float2(__uint_as_float(x & 0xF00u), __uint_as_float(x & 0xF000u)), r0);
              r1 = __ffma2_rn(make_float2(a1.x, a1.y),
                              make_float2(__uint_as_float(y & 0xFu), __uint_as_float(y & 0xF0u)), r1);
              r1 = __ffma2_rn(make_float2(a1.z, a1.w),
                              make_float2(__uint_as_float(y & 0xF00u), __uint_as_float(y & 0xF000u)), r1);
              acc[hh][0] = r0;
              acc[hh][1] = r1;
            }
          }
#pragma unroll 2
          for (int w = 0; w < (D - HI) / 16; ++w) {
            const uint32_t x = row[HI / 8 + w], y = x >> 16;
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) {
              const float *aw = sa + hh * D + HI + 16 * w;
              float2 r0 = acc[hh][0], r1 = acc[hh][1];
#pragma unroll
              for (int e = 0; e < 8; e += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(aw + e);
                r0 = __ffma2_rn(make_float2(a4.x, a4.y),
                                make_float2(__uint_as_float(x & (3u << (2 * e))),
                                            __uint_as_float(x & (3u << (2 * e + 2)))), r0);
                r0 = __ffma2_rn(make_float2(a4.z, a4.w),
                                make_float2(__uint_as_float(x & (3u << (2 * e + 4))),
                                            __uint_as_float(x & (3u << (2 * e + 6)))), r0);
                const float4 b4 = *reinterpret_cast<const float4 *>(aw + 8 + e);
                r1 = __ffma2_rn(make_float2(b4.x, b4.y),
                                make_float2(__uint_as_float(y & (3u << (2 * e))),
                                            __uint_as_float(y & (3u << (2 * e + 2)))), r1);
                r1 = __ffma2_rn(make_float2(b4.z, b4.w),
                                make_float2(__uint_as_float(y & (3u << (2 * e + 4))),
                                            __uint_as_float(y & (3u << (2 * e + 6)))), r1);
              }
              acc[hh][0] = r0;
              acc[hh][1] = r1;
            }
          }
        }
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh)
          sc[hh] = lane < bt ? fmaf((acc[hh][0].x + acc[hh][0].y) + (acc[hh][1].x + acc[hh][1].y),
                                    pow2(kCarry), beta[hh])
                             : -INFINITY;
      }
      float p[GQ];
      fold(sc, p);
      values(reinterpret_cast<const __half *>(st + SG::VF), bt, p, D);
      __syncwarp();
      if (pc.G < Gend) {
        // every lane's reads of the stage come before the copies into it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue(pc, s);
        pending |= 1u << s;
        advance(pc);
      }
      advance(cc);
      if (++s == kStages) s = 0;
    }
    if (failed) {
      if (lane == 0 && args.err) atomicOr(args.err, 1u);
      // let the copies still in flight land (bounded) before the CTA ends
      for (int j = 0; j < kStages; ++j)
        if (pending & (1u << j)) mbar_wait(&bars[j], (phase >> j) & 1u);
    }
  }

  // the warp's (m, l, o) -> its a' region, then the CTA's log-sum-exp merge
  __syncwarp();
#pragma unroll
  for (int hh = 0; hh < GQ; ++hh) {
    const float lsum = warp_sum(l[hh]);
    if (lane == 0) { red_m[warp][hh] = m[hh]; red_l[warp][hh] = lsum; }
#pragma unroll
    for (int u = 0; u < CPL; ++u) sa[hh * D + lane * CPL + u] = o[hh][u];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < GQ * (D + 2); i += kThreads) {
    const int hh = i / (D + 2), c = i % (D + 2);
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, red_m[ww][hh]);
    float acc = 0.f;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) {
      const float f = red_m[ww][hh] == -INFINITY ? 0.f : exp2f(red_m[ww][hh] - M);
      const float *so = reinterpret_cast<const float *>(
          smem + SM::OFF_W0 + ww * SM::PER_WARP + SM::W_SA);
      acc += f * (c < D ? so[hh * D + c] : red_l[ww][hh]);
    }
    const int hq = h * GQ + hh;
    float *dst = pl.part + (((size_t)b * geo.H_q + hq) * geo.max_items + k) * (D + 2);
    dst[c] = c == D ? M : acc;
  }
}

struct KitKernel {
  const void *f = nullptr;
  int smem = 0;          // dynamic shared memory the kernel needs
  int smem_static = 0;   // its static shared memory
  int occ = 0;           // CTAs per SM at smem
};

// the decode instance of (D, GQ) on the current device: its dynamic shared
// memory limit raised to the device's (so that a launch may pad its request
// to cap the CTAs per SM) and its occupancy, both set up once per device
template <int D, int GQ>
KitKernel kit_kernel() {
  static std::mutex mu;
  static std::atomic<uint64_t> done{0};
  static KitKernel dev_k[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return {};
  if (!((done.load(std::memory_order_acquire) >> dev) & 1u)) {
    std::lock_guard<std::mutex> lock(mu);
    if (!((done.load(std::memory_order_relaxed) >> dev) & 1u)) {
      KitKernel kk;
      kk.f = reinterpret_cast<const void *>(&k_decode_kitty<D, GQ>);
      kk.smem = KitSmem<D, GQ>::BYTES;
      cudaFuncAttributes fa;
      int optin = 0;
      if (cudaFuncGetAttributes(&fa, kk.f) != cudaSuccess ||
          cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
              cudaSuccess ||
          cudaFuncSetAttribute(kk.f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               optin - (int)fa.sharedSizeBytes) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&kk.occ, kk.f, kThreads, kk.smem) !=
              cudaSuccess)
        return {};
      kk.smem_static = (int)fa.sharedSizeBytes;
      dev_k[dev] = kk;
      done.fetch_or(1ull << dev, std::memory_order_release);
    }
  }
  return dev_k[dev];
}

// the instance for H_q / H_kv = gq at this D (f == nullptr: none)
template <int D>
KitKernel pick(int gq) {
  switch (gq) {
    case 1: return kit_kernel<D, 1>();
    case 2: return kit_kernel<D, 2>();
    case 3: return kit_kernel<D, 3>();
    case 4: return kit_kernel<D, 4>();
    case 5: return kit_kernel<D, 5>();
    case 6: return kit_kernel<D, 6>();
    case 7: return kit_kernel<D, 7>();
    case 8: return kit_kernel<D, 8>();
    default: return {};
  }
}

KitKernel pick_d64(int gq);
KitKernel pick_d128(int gq);

}  // namespace kitdec
}  // namespace vqk
