// AgeTieredKV fused decode (the kernel template; age_decode_d64.cu and
// age_decode_d128.cu instantiate it per query heads per kv head, age.cu
// plans and launches).
//
// Method: VeloxQuant-MLX method overview, AgeTieredKV entry (three widths
// of the KIVI group quantizer by token age) and changelog v0.42.0 "Added"
// (attention directly over the group-affine cache, k_hat / v_hat never
// written to memory, online softmax in fp32).  A group's rows are packed
// densely at its width (age_row_off).
#pragma once

#include <atomic>
#include <mutex>
#include <type_traits>

#include "bulk_pipe.cuh"
#include "vqk_internal.cuh"

namespace vqk {
namespace agedec {

__device__ __forceinline__ int find_seq(const int32_t *prefix, int B, int item) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  return lo;
}

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
constexpr unsigned kFull = 0xffffffffu;
// Code fields enter the products as fp32 subnormals: a w-bit field masked in
// place at bit position pos of a 32-bit word (pos + w <= 16) reads as
// code * 2^(pos - 149), exactly.  Its factor carries 2^(149 - kCarry - pos),
// so every product is the exact one times 2^-kCarry: one and-mask and one
// FMA per field, no integer-to-float conversion.  kCarry = 64 keeps the
// factors finite for q' s and p s below 2^40 and the products normal down to
// 2^-62 of the largest.  This needs IEEE subnormals on the FMA path (the
// library is built without flush-to-zero).
constexpr int kCarry = 64;
// tokens of a residual-window block (lanes 0 ... kWinT - 1 score one each)
constexpr int kWinT = 8;

__device__ __forceinline__ float pow2(int e) {   // 2^e, -126 <= e <= 127
  return __int_as_float((127 + e) << 23);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// A warp's stage holds one block of bt tokens of one key group (bt = 64 / w
// tokens at width w, at most g: 8 D bytes of codes per plane): the block's
// key rows and value rows, the value scale and zero rows of its tokens, and
// with a group's first block the group's key scale and zero rows.  Small
// stages keep five CTAs on an SM; the narrow tiers, which hold most tokens,
// fill all 32 lanes of the key loop.
template <int D> struct AgeStage {
  static constexpr int KC = 0, VC = 8 * D, VS = 16 * D, VZ = 18 * D,
                       KS = 20 * D, KZ = 22 * D, BYTES = 24 * D;
};

// Shared memory of a CTA: q' [GQ][D] (fp32), then per warp its mbarriers,
// a' [GQ][D] of its current group (fp32), the block's value weights (w', u)
// [GQ][bt][D/g] (float2, at most 8 D bytes per head) and kStages stages.
template <int D, int GQ> struct AgeSmem {
  static constexpr int SQ = GQ * D * 4;
  static constexpr int OFF_W0 = (SQ + 127) / 128 * 128;
  static constexpr int W_BAR = 0;
  static constexpr int W_SA = 32;
  static constexpr int W_WU = W_SA + GQ * D * 4;
  static constexpr int W_ST = (W_WU + GQ * 8 * D + 127) / 128 * 128;
  static constexpr int PER_WARP = W_ST + kStages * AgeStage<D>::BYTES;
  static constexpr int BYTES = OFF_W0 + kWarps * PER_WARP;
  static_assert(PER_WARP % 128 == 0, "stages stay 128-byte aligned");
};

// Fused decode over an age-tiered cache.  One CTA of 4 warps per (work
// item, kv head); the sequence's staged blocks are dealt round robin over
// its items' warps, each warp streaming its blocks through its own
// bulk-copy pipeline (kStages stages, one mbarrier each, bounded waits).
// Per block:
//  - scores, one token per lane: its key row's fields against
//    a'_c = q'_c s_Gc (the group's a' built when the warp's block is of
//    another group than its previous one), plus the group's zero-point term
//    beta = sum_c q'_c z_Gc;
//  - a per-block online softmax per query head (the warp maximum reduced
//    only when some score exceeds the running one; sums stay per lane);
//  - value weights, one token per lane: w' = p s_tj and u = p z_tj per value
//    group j, through shared memory;
//  - values, lanes over channels (lane*CPL ...): o_c += w' code_tc per token
//    and the zero-point sum sum_t u_tj.
// The fp16 residual window's blocks are dealt after the groups', read from
// global memory.  The CTA's warps are merged with a log-sum-exp into one
// partial per item.
template <int D, int GQ>
__global__ void __launch_bounds__(kThreads)
k_decode_age(Geometry geo, Planes pl, DecodeArgs args, DecodeTable tab) {
  using SG = AgeStage<D>;
  using SM = AgeSmem<D, GQ>;
  constexpr int CPL = D / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float red_m[kWarps][GQ], red_l[kWarps][GQ];
  float *sq = reinterpret_cast<float *>(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char *ws = smem + SM::OFF_W0 + warp * SM::PER_WARP;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ws + SM::W_BAR);
  float *sa = reinterpret_cast<float *>(ws + SM::W_SA);
  float2 *wu = reinterpret_cast<float2 *>(ws + SM::W_WU);
  unsigned char *stage0 = ws + SM::W_ST;

  const int item = blockIdx.x, h = blockIdx.y;
  const int b = find_seq(tab.prefix, geo.B, item);
  const int k = item - tab.prefix[b];
  const int g = geo.g, NJ = D / g;
  const int jv = lane * CPL / g;     // value group of the lane's channels
  const size_t bh = (size_t)b * geo.H_kv + h;
  const int Tq = tab.Tq[b];
  const int S = Tq + tab.nres[b];
  // The sequence's work in staged blocks: its Gend quantized key groups,
  // each in nb = max(1, g w / 64) blocks of 64 / w tokens at its tier's
  // width w (tier 2's groups first, then tier 1's, then tier 0's), then the
  // fp16 residual window in kWinT-token blocks.  Block x goes to item
  // x mod nq, warp (x / nq) mod kWarps: every warp of every item takes the
  // same mix of widths and window blocks, whatever their relative costs
  // (groups of the recent, wider tiers are several blocks; a whole group per
  // warp left the warps that held one a block or more behind the rest).
  const int nq = tab.nq[b];
  const int Gend = Tq / g;
  // tiers by group index (age_tier): groups G < Ga are in tier 2, G < Gb
  // in tier 1 or 2, the rest in tier 0
  const int Ga = min(max(0, (S - geo.age_b2) / g), Gend);
  const int Gb = min(max(Ga, (S - geo.age_b1) / g), Gend);
  const int wA = geo.age_bits[2], wB = geo.age_bits[1], wC = geo.age_bits[0];
  // log2 of the blocks per group (g is 16 ... 128 and w 2, 4 or 8, so
  // nb is a power of two)
  const int lA = __ffs(max(1, g * wA / 64)) - 1, lB = __ffs(max(1, g * wB / 64)) - 1,
            lC = __ffs(max(1, g * wC / 64)) - 1;
  const int XA = Ga << lA, XB = XA + ((Gb - Ga) << lB), XQ = XB + ((Gend - Gb) << lC);
  const int nblk = (tab.nres[b] + kWinT - 1) / kWinT;
  const int stride = nq * kWarps;
  const int x0 = k + nq * warp;         // this warp's first block
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

  float m[GQ], l[GQ], o[GQ][CPL], zl[GQ];
#pragma unroll
  for (int hh = 0; hh < GQ; ++hh) {
    m[hh] = -INFINITY; l[hh] = 0.f; zl[hh] = 0.f;
#pragma unroll
    for (int u = 0; u < CPL; ++u) o[hh][u] = 0.f;
  }
  // online softmax of one score per lane (-inf where absent): updates the
  // running maximum (rescaling o, zl and the lane's sum) and returns the
  // lane's weights
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
        zl[hh] *= alpha;
#pragma unroll
        for (int u = 0; u < CPL; ++u) o[hh][u] *= alpha;
        m[hh] = mn;
      }
      p[hh] = sc[hh] == -INFINITY ? 0.f : exp2f(sc[hh] - m[hh]);
      l[hh] += p[hh];
    }
  };

  int w_acc = 0;        // width the value sums o are carried at (0: none)
  bool failed = false;
  uint32_t phase = 0, pending = 0;
  {
    // the (b, h) planes
    const unsigned char *kc0 = pl.Kc + bh * geo.Tcap * D;
    const unsigned char *vc0 = pl.Vc + bh * geo.Tcap * D;
    const __half *vs0 = pl.Vs + bh * geo.Tcap * NJ;
    const __half *vz0 = pl.Vz + bh * geo.Tcap * NJ;
    const __half *ks0 = pl.Ks + bh * (geo.Tcap / g) * D;
    const __half *kz0 = pl.Kz + bh * (geo.Tcap / g) * D;
    // this warp's blocks in order, x0 + stride i < XQ: block x is block
    // blk of group G at width w; `first` when the warp's previous block was
    // of another group (the stage then also takes the group's key scale and
    // zero rows, and the warp builds the group's a' and beta)
    struct Cur { int x, G, blk, w; bool first; };
    auto at = [&](int x, int Gprev) {
      Cur c{x, Gend, 0, 2, false};
      if (x < XA) {
        c.G = x >> lA; c.blk = x & ((1 << lA) - 1); c.w = wA;
      } else if (x < XB) {
        const int y = x - XA;
        c.G = Ga + (y >> lB); c.blk = y & ((1 << lB) - 1); c.w = wB;
      } else if (x < XQ) {
        const int y = x - XB;
        c.G = Gb + (y >> lC); c.blk = y & ((1 << lC) - 1); c.w = wC;
      }
      c.first = c.G != Gprev;
      return c;
    };
    auto advance = [&](Cur &c) { c = at(c.x + stride, c.G); };
    auto issue = [&](const Cur &c, int s) {
      if (lane == 0) {
        const int bt = min(g, 64 / c.w);
        const uint32_t cb = bt * (D * c.w / 8), vb = bt * NJ * 2;
        unsigned char *st = stage0 + s * SG::BYTES;
        const int r0 = c.G * g + c.blk * bt;      // first token of the block
        const size_t co = (size_t)c.G * g * D + (size_t)c.blk * cb;
        mbar_expect_tx(&bars[s], 2 * cb + 2 * vb + (c.first ? 4 * D : 0));
        bulk_g2s(st + SG::KC, kc0 + co, cb, &bars[s]);
        bulk_g2s(st + SG::VC, vc0 + co, cb, &bars[s]);
        bulk_g2s(st + SG::VS, vs0 + (size_t)r0 * NJ, vb, &bars[s]);
        bulk_g2s(st + SG::VZ, vz0 + (size_t)r0 * NJ, vb, &bars[s]);
        if (c.first) {
          bulk_g2s(st + SG::KS, ks0 + (size_t)c.G * D, 2 * D, &bars[s]);
          bulk_g2s(st + SG::KZ, kz0 + (size_t)c.G * D, 2 * D, &bars[s]);
        }
      }
    };
    Cur pc = at(x0, -1);          // next block to copy
    Cur cc = pc;                  // next block to compute
    for (int s = 0; s < kStages && pc.x < XQ; ++s) {
      issue(pc, s);
      pending |= 1u << s;
      advance(pc);
    }
    float beta[GQ];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) beta[hh] = 0.f;

    // one staged block at width W
    auto block = [&](auto w_tag, auto bt_tag, const unsigned char *st, bool first) {
      constexpr int W = decltype(w_tag)::value;
      constexpr int bt = decltype(bt_tag)::value;   // tokens of the block
      constexpr uint32_t CM = (1u << W) - 1u;
      constexpr int PER = 32 / W;         // fields per 32-bit word
      constexpr int RB = D * W / 8;       // row bytes
      if (first) {
        // the group's a' = q' s 2^(149 - kCarry - pos), pos = c W mod 16 (the
        // field's place after the key loop's optional 16-bit shift), and
        // beta = q'.z, lanes over channels
        const __half *ks = reinterpret_cast<const __half *>(st + SG::KS);
        const __half *kz = reinterpret_cast<const __half *>(st + SG::KZ);
        float sv[CPL], zv[CPL];
#pragma unroll
        for (int u = 0; u < CPL; ++u) {
          sv[u] = __half2float(ks[lane * CPL + u]);
          zv[u] = __half2float(kz[lane * CPL + u]);
        }
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
          float part = 0.f;
#pragma unroll
          for (int u = 0; u < CPL; ++u) {
            const int c = lane * CPL + u;
            const float qc = sq[hh * D + c];
            sa[hh * D + c] = qc * sv[u] * pow2(149 - kCarry - ((c * W) & 15));
            part = fmaf(qc, zv[u], part);
          }
          beta[hh] = warp_sum(part);
        }
        // the value sums move to this width's field positions
        if (w_acc != W) {
          if (w_acc) {
#pragma unroll
            for (int u = 0; u < CPL; ++u) {
              const float f = pow2(((u * W) & 15) - ((u * w_acc) & 15));
#pragma unroll
              for (int hh = 0; hh < GQ; ++hh) o[hh][u] *= f;
            }
          }
          w_acc = W;
        }
        __syncwarp();
      }
      // scores: lane = token
      float sc[GQ];
      {
        // one partial sum per word of a 16-byte load: four chains of packed
        // two-channel FMAs (f32x2: two fields per instruction)
        float2 acc[GQ][4];
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh)
#pragma unroll
          for (int jw = 0; jw < 4; ++jw) acc[hh][jw] = make_float2(0.f, 0.f);
        if (lane < bt) {
          const uint4 *row = reinterpret_cast<const uint4 *>(st + SG::KC + lane * RB);
#pragma unroll 2
          for (int qd = 0; qd < RB / 16; ++qd) {
            const uint4 x4 = row[qd];
            const uint32_t xw[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
            for (int jw = 0; jw < 4; ++jw) {
              const uint32_t x = xw[jw], y = x >> 16;
              const int cw = (qd * 4 + jw) * PER;     // first channel of the word
#pragma unroll
              for (int e = 0; e < PER; e += 4) {
                float f[4];
#pragma unroll
                for (int ee = 0; ee < 4; ++ee) {
                  const int fe = e + ee;
                  const uint32_t src = fe * W < 16 ? x : y;
                  f[ee] = __uint_as_float(src & (CM << ((fe * W) & 15)));
                }
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                  const float4 a4 = *reinterpret_cast<const float4 *>(sa + hh * D + cw + e);
                  float2 r = acc[hh][jw];
                  r = __ffma2_rn(make_float2(a4.x, a4.y), make_float2(f[0], f[1]), r);
                  r = __ffma2_rn(make_float2(a4.z, a4.w), make_float2(f[2], f[3]), r);
                  acc[hh][jw] = r;
                }
              }
            }
          }
        }
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
          const float a = ((acc[hh][0].x + acc[hh][0].y) + (acc[hh][1].x + acc[hh][1].y)) +
                          ((acc[hh][2].x + acc[hh][2].y) + (acc[hh][3].x + acc[hh][3].y));
          sc[hh] = lane < bt ? fmaf(a, pow2(kCarry), beta[hh]) : -INFINITY;
        }
      }
      float p[GQ];
      fold(sc, p);
      // value weights, lane = token: w' = p s 2^(149 - kCarry), u = p z
      if (lane < bt) {
        const __half *vs = reinterpret_cast<const __half *>(st + SG::VS) + lane * NJ;
        const __half *vz = reinterpret_cast<const __half *>(st + SG::VZ) + lane * NJ;
        // (w', u) of (head hh, value group j) at [(hh NJ + j) bt + token]
        for (int j = 0; j < NJ; ++j) {
          const float s = __half2float(vs[j]) * pow2(149 - kCarry);
          const float z = __half2float(vz[j]);
#pragma unroll
          for (int hh = 0; hh < GQ; ++hh)
            wu[(hh * NJ + j) * bt + lane] = make_float2(p[hh] * s, p[hh] * z);
        }
      }
      __syncwarp();
      // values: lane owns channels c0 ... c0 + CPL - 1 (value group j), its
      // CPL * W bits of each row from bit c0 * W; the token loop is unrolled
      // whole, so rows and weights are read at constant offsets
      constexpr int NB = CPL * W;
      const int c0 = lane * CPL;
      const unsigned char *vrow = st + SG::VC + ((c0 * W) >> 3);
      const float2 *wh[GQ];
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) wh[hh] = wu + (hh * NJ + jv) * bt;
#pragma unroll
      for (int jj = 0; jj < bt; ++jj) {
        uint32_t yv;
        if constexpr (NB == 32) yv = *reinterpret_cast<const uint32_t *>(vrow + jj * RB);
        else if constexpr (NB == 16) yv = *reinterpret_cast<const uint16_t *>(vrow + jj * RB);
        else if constexpr (NB == 8) yv = vrow[jj * RB];
        else yv = (uint32_t)vrow[jj * RB] >> ((c0 * W) & 7);
        const uint32_t yh = yv >> 16;
        float f[CPL];
#pragma unroll
        for (int u = 0; u < CPL; ++u)
          f[u] = __uint_as_float((u * W < 16 ? yv : yh) & (CM << ((u * W) & 15)));
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
          const float2 q2 = wh[hh][jj];
          // two channels per packed FMA
#pragma unroll
          for (int u = 0; u < CPL; u += 2) {
            const float2 r = __ffma2_rn(make_float2(q2.x, q2.x), make_float2(f[u], f[u + 1]),
                                        make_float2(o[hh][u], o[hh][u + 1]));
            o[hh][u] = r.x;
            o[hh][u + 1] = r.y;
          }
          zl[hh] += q2.y;
        }
      }
    };

    int s = 0;
    while (cc.x < XQ) {
      const bool ok = __all_sync(kFull, mbar_wait(&bars[s], (phase >> s) & 1u));
      if (!ok) { failed = true; break; }
      phase ^= 1u << s;
      pending &= ~(1u << s);
      const unsigned char *st = stage0 + s * SG::BYTES;
      const int w = cc.w;
      using I8 = std::integral_constant<int, 8>;
      using I16 = std::integral_constant<int, 16>;
      using I32 = std::integral_constant<int, 32>;
      if (w == 2) {
        if (g >= 32) block(std::integral_constant<int, 2>{}, I32{}, st, cc.first);
        else block(std::integral_constant<int, 2>{}, I16{}, st, cc.first);
      } else if (w == 4) {
        block(std::integral_constant<int, 4>{}, I16{}, st, cc.first);
      } else {
        block(std::integral_constant<int, 8>{}, I8{}, st, cc.first);
      }
      __syncwarp();
      if (pc.x < XQ) {
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
    // o at its true scale: 2^(kCarry - pos), plus the zero-point sums
    if (w_acc) {
#pragma unroll
      for (int u = 0; u < CPL; ++u) {
        const float f = pow2(kCarry - ((u * w_acc) & 15));
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) o[hh][u] = fmaf(o[hh][u], f, zl[hh]);
      }
    }
  }
  {
    // this warp's blocks of the fp16 residual window (block x = XQ + j is
    // window block j), folded into the running states after the groups (the
    // value sums are at true scale by now); lanes 0 ... kWinT - 1 score a
    // token each, lanes over channels sum the values
    int xw = x0;
    if (xw < XQ) xw += (XQ - xw + stride - 1) / stride * stride;
#pragma unroll 1
    for (; xw < XQ + nblk; xw += stride) {
      const int i0 = (xw - XQ) * kWinT;
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

  // the warp's (m, l, o) -> its a' region, then the CTA's log-sum-exp merge
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

struct AgeKernel {
  const void *f = nullptr;
  int smem = 0;          // dynamic shared memory the kernel needs
  int smem_static = 0;   // its static shared memory
  int occ = 0;           // CTAs per SM at smem
};

// the decode instance of (D, GQ) on the current device: its dynamic shared
// memory limit raised to the device's (so that a launch may pad its request
// to cap the CTAs per SM) and its occupancy, both set up once per device
template <int D, int GQ>
AgeKernel age_kernel() {
  static std::mutex mu;
  static std::atomic<uint64_t> done{0};
  static AgeKernel dev_k[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return {};
  if (!((done.load(std::memory_order_acquire) >> dev) & 1u)) {
    std::lock_guard<std::mutex> lock(mu);
    if (!((done.load(std::memory_order_relaxed) >> dev) & 1u)) {
      AgeKernel k;
      k.f = reinterpret_cast<const void *>(&k_decode_age<D, GQ>);
      k.smem = AgeSmem<D, GQ>::BYTES;
      cudaFuncAttributes fa;
      int optin = 0;
      if (cudaFuncGetAttributes(&fa, k.f) != cudaSuccess ||
          cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
              cudaSuccess ||
          cudaFuncSetAttribute(k.f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               optin - (int)fa.sharedSizeBytes) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k.occ, k.f, kThreads, k.smem) !=
              cudaSuccess)
        return {};
      k.smem_static = (int)fa.sharedSizeBytes;
      dev_k[dev] = k;
      done.fetch_or(1ull << dev, std::memory_order_release);
    }
  }
  return dev_k[dev];
}

// the instance for H_q / H_kv = gq at this D (f == nullptr: none)
template <int D>
AgeKernel pick(int gq) {
  switch (gq) {
    case 1: return age_kernel<D, 1>();
    case 2: return age_kernel<D, 2>();
    case 3: return age_kernel<D, 3>();
    case 4: return age_kernel<D, 4>();
    case 5: return age_kernel<D, 5>();
    case 6: return age_kernel<D, 6>();
    case 7: return age_kernel<D, 7>();
    case 8: return age_kernel<D, 8>();
    default: return {};
  }
}

AgeKernel pick_d64(int gq);
AgeKernel pick_d128(int gq);
constexpr int kDecodeThreads = kThreads;

}  // namespace agedec
}  // namespace vqk
