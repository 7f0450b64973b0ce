// Kitty: channel-wise mixed-precision keys (4-bit channels of high running
// variance, 2-bit for the rest) and fp16 values; its flush and its fused
// decode.
//
// Method: VeloxQuant-MLX changelog v0.11.0 "New" (Kitty: key channels ranked
// by online per-channel variance, the top 25% quantized in 4 bits and the
// rest in 2 bits with KIVI's asymmetric group quantization; values left at
// fp16) on the KIVI cache of v0.8.0 (key groups of g tokens per channel,
// fp16 residual window).  The ranking of a key group uses the running
// variance over the tokens up to the group's last one, computed exactly:
// every fp16 value is an integer multiple of 2^-24, so with m = x * 2^24
// the sums S1 = sum m (int64) and S2 = sum m^2 (a 128-bit integer) are
// exact and N S2 - S1^2 = N^2 var is compared as a 128-bit integer (N <=
// 2^20 keeps it below 2^120).  The smaller channel wins a tie.
#include "vqk_internal.cuh"

namespace vqk {
namespace {

typedef unsigned __int128 u128;

__device__ __forceinline__ int find_seq(const int32_t *prefix, int B, int item) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// fp16 bits -> the value in units of 2^-24 (exact)
__device__ __forceinline__ long long f16_units(unsigned short bits) {
  const int e = (bits >> 10) & 31;
  const long long m = bits & 1023;
  const long long v = e == 0 ? m : (m | 1024) << (e - 1);
  return (bits & 0x8000) ? -v : v;
}

// the fp16 row of token position p of (b, h) during a flush: the residual
// ring below src_split, the input rows above (as in the KIVI flush)
__device__ __forceinline__ const __half *src_row(const Geometry &geo, const Planes &pl,
                                                 const __half *in, int64_t in_stride,
                                                 size_t bh, int p, int split) {
  return p < split ? pl.Kr + (bh * geo.Rcap + (p % geo.Rcap)) * geo.D
                   : in + (bh * in_stride + (p - split)) * geo.D;
}

// One CTA of kRankThreads per (kv head, sequence): NS = kRankThreads / D
// slices of one thread per channel take NS consecutive groups of this
// flush at a time.  Each slice sums its group's keys (m and m^2 per
// channel, its rows' loads all in flight), the slices' sums are carried in
// shared memory (slice j adds slices 0 ... j to the running sums), and
// every slice ranks its channels by the running variance through its
// group's last token.
constexpr int kRankThreads = 1024;

__global__ void __launch_bounds__(kRankThreads)
k_kitty_rank(Geometry geo, Planes pl, const __half *__restrict__ Kin,
             int64_t in_stride, FlushTable tab) {
  extern __shared__ unsigned long long rsm[];
  const int D = geo.D, g = geo.g, NS = kRankThreads / D;
  const int c = threadIdx.x % D, sl = threadIdx.x / D;
  // per (slice, channel): the group's sums, then the running variance
  unsigned long long *q1 = rsm, *q2lo = q1 + NS * D, *q2hi = q2lo + NS * D;
  unsigned long long *vlo = q2hi + NS * D, *vhi = vlo + NS * D;
  const int h = blockIdx.x, b = blockIdx.y;
  const int n = tab.prefix[b + 1] - tab.prefix[b];
  if (n == 0) return;
  const size_t bh = (size_t)b * geo.H_kv + h;
  long long s1 = pl.ksum[bh * D + c];
  u128 s2 = ((u128)pl.ksq[(bh * D + c) * 2 + 1] << 64) | pl.ksq[(bh * D + c) * 2];
  const int split = tab.src_split[b];
  for (int k0 = 0; k0 < n; k0 += NS) {
    const int k = k0 + sl;
    const int P0 = tab.first_pos[b] + k * g;
    long long g1 = 0;
    u128 g2 = 0;
    if (k < n) {
#pragma unroll 8
      for (int i = 0; i < g; ++i) {
        const __half *row = src_row(geo, pl, Kin, in_stride, bh, P0 + i, split);
        const long long m = f16_units(__half_as_ushort(row[c]));
        g1 += m;
        g2 += (u128)((__int128)m * m);
      }
    }
    q1[sl * D + c] = (unsigned long long)g1;
    q2lo[sl * D + c] = (unsigned long long)g2;
    q2hi[sl * D + c] = (unsigned long long)(g2 >> 64);
    __syncthreads();
    // running sums through this slice's group (r), and through all NS
    // groups (the next step's start)
    long long r1 = 0;
    u128 r2 = 0;
    for (int j = 0; j < NS; ++j) {
      s1 += (long long)q1[j * D + c];
      s2 += ((u128)q2hi[j * D + c] << 64) | q2lo[j * D + c];
      if (j == sl) { r1 = s1; r2 = s2; }
    }
    u128 var = 0;
    if (k < n) {
      const u128 N = (u128)(P0 + g);
      const u128 a = (u128)(r1 < 0 ? -r1 : r1);
      var = N * r2 - a * a;
    }
    vlo[sl * D + c] = (unsigned long long)var;
    vhi[sl * D + c] = (unsigned long long)(var >> 64);
    __syncthreads();
    if (k < n) {
      int rank = 0;
      for (int o = 0; o < D; ++o) {
        const u128 vo = ((u128)vhi[sl * D + o] << 64) | vlo[sl * D + o];
        rank += (vo > var || (vo == var && o < c)) ? 1 : 0;
      }
      const unsigned word = __ballot_sync(0xffffffffu, rank < geo.kitty_hi);
      if ((c & 31) == 0)
        pl.kmask[(bh * (geo.Tcap / g) + P0 / g) * (D / 32) + (c >> 5)] = word;
    }
    __syncthreads();
  }
  if (sl == 0) {
    pl.ksum[bh * D + c] = s1;
    pl.ksq[(bh * D + c) * 2] = (unsigned long long)s2;
    pl.ksq[(bh * D + c) * 2 + 1] = (unsigned long long)(s2 >> 64);
  }
}

// One CTA per (group, kv head), one thread per channel: per channel a 4- or
// 2-bit group quantizer (fp32, IEEE, ties to even, as the KIVI flush), the
// codes OR-ed into the group's packed rows in shared memory (4- and 2-bit
// fields never straddle a 32-bit word), then the rows and the group's fp16
// values stored.
__global__ void k_flush_kitty(Geometry geo, Planes pl, const __half *__restrict__ Kin,
                              const __half *__restrict__ Vin, int64_t in_stride,
                              FlushTable tab) {
  extern __shared__ __align__(16) unsigned char ksm[];
  const int D = geo.D, g = geo.g, c = threadIdx.x;
  const int krow = (D + geo.kitty_hi) / 4;              // bytes per token row
  uint32_t *rows = reinterpret_cast<uint32_t *>(ksm);   // [g][krow / 4]
  const int item = blockIdx.x, h = blockIdx.y;
  const int b = find_seq(tab.prefix, geo.B, item);
  const int P0 = tab.first_pos[b] + (item - tab.prefix[b]) * g;
  const int split = tab.src_split[b];
  const size_t bh = (size_t)b * geo.H_kv + h;
  for (int i = c; i < g * krow / 4; i += blockDim.x) rows[i] = 0u;

  // this channel's width and bit offset within a row
  const uint32_t *mk = pl.kmask + (bh * (geo.Tcap / g) + P0 / g) * (D / 32);
  int below = 0;
  for (int w = 0; w < (c >> 5); ++w) below += __popc(mk[w]);
  const uint32_t mw = mk[c >> 5];
  below += __popc(mw & ((1u << (c & 31)) - 1u));
  const bool hi = (mw >> (c & 31)) & 1u;
  const int off = hi ? 4 * below : 4 * geo.kitty_hi + 2 * (c - below);
  const int levels = hi ? 15 : 3;
  __syncthreads();

  float mn = INFINITY, mx = -INFINITY;
  for (int i = 0; i < g; ++i) {
    const float x = __half2float(src_row(geo, pl, Kin, in_stride, bh, P0 + i, split)[c]);
    mn = fminf(mn, x);
    mx = fmaxf(mx, x);
  }
  mn = __fadd_rn(mn, 0.0f);   // a -0.0 minimum is stored as +0.0
  const float scale = __fdiv_rn(__fadd_rn(__fsub_rn(mx, mn), 0.0f), (float)levels);
  const size_t gi = (bh * (geo.Tcap / g) + P0 / g) * D + c;
  pl.Ks[gi] = __float2half_rn(scale);
  pl.Kz[gi] = __float2half_rn(mn);
  for (int i = 0; i < g; ++i) {
    uint32_t code = 0;
    if (scale != 0.0f) {
      const float x = __half2float(src_row(geo, pl, Kin, in_stride, bh, P0 + i, split)[c]);
      float r = rintf(__fdiv_rn(__fsub_rn(x, mn), scale));
      r = fminf(fmaxf(r, 0.0f), (float)levels);
      code = (uint32_t)r;
    }
    if (code) atomicOr(&rows[i * (krow / 4) + (off >> 5)], code << (off & 31));
  }
  __syncthreads();
  // the group's rows are contiguous: g * krow bytes (a multiple of 16)
  uint4 *dst = reinterpret_cast<uint4 *>(pl.Kc + (bh * geo.Tcap + P0) * krow);
  const uint4 *srow = reinterpret_cast<const uint4 *>(rows);
  for (int i = c; i < g * krow / 16; i += blockDim.x) dst[i] = srow[i];
  // the fp16 values of the group's tokens
  const int cpr = D / 8;
  for (int idx = c; idx < g * cpr; idx += blockDim.x) {
    const int i = idx / cpr, c8 = (idx - i * cpr) * 8;
    const int p = P0 + i;
    const __half *vs = p < split ? pl.Vr + (bh * geo.Rcap + (p % geo.Rcap)) * D
                                 : Vin + (bh * in_stride + (p - split)) * D;
    *reinterpret_cast<uint4 *>(pl.Vf + (bh * geo.Tcap + p) * D + c8) =
        *reinterpret_cast<const uint4 *>(vs + c8);
  }
}

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Fused decode over a Kitty cache: one CTA per (work item, kv head); each
// warp owns whole key groups and takes them in blocks of 32 tokens, one
// token per lane for the scores and all lanes over the channels for the
// values.  Scores: q . k_hat_t = sum_j a_j f_tj + beta, where f_tj is field
// j of token t's row (the 4-bit channels' codes, then the 2-bit ones) and
// a_j = q_c s_Gc of the channel c it belongs to: a is laid out in field
// order in shared memory once per group (and per query head), and each lane
// walks its own row's fields against it (broadcast reads).  Softmax: per
// block, the maximum and the sum over the warp, one rescale of the lane's
// output channels.  Values: the block's p_t passed by shuffles, the fp16
// rows read 8 bytes per lane (lane owns channels lane*CPL ...).  The fp16
// residual window is its own work item (one token per step).  Partials as
// the CUDA-core KIVI decode (launch_combine merges them).
template <int D, int GQ>
__global__ void __launch_bounds__(kThreads)
k_decode_kitty(Geometry geo, Planes pl, DecodeArgs args, DecodeTable tab) {
  constexpr int CPL = D / 32;   // GQ: query heads per kv head
  __shared__ float sq[GQ][D];
  __shared__ __align__(16) float sa[kWarps][GQ][D]; // a in field order
  __shared__ float sm[kWarps][GQ], sl[kWarps][GQ];
  __shared__ float so[kWarps][GQ][D];
  // the combine kernel behind this one waits for its completion
  asm volatile("griddepcontrol.launch_dependents;");
  const int item = blockIdx.x, h = blockIdx.y;
  const int b = find_seq(tab.prefix, geo.B, item);
  const int k = item - tab.prefix[b];
  constexpr int gq = GQ;
  const int g = geo.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const size_t bh = (size_t)b * geo.H_kv + h;
  const int HI = geo.kitty_hi;
  const int krow = (D + HI) / 4;                // bytes per row, a multiple of 4
  for (int i = threadIdx.x; i < GQ * D; i += kThreads) {
    const int hh = i / D, c = i % D;
    sq[hh][c] = __half2float(args.q[((size_t)b * geo.H_q + h * GQ + hh) * D + c]) *
                args.scale_log2;
  }
  __syncthreads();
  float m[GQ], l[GQ], o[GQ][CPL];
#pragma unroll
  for (int hh = 0; hh < GQ; ++hh) {
    m[hh] = -INFINITY; l[hh] = 0.f;
#pragma unroll
    for (int u = 0; u < CPL; ++u) o[hh][u] = 0.f;
  }
  // fold a block of scores (one per lane, -inf for absent tokens) of head
  // hh: returns this lane's weight
  auto block_softmax = [&](int hh, float s) {
    float mb = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
    const float mn = fmaxf(m[hh], mb);
    const float alpha = m[hh] == -INFINITY ? 0.f : exp2f(m[hh] - mn);
    const float p = s == -INFINITY ? 0.f : exp2f(s - mn);
    float ps = p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l[hh] = l[hh] * alpha + ps;
#pragma unroll
    for (int u = 0; u < CPL; ++u) o[hh][u] *= alpha;
    m[hh] = mn;
    return p;
  };

  if (k < tab.nq[b]) {
    const int t0 = k * args.tps, t1 = min(t0 + args.tps, tab.Tq[b]);
    const int bt = g < 32 ? g : 32;             // tokens per block
    for (int G = t0 / g + warp; G * g < t1; G += kWarps) {
      const size_t gidx = (bh * (geo.Tcap / g) + G) * D;
      const uint32_t *mk = pl.kmask + (bh * (geo.Tcap / g) + G) * (D / 32);
      // field index of each of the lane's channels
      int fj[CPL];
      float s_c[CPL], z_c[CPL];
#pragma unroll
      for (int u = 0; u < CPL; ++u) {
        const int c = lane * CPL + u;
        int below = 0;
        for (int w = 0; w < (c >> 5); ++w) below += __popc(mk[w]);
        const uint32_t mw = mk[c >> 5];
        below += __popc(mw & ((1u << (c & 31)) - 1u));
        fj[u] = ((mw >> (c & 31)) & 1u) ? below : HI + (c - below);
        s_c[u] = __half2float(pl.Ks[gidx + c]);
        z_c[u] = __half2float(pl.Kz[gidx + c]);
      }
      float beta[GQ];
      __syncwarp();
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) {
        float part = 0.f;
#pragma unroll
        for (int u = 0; u < CPL; ++u) {
          const float qc = sq[hh][lane * CPL + u];
          part = fmaf(qc, z_c[u], part);
          sa[warp][hh][fj[u]] = qc * s_c[u];
        }
        beta[hh] = warp_sum(part);
      }
      __syncwarp();
      for (int tb = G * g; tb < G * g + g; tb += bt) {
        float acc[GQ];
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) acc[hh] = 0.f;
        if (lane < bt) {
          const uint32_t *row = reinterpret_cast<const uint32_t *>(
              pl.Kc + (bh * geo.Tcap + tb + lane) * krow);
          // 4-bit fields: 8 per word
#pragma unroll 1
          for (int w = 0; w < HI / 8; ++w) {
            const uint32_t x = __ldg(row + w);
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) {
              const float4 a0 = *reinterpret_cast<const float4 *>(&sa[warp][hh][8 * w]);
              const float4 a1 = *reinterpret_cast<const float4 *>(&sa[warp][hh][8 * w + 4]);
              float r = acc[hh];
              r = fmaf(a0.x, (float)(x & 15u), r);
              r = fmaf(a0.y, (float)((x >> 4) & 15u), r);
              r = fmaf(a0.z, (float)((x >> 8) & 15u), r);
              r = fmaf(a0.w, (float)((x >> 12) & 15u), r);
              r = fmaf(a1.x, (float)((x >> 16) & 15u), r);
              r = fmaf(a1.y, (float)((x >> 20) & 15u), r);
              r = fmaf(a1.z, (float)((x >> 24) & 15u), r);
              r = fmaf(a1.w, (float)(x >> 28), r);
              acc[hh] = r;
            }
          }
          // 2-bit fields: 16 per word
#pragma unroll 1
          for (int w = 0; w < (D - HI) / 16; ++w) {
            const uint32_t x = __ldg(row + HI / 8 + w);
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) {
              const float *aw = &sa[warp][hh][HI + 16 * w];
              float r = acc[hh];
#pragma unroll
              for (int e = 0; e < 16; e += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(aw + e);
                r = fmaf(a4.x, (float)((x >> (2 * e)) & 3u), r);
                r = fmaf(a4.y, (float)((x >> (2 * e + 2)) & 3u), r);
                r = fmaf(a4.z, (float)((x >> (2 * e + 4)) & 3u), r);
                r = fmaf(a4.w, (float)((x >> (2 * e + 6)) & 3u), r);
              }
              acc[hh] = r;
            }
          }
        }
        float p[GQ];
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
          // online softmax over the block (written out here so that every
          // index of m, l, o stays a compile-time constant)
          const float s = lane < bt ? acc[hh] + beta[hh] : -INFINITY;
          float mb = s;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1)
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
          const float mn = fmaxf(m[hh], mb);
          const float alpha = m[hh] == -INFINITY ? 0.f : exp2f(m[hh] - mn);
          p[hh] = s == -INFINITY ? 0.f : exp2f(s - mn);
          const float ps = warp_sum(p[hh]);
          l[hh] = l[hh] * alpha + ps;
#pragma unroll
          for (int u = 0; u < CPL; ++u) o[hh][u] *= alpha;
          m[hh] = mn;
        }
        // values of the block's tokens
        const __half *vbase = pl.Vf + (bh * geo.Tcap + tb) * D + lane * CPL;
        // 8 rows in flight per lane: the loads of a block do not depend on
        // one another, only the accumulation does
#pragma unroll 8
        for (int j = 0; j < bt; ++j) {
          const __half *vr = vbase + (size_t)j * D;
          float v[CPL];
          if constexpr (CPL == 4) {
            const uint2 r = __ldg(reinterpret_cast<const uint2 *>(vr));
            const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
            const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
            v[0] = v01.x; v[1] = v01.y; v[2] = v23.x; v[3] = v23.y;
          } else {
#pragma unroll
            for (int u = 0; u < CPL; ++u) v[u] = __half2float(vr[u]);
          }
#pragma unroll
          for (int hh = 0; hh < GQ; ++hh) {
            const float pj = __shfl_sync(0xffffffffu, p[hh], j);
#pragma unroll
            for (int u = 0; u < CPL; ++u) o[hh][u] = fmaf(pj, v[u], o[hh][u]);
          }
        }
      }
    }
  } else {
    const int Tq = tab.Tq[b];
    for (int i0 = warp * 32; i0 < tab.nres[b]; i0 += kWarps * 32) {
      // a block of up to 32 residual tokens: lane i scores token Tq + i0 + i
      const int i = i0 + lane;
      const bool ok = i < tab.nres[b];
      const int slot = (Tq + (ok ? i : i0)) % geo.Rcap;
      const __half *kr = pl.Kr + (bh * geo.Rcap + slot) * D;
      float acc[GQ];
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) acc[hh] = 0.f;
#pragma unroll 4
      for (int c = 0; c < D; c += 2) {
        const float2 kv = __half22float2(*reinterpret_cast<const __half2 *>(kr + c));
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh)
          acc[hh] = fmaf(sq[hh][c], kv.x, fmaf(sq[hh][c + 1], kv.y, acc[hh]));
      }
      float p[GQ];
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) p[hh] = block_softmax(hh, ok ? acc[hh] : -INFINITY);
      const int nb = min(32, tab.nres[b] - i0);
      for (int j = 0; j < nb; ++j) {
        const __half *vr = pl.Vr + (bh * geo.Rcap + (Tq + i0 + j) % geo.Rcap) * D + lane * CPL;
        float v[CPL];
#pragma unroll
        for (int u = 0; u < CPL; ++u) v[u] = __half2float(vr[u]);
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
          const float pj = __shfl_sync(0xffffffffu, p[hh], j);
#pragma unroll
          for (int u = 0; u < CPL; ++u) o[hh][u] = fmaf(pj, v[u], o[hh][u]);
        }
      }
    }
  }

#pragma unroll
  for (int hh = 0; hh < GQ; ++hh) {
    if (hh >= gq) break;
    if (lane == 0) { sm[warp][hh] = m[hh]; sl[warp][hh] = l[hh]; }
#pragma unroll
    for (int u = 0; u < CPL; ++u) so[warp][hh][lane * CPL + u] = o[hh][u];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < gq * (D + 2); i += kThreads) {
    const int hh = i / (D + 2), c = i % (D + 2);
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm[w][hh]);
    float acc = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      const float f = sm[w][hh] == -INFINITY ? 0.f : exp2f(sm[w][hh] - M);
      acc += f * (c < D ? so[w][hh][c] : sl[w][hh]);
    }
    const int hq = h * gq + hh;
    float *dst = pl.part + (((size_t)b * geo.H_q + hq) * geo.max_items + k) * (D + 2);
    dst[c] = c == D ? M : acc;
  }
}

}  // namespace

cudaError_t launch_flush_kitty(const Geometry &geo, const Planes &pl,
                               const __half *Kin, const __half *Vin,
                               int64_t in_stride, const FlushTable &tab,
                               int total_groups, cudaStream_t st) {
  if (total_groups <= 0) return cudaSuccess;
  const size_t rsmem = (size_t)5 * kRankThreads * sizeof(unsigned long long);
  if (rsmem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_kitty_rank, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)rsmem);
    if (e != cudaSuccess) return e;
  }
  k_kitty_rank<<<dim3(geo.H_kv, geo.B), kRankThreads, rsmem, st>>>(geo, pl, Kin, in_stride, tab);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)geo.g * (geo.D + geo.kitty_hi) / 4;
  k_flush_kitty<<<dim3(total_groups, geo.H_kv), geo.D, smem, st>>>(geo, pl, Kin, Vin,
                                                                   in_stride, tab);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_decode_kitty(const Geometry &geo, const Planes &pl,
                                const DecodeArgs &args, const DecodeTable &tab,
                                cudaStream_t st) {
  if (args.total_items > 0) {
    dim3 grid(args.total_items, geo.H_kv);
    const int gq = geo.H_q / geo.H_kv;
#define VQK_KITTY(DD, QQ)                                                   \
  if (geo.D == DD && gq == QQ) {                                            \
    k_decode_kitty<DD, QQ><<<grid, kThreads, 0, st>>>(geo, pl, args, tab); \
  } else
#define VQK_KITTY_D(DD) VQK_KITTY(DD, 1) VQK_KITTY(DD, 2) VQK_KITTY(DD, 3)  \
  VQK_KITTY(DD, 4) VQK_KITTY(DD, 5) VQK_KITTY(DD, 6) VQK_KITTY(DD, 7)       \
  VQK_KITTY(DD, 8)
    VQK_KITTY_D(64) VQK_KITTY_D(128)
    { return cudaErrorInvalidValue; }
#undef VQK_KITTY_D
#undef VQK_KITTY
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_combine(geo, pl, args, tab, st);
}

}  // namespace vqk
