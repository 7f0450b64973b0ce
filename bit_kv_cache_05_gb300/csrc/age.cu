// AgeTieredKV: quantization width by token age (three tiers of the KIVI
// group quantizer), its flush (quantize and demote) and its fused decode.
//
// Method: VeloxQuant-MLX method overview, AgeTieredKV entry (three tiers,
// default 8 / 4 / 2 bits, chosen by current position minus token position
// against two boundaries, default 128 and 1024 tokens; the shared min/max
// group quantizer of KIVI), on the KIVI cache of changelog v0.8.0 (keys per
// channel over g tokens, values per token over g channels).  A group's age
// counts from its newest token; a group enters at the top tier and moves
// down one tier at a time, re-quantized from its values rebuilt in fp32
// (code * scale rounded, then + zero rounded), so that a prefill and any
// chunking of appends give the same cache.  Rows are D bytes (the widest
// tier); a group's codes fill the leading D * bits / 8 bytes, packed LSB
// first, the rest zero.
#include <type_traits>

#include "vqk_internal.cuh"

namespace vqk {
namespace {

__device__ __forceinline__ int find_seq(const int32_t *prefix, int B, int item) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// the group quantizer on fp32 inputs (IEEE, ties to even, as the KIVI flush)
__device__ __forceinline__ void group_params(float mn, float mx, int levels,
                                             float &zero, float &scale) {
  zero = __fadd_rn(mn, 0.0f);                       // -0.0 -> +0.0
  scale = __fdiv_rn(__fadd_rn(__fsub_rn(mx, zero), 0.0f), (float)levels);
}
__device__ __forceinline__ uint32_t group_code(float x, float zero, float scale,
                                               int levels) {
  if (scale == 0.0f) return 0u;
  float r = rintf(__fdiv_rn(__fsub_rn(x, zero), scale));
  return (uint32_t)fminf(fmaxf(r, 0.0f), (float)levels);
}

// One CTA per (item, kv head), one thread per channel (D threads).  Item:
// a new group (from fp16, to its tier) or a stored group (from its old tier
// to its new one).  The group's keys and values are held in fp32 in shared
// memory; each step quantizes them at the next tier's width (keys per
// channel: thread c; values per token and channel group: thread (i, j)) and,
// unless it is the last step, rebuilds them from the codes.
__global__ void k_age_flush(Geometry geo, Planes pl, const __half *__restrict__ Kin,
                            const __half *__restrict__ Vin, int64_t in_stride,
                            AgeTable tab) {
  extern __shared__ __align__(16) unsigned char asmem[];
  const int D = geo.D, g = geo.g, c = threadIdx.x, NJ = D / g;
  float *xk = reinterpret_cast<float *>(asmem);           // [g][D]
  float *xv = xk + g * D;                                  // [g][D]
  uint8_t *ck = reinterpret_cast<uint8_t *>(xv + g * D);   // [g][D]
  uint8_t *cv = ck + g * D;                                // [g][D]
  const int item = blockIdx.x, h = blockIdx.y;
  const int b = find_seq(tab.prefix, geo.B, item);
  const int local = item - tab.prefix[b];
  const int nnew = tab.gn1[b] - tab.gn0[b];
  const bool fresh = local < nnew;
  const int G = fresh ? tab.gn0[b] + local : tab.gd0[b] + (local - nnew);
  const int t_to = age_tier(geo, tab.S_new[b], G);
  int t = fresh ? -1 : age_tier(geo, tab.S_old[b], G);
  if (t >= t_to) return;                                   // no move for this group
  const size_t bh = (size_t)b * geo.H_kv + h;
  const size_t kg = (bh * (geo.Tcap / g) + G) * D;         // key scale/zero row
  const size_t r0 = bh * geo.Tcap + (size_t)G * g;         // first token row

  // ---- load the group in fp32 ----
  if (fresh) {
    const int split = tab.src_split[b];
    for (int idx = c; idx < g * D; idx += blockDim.x) {
      const int i = idx / D, ch = idx - i * D;
      const int p = G * g + i;
      const size_t src = p < split ? (bh * geo.Rcap + (p % geo.Rcap)) * D + ch
                                   : (bh * in_stride + (p - split)) * D + ch;
      xk[idx] = __half2float(p < split ? pl.Kr[src] : Kin[src]);
      xv[idx] = __half2float(p < split ? pl.Vr[src] : Vin[src]);
    }
  } else {
    const int w = geo.age_bits[t];
    const uint32_t m = (1u << w) - 1u;
    for (int idx = c; idx < g * D; idx += blockDim.x) {
      const int i = idx / D, ch = idx - i * D;
      const int bit = ch * w;
      const uint8_t kb = pl.Kc[(r0 + i) * D + (bit >> 3)];
      const uint8_t vb = pl.Vc[(r0 + i) * D + (bit >> 3)];
      const float kcode = (float)((kb >> (bit & 7)) & m);
      const float vcode = (float)((vb >> (bit & 7)) & m);
      xk[idx] = __fadd_rn(__fmul_rn(kcode, __half2float(pl.Ks[kg + ch])),
                          __half2float(pl.Kz[kg + ch]));
      const size_t vi = (r0 + i) * NJ + ch / g;
      xv[idx] = __fadd_rn(__fmul_rn(vcode, __half2float(pl.Vs[vi])),
                          __half2float(pl.Vz[vi]));
    }
  }
  __syncthreads();

  // ---- the chain of tiers ----
  float kzero = 0.f, kscale = 0.f, vzero = 0.f, vscale = 0.f;
  const int vi_tok = c / NJ, vi_grp = c - (c / NJ) * NJ;   // thread's value group
  while (t < t_to) {
    ++t;
    const int levels = (1 << geo.age_bits[t]) - 1;
    // keys: channel c over the g tokens
    {
      float mn = INFINITY, mx = -INFINITY;
      for (int i = 0; i < g; ++i) {
        mn = fminf(mn, xk[i * D + c]);
        mx = fmaxf(mx, xk[i * D + c]);
      }
      group_params(mn, mx, levels, kzero, kscale);
      for (int i = 0; i < g; ++i) ck[i * D + c] = (uint8_t)group_code(xk[i * D + c], kzero, kscale, levels);
    }
    // values: token vi_tok, channels vi_grp*g ... +g-1
    {
      const float *row = xv + vi_tok * D + vi_grp * g;
      float mn = INFINITY, mx = -INFINITY;
      for (int k = 0; k < g; ++k) {
        mn = fminf(mn, row[k]);
        mx = fmaxf(mx, row[k]);
      }
      group_params(mn, mx, levels, vzero, vscale);
      for (int k = 0; k < g; ++k)
        cv[vi_tok * D + vi_grp * g + k] = (uint8_t)group_code(row[k], vzero, vscale, levels);
    }
    __syncthreads();
    if (t < t_to) {
      // rebuild in fp32 from the stored (fp16) scale and zero
      const float ks16 = __half2float(__float2half_rn(kscale));
      const float kz16 = __half2float(__float2half_rn(kzero));
      for (int i = 0; i < g; ++i)
        xk[i * D + c] = __fadd_rn(__fmul_rn((float)ck[i * D + c], ks16), kz16);
      const float vs16 = __half2float(__float2half_rn(vscale));
      const float vz16 = __half2float(__float2half_rn(vzero));
      for (int k = 0; k < g; ++k) {
        const int at = vi_tok * D + vi_grp * g + k;
        xv[at] = __fadd_rn(__fmul_rn((float)cv[at], vs16), vz16);
      }
      __syncthreads();
    }
  }

  // ---- store: scales, zeros, rows at the final width ----
  pl.Ks[kg + c] = __float2half_rn(kscale);
  pl.Kz[kg + c] = __float2half_rn(kzero);
  pl.Vs[(r0 + vi_tok) * NJ + vi_grp] = __float2half_rn(vscale);
  pl.Vz[(r0 + vi_tok) * NJ + vi_grp] = __float2half_rn(vzero);
  const int w = geo.age_bits[t_to];
  const int per = 32 / w, words = D / 4;                   // 32-bit words per row
  for (int idx = c; idx < g * words; idx += blockDim.x) {
    const int i = idx / words, k = idx - i * words;
    uint32_t ak = 0, av = 0;
    if (k < D * w / 32) {
      for (int e = 0; e < per; ++e) {
        ak |= (uint32_t)ck[i * D + k * per + e] << (w * e);
        av |= (uint32_t)cv[i * D + k * per + e] << (w * e);
      }
    }
    reinterpret_cast<uint32_t *>(pl.Kc + (r0 + i) * D)[k] = ak;
    reinterpret_cast<uint32_t *>(pl.Vc + (r0 + i) * D)[k] = av;
  }
  if (c == 0) pl.tier[bh * (geo.Tcap / g) + G] = (int8_t)t_to;
}

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Fused decode over an age-tiered cache: one CTA per (work item, kv head);
// each warp owns whole key groups, in blocks of up to 32 tokens: one token
// per lane for the scores (q'.s per channel in shared memory, the lane's
// row read at the group's width), a per-block online softmax, then the
// values with the lane owning channels lane*CPL ...: the weighted code sums
// sum_t p_t s_t,j code_t,c and the zero-point sums sum_t p_t z_t,j.
template <int D, int GQ>
__global__ void __launch_bounds__(kThreads)
k_decode_age(Geometry geo, Planes pl, DecodeArgs args, DecodeTable tab) {
  constexpr int CPL = D / 32;
  __shared__ float sq[GQ][D];
  __shared__ __align__(16) float sa[kWarps][GQ][D];
  __shared__ float sm[kWarps][GQ], sl[kWarps][GQ];
  __shared__ float so[kWarps][GQ][D];
  const int item = blockIdx.x, h = blockIdx.y;
  const int b = find_seq(tab.prefix, geo.B, item);
  const int k = item - tab.prefix[b];
  const int g = geo.g, NJ = D / g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const size_t bh = (size_t)b * geo.H_kv + h;
  const int S = tab.Tq[b] + tab.nres[b];
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
  // online softmax of a block (one score per lane, -inf when absent);
  // returns the lane's weight
  auto fold = [&](float (&s)[GQ], float (&p)[GQ]) {
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
      float mb = s[hh];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
      const float mn = fmaxf(m[hh], mb);
      const float alpha = m[hh] == -INFINITY ? 0.f : exp2f(m[hh] - mn);
      p[hh] = s[hh] == -INFINITY ? 0.f : exp2f(s[hh] - mn);
      l[hh] = l[hh] * alpha + warp_sum(p[hh]);
#pragma unroll
      for (int u = 0; u < CPL; ++u) o[hh][u] *= alpha;
      m[hh] = mn;
    }
  };

  if (k < tab.nq[b]) {
    const int t0 = k * args.tps, t1 = min(t0 + args.tps, tab.Tq[b]);
    const int bt = g < 32 ? g : 32;
    for (int G = t0 / g + warp; G * g < t1; G += kWarps) {
      const int w = geo.age_bits[age_tier(geo, S, G)];
      const uint32_t cm = (1u << w) - 1u;
      const size_t gidx = (bh * (geo.Tcap / g) + G) * D;
      float beta[GQ];
      __syncwarp();
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) {
        float part = 0.f;
#pragma unroll
        for (int u = 0; u < CPL; ++u) {
          const int c = lane * CPL + u;
          const float qc = sq[hh][c];
          part = fmaf(qc, __half2float(pl.Kz[gidx + c]), part);
          sa[warp][hh][c] = qc * __half2float(pl.Ks[gidx + c]);
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
              pl.Kc + (bh * geo.Tcap + tb + lane) * D);
          // the lane's row at the group's width, the field loop unrolled per
          // width
          auto walk = [&](auto w_tag) {
            constexpr int W = decltype(w_tag)::value, PER = 32 / W;
            constexpr uint32_t CM = (1u << W) - 1u;
#pragma unroll 2
            for (int wi = 0; wi < D * W / 32; ++wi) {
              const uint32_t x = __ldg(row + wi);
#pragma unroll
              for (int e = 0; e < PER; e += 4) {
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                  const float4 a4 = *reinterpret_cast<const float4 *>(&sa[warp][hh][wi * PER + e]);
                  float r = acc[hh];
                  r = fmaf(a4.x, (float)((x >> (W * e)) & CM), r);
                  r = fmaf(a4.y, (float)((x >> (W * (e + 1))) & CM), r);
                  r = fmaf(a4.z, (float)((x >> (W * (e + 2))) & CM), r);
                  r = fmaf(a4.w, (float)((x >> (W * (e + 3))) & CM), r);
                  acc[hh] = r;
                }
              }
            }
          };
          if (w == 2) walk(std::integral_constant<int, 2>{});
          else if (w == 4) walk(std::integral_constant<int, 4>{});
          else walk(std::integral_constant<int, 8>{});
        }
        float s[GQ], p[GQ];
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) s[hh] = lane < bt ? acc[hh] + beta[hh] : -INFINITY;
        fold(s, p);
        // values: o_c += sum_t p_t (code_tc s_tj + z_tj)
        const int c0 = lane * CPL, j = c0 / g;
#pragma unroll 8
        for (int jj = 0; jj < bt; ++jj) {
          const size_t r = bh * geo.Tcap + tb + jj;
          const float vs = __half2float(pl.Vs[r * NJ + j]);
          const float vz = __half2float(pl.Vz[r * NJ + j]);
          // the lane's CPL codes: CPL * w bits at bit c0 * w of the row
          const int bit = c0 * w;
          uint32_t x;
          if (CPL * w <= 8) x = pl.Vc[r * D + (bit >> 3)] >> (bit & 7);
          else if (CPL * w <= 16) x = *reinterpret_cast<const uint16_t *>(pl.Vc + r * D + (bit >> 3));
          else x = *reinterpret_cast<const uint32_t *>(pl.Vc + r * D + (bit >> 3));
          float v[CPL];
#pragma unroll
          for (int u = 0; u < CPL; ++u) v[u] = fmaf((float)((x >> (w * u)) & cm), vs, vz);
#pragma unroll
          for (int hh = 0; hh < GQ; ++hh) {
            const float pj = __shfl_sync(0xffffffffu, p[hh], jj);
#pragma unroll
            for (int u = 0; u < CPL; ++u) o[hh][u] = fmaf(pj, v[u], o[hh][u]);
          }
        }
      }
    }
  } else {
    const int Tq = tab.Tq[b];
    for (int i0 = warp * 32; i0 < tab.nres[b]; i0 += kWarps * 32) {
      const int i = i0 + lane;
      const bool ok = i < tab.nres[b];
      const __half *kr = pl.Kr + (bh * geo.Rcap + (Tq + (ok ? i : i0)) % geo.Rcap) * D;
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
      float s[GQ], p[GQ];
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) s[hh] = ok ? acc[hh] : -INFINITY;
      fold(s, p);
      const int nb = min(32, tab.nres[b] - i0);
      for (int jj = 0; jj < nb; ++jj) {
        const __half *vr = pl.Vr + (bh * geo.Rcap + (Tq + i0 + jj) % geo.Rcap) * D + lane * CPL;
        float v[CPL];
#pragma unroll
        for (int u = 0; u < CPL; ++u) v[u] = __half2float(vr[u]);
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
          const float pj = __shfl_sync(0xffffffffu, p[hh], jj);
#pragma unroll
          for (int u = 0; u < CPL; ++u) o[hh][u] = fmaf(pj, v[u], o[hh][u]);
        }
      }
    }
  }

#pragma unroll
  for (int hh = 0; hh < GQ; ++hh) {
    if (lane == 0) { sm[warp][hh] = m[hh]; sl[warp][hh] = l[hh]; }
#pragma unroll
    for (int u = 0; u < CPL; ++u) so[warp][hh][lane * CPL + u] = o[hh][u];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < GQ * (D + 2); i += kThreads) {
    const int hh = i / (D + 2), c = i % (D + 2);
    float M = -INFINITY;
    for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, sm[ww][hh]);
    float acc = 0.f;
    for (int ww = 0; ww < kWarps; ++ww) {
      const float f = sm[ww][hh] == -INFINITY ? 0.f : exp2f(sm[ww][hh] - M);
      acc += f * (c < D ? so[ww][hh][c] : sl[ww][hh]);
    }
    const int hq = h * GQ + hh;
    float *dst = pl.part + (((size_t)b * geo.H_q + hq) * geo.max_items + k) * (D + 2);
    dst[c] = c == D ? M : acc;
  }
}

}  // namespace

cudaError_t launch_age_flush(const Geometry &geo, const Planes &pl,
                             const __half *Kin, const __half *Vin,
                             int64_t in_stride, const AgeTable &tab,
                             cudaStream_t st) {
  const int items = tab.prefix[geo.B];
  if (items <= 0) return cudaSuccess;
  const size_t smem = (size_t)geo.g * geo.D * (4 + 4 + 1 + 1);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_age_flush,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  k_age_flush<<<dim3(items, geo.H_kv), geo.D, smem, st>>>(geo, pl, Kin, Vin, in_stride, tab);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_decode_age(const Geometry &geo, const Planes &pl,
                              const DecodeArgs &args, const DecodeTable &tab,
                              cudaStream_t st) {
  if (args.total_items > 0) {
    dim3 grid(args.total_items, geo.H_kv);
    const int gq = geo.H_q / geo.H_kv;
#define VQK_AGE(DD, QQ)                                                   \
  if (geo.D == DD && gq == QQ) {                                          \
    k_decode_age<DD, QQ><<<grid, kThreads, 0, st>>>(geo, pl, args, tab); \
  } else
#define VQK_AGE_D(DD) VQK_AGE(DD, 1) VQK_AGE(DD, 2) VQK_AGE(DD, 3) VQK_AGE(DD, 4) \
  VQK_AGE(DD, 5) VQK_AGE(DD, 6) VQK_AGE(DD, 7) VQK_AGE(DD, 8)
    VQK_AGE_D(64) VQK_AGE_D(128)
    { return cudaErrorInvalidValue; }
#undef VQK_AGE_D
#undef VQK_AGE
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_combine(geo, pl, args, tab, st);
}

}  // namespace vqk
