// Fused decode step over the quantized cache: split-KV online softmax with
// k_hat / v_hat rebuilt in registers, then a log-sum-exp merge of the splits.
//
// Method: VeloxQuant-MLX changelog v0.42.0 "Added" (scalar_fused_decode_attend:
// SDP attention directly over the group-affine cache, k_hat/v_hat rebuilt
// in-register inside a FlashAttention-style online softmax with fp32
// accumulation, no dequantized K/V written to memory).
//
// Algebra used here (all fp32):
//   key group G, channel c:  k_hat = code * s_Gc + z_Gc, so
//     q . k_hat_t = sum_c (q_c s_Gc) code_tc + sum_c q_c z_Gc = a_G . code_t + beta_G
//   value token t, channel group j:  v_hat = code * s_tj + z_tj.
// Scores are kept in base 2: s2 = scale * log2(e) * q . k_hat.
#include "vqk_internal.cuh"

namespace vqk {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ int find_seq(const int32_t *prefix, int B,
                                        int item) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

template <int BITS>
__device__ __forceinline__ float code_at(const uint8_t *row, int c) {
  const int bit = c * BITS;
  return (float)((row[bit >> 3] >> (bit & 7)) & ((1 << BITS) - 1));
}

// One block per (work item, kv head).  Each warp owns whole key groups (or
// residual tokens) and keeps its own (m, l, o) per query head; lane owns
// channels [lane*CPL, lane*CPL + CPL).
template <int D, int BITS>
__global__ void __launch_bounds__(kThreads)
k_decode_split(Geometry geo, Planes pl, DecodeArgs args, DecodeTable tab) {
  constexpr int CPL = D / 32;
  constexpr int GQ = kMaxGroupHeads;
  __shared__ float sq[GQ][D];
  __shared__ float sm[kWarps][GQ], sl[kWarps][GQ];
  __shared__ float so[kWarps][GQ][D];
  // the combine kernel behind this one waits for its completion
  asm volatile("griddepcontrol.launch_dependents;");

  const int item = blockIdx.x, h = blockIdx.y;
  const int b = find_seq(tab.prefix, geo.B, item);
  const int k = item - tab.prefix[b];
  const int gq = geo.H_q / geo.H_kv;
  const int g = geo.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const size_t bh = (size_t)b * geo.H_kv + h;

  for (int i = threadIdx.x; i < gq * D; i += kThreads) {
    const int hh = i / D, c = i % D;
    sq[hh][c] = __half2float(args.q[((size_t)b * geo.H_q + h * gq + hh) * D + c]);
  }
  __syncthreads();

  float m[GQ], l[GQ], o[GQ][CPL];
#pragma unroll
  for (int hh = 0; hh < GQ; ++hh) {
    m[hh] = -INFINITY; l[hh] = 0.f;
#pragma unroll
    for (int u = 0; u < CPL; ++u) o[hh][u] = 0.f;
  }

  auto online = [&](int hh, float s2, const float *v) {
    const float mn = fmaxf(m[hh], s2);
    const float alpha = exp2f(m[hh] - mn);
    const float p = exp2f(s2 - mn);
    l[hh] = l[hh] * alpha + p;
#pragma unroll
    for (int u = 0; u < CPL; ++u) o[hh][u] = o[hh][u] * alpha + p * v[u];
    m[hh] = mn;
  };

  // KIVI-Sink: the sinks of this (b, h); a sink of the quantized region is
  // read from its fp16 rows
  __shared__ int ssk[kMaxSink];
  const int nsk = geo.n_sink;
  if (nsk > 0) {
    if (threadIdx.x < nsk) ssk[threadIdx.x] = pl.sink_pos[bh * nsk + threadIdx.x];
    __syncthreads();
  }

  if (k < tab.nq[b]) {
    const int t0 = k * args.tps;
    const int t1 = min(t0 + args.tps, tab.Tq[b]);
    const int ngrp = D / g;
    for (int G = t0 / g + warp; G * g < t1; G += kWarps) {
      const size_t gidx = (bh * (geo.Tcap / g) + G) * D;
      float a[GQ][CPL], beta[GQ];
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) {
        float part = 0.f;
#pragma unroll
        for (int u = 0; u < CPL; ++u) {
          const int c = lane * CPL + u;
          const float s = __half2float(pl.Ks[gidx + c]);
          const float z = __half2float(pl.Kz[gidx + c]);
          const float qc = hh < gq ? sq[hh][c] : 0.f;
          a[hh][u] = qc * s;
          part += qc * z;
        }
        beta[hh] = warp_sum(part);
      }
      for (int t = G * g; t < G * g + g; ++t) {
        int slot = -1;
        for (int j = 0; j < nsk; ++j)
          if (ssk[j] == t) slot = j;
        if (slot >= 0) {
          const __half *kr = pl.sink_k + (bh * nsk + slot) * D;
          const __half *vr = pl.sink_v + (bh * nsk + slot) * D;
          float kv[CPL], v[CPL];
#pragma unroll
          for (int u = 0; u < CPL; ++u) {
            kv[u] = __half2float(kr[lane * CPL + u]);
            v[u] = __half2float(vr[lane * CPL + u]);
          }
#pragma unroll
          for (int hh = 0; hh < GQ; ++hh) {
            if (hh >= gq) break;
            float part = 0.f;
#pragma unroll
            for (int u = 0; u < CPL; ++u) part += sq[hh][lane * CPL + u] * kv[u];
            online(hh, warp_sum(part) * args.scale_log2, v);
          }
          continue;
        }
        const uint8_t *krow = pl.Kc + (bh * geo.Tcap + t) * geo.row;
        const uint8_t *vrow = pl.Vc + (bh * geo.Tcap + t) * geo.row;
        float kc[CPL], v[CPL];
#pragma unroll
        for (int u = 0; u < CPL; ++u) {
          const int c = lane * CPL + u;
          kc[u] = code_at<BITS>(krow, c);
          const size_t vi = (bh * geo.Tcap + t) * ngrp + c / g;
          v[u] = code_at<BITS>(vrow, c) * __half2float(pl.Vs[vi]) +
                 __half2float(pl.Vz[vi]);
        }
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
          if (hh >= gq) break;
          float part = 0.f;
#pragma unroll
          for (int u = 0; u < CPL; ++u) part += a[hh][u] * kc[u];
          const float s2 = (warp_sum(part) + beta[hh]) * args.scale_log2;
          online(hh, s2, v);
        }
      }
    }
  } else {
    const int Tq = tab.Tq[b];
    for (int i = warp; i < tab.nres[b]; i += kWarps) {
      const int slot = (Tq + i) % geo.Rcap;
      const __half *kr = pl.Kr + (bh * geo.Rcap + slot) * D;
      const __half *vr = pl.Vr + (bh * geo.Rcap + slot) * D;
      float kv[CPL], v[CPL];
#pragma unroll
      for (int u = 0; u < CPL; ++u) {
        kv[u] = __half2float(kr[lane * CPL + u]);
        v[u] = __half2float(vr[lane * CPL + u]);
      }
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) {
        if (hh >= gq) break;
        float part = 0.f;
#pragma unroll
        for (int u = 0; u < CPL; ++u) part += sq[hh][lane * CPL + u] * kv[u];
        online(hh, warp_sum(part) * args.scale_log2, v);
      }
    }
  }

  // merge the warps' states and write this item's partial per query head
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
    dst[c] = c == D ? M : (c == D + 1 ? acc : acc);
  }
}

// out[b][hq] = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k over the n
// split partials of (b, hq).  Launched as a programmatic dependent of the
// decode kernel (which releases it early): it waits for the partials, reads
// the n (m_k, l_k) pairs at once and builds the weights 2^(m_k - M) in
// shared memory; then warp w sums the partial rows w, w + 8, ... (lanes
// over channel pairs, four rows in flight per warp) and the warps' sums are
// added in shared memory.
constexpr int kCombineWarps = 8;
constexpr int kCombineThreads = kCombineWarps * 32;

__device__ __forceinline__ float block_reduce(float v, bool is_max, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float x = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, x) : v + x;
  }
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[0];
  for (int w = 1; w < kCombineWarps; ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
  __syncthreads();
  return v;
}

__global__ void __launch_bounds__(kCombineThreads)
k_combine(Geometry geo, Planes pl, DecodeArgs args, DecodeTable tab) {
  extern __shared__ float csm[];   // weights [max_items], then [8][D] sums
  __shared__ float red[kCombineWarps];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int b = blockIdx.x / geo.H_q, hq = blockIdx.x % geo.H_q;
  const int D = geo.D, P = D + 2, PPL = D / 64;   // channel pairs per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float *fw = csm;
  float *ws = csm + ((geo.max_items + 1) & ~1);   // 8-byte aligned
  const int n = tab.prefix[b + 1] - tab.prefix[b];
  const float *base = pl.part + ((size_t)b * geo.H_q + hq) * geo.max_items * P;
  float mloc = -INFINITY;
  for (int k = threadIdx.x; k < n; k += kCombineThreads) {
    fw[k] = __ldcg(base + (size_t)k * P + D);
    mloc = fmaxf(mloc, fw[k]);
  }
  const float M = block_reduce(mloc, true, red);
  float lloc = 0.f;
  for (int k = threadIdx.x; k < n; k += kCombineThreads) {
    const float f = fw[k] == -INFINITY ? 0.f : exp2f(fw[k] - M);
    lloc += f * __ldcg(base + (size_t)k * P + D + 1);
    fw[k] = f;
  }
  const float L = block_reduce(lloc, false, red);   // its barriers publish fw
  float2 acc[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) acc[p] = make_float2(0.f, 0.f);
  for (int k0 = warp; k0 < n; k0 += 4 * kCombineWarps) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = k0 + u * kCombineWarps;
      if (k < n) {
        const float f = fw[k];
        const float2 *row = reinterpret_cast<const float2 *>(base + (size_t)k * P);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          if (p < PPL) {
            const float2 v = __ldcg(row + lane + 32 * p);
            acc[p].x = fmaf(f, v.x, acc[p].x);
            acc[p].y = fmaf(f, v.y, acc[p].y);
          }
        }
      }
    }
  }
#pragma unroll
  for (int p = 0; p < 4; ++p)
    if (p < PPL) reinterpret_cast<float2 *>(ws + warp * D)[lane + 32 * p] = acc[p];
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += kCombineThreads) {
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) o += ws[w * D + c];
    args.out[((size_t)b * geo.H_q + hq) * D + c] = n ? o / L : 0.f;
  }
}

}  // namespace

cudaError_t launch_decode(const Geometry &geo, const Planes &pl,
                          const DecodeArgs &args, const DecodeTable &tab,
                          cudaStream_t st) {
  if (geo.kitty) return launch_decode_kitty(geo, pl, args, tab, st);
  if (geo.age_b1 > 0) return launch_decode_age(geo, pl, args, tab, st);
  if (args.total_items > 0) {
    dim3 grid(args.total_items, geo.H_kv);
#define VQK_CASE(DD, BB)                                                    \
  if (geo.D == DD && geo.bits == BB) {                                      \
    k_decode_split<DD, BB><<<grid, kThreads, 0, st>>>(geo, pl, args, tab);  \
  } else
    VQK_CASE(64, 2) VQK_CASE(64, 4) VQK_CASE(64, 8)
    VQK_CASE(128, 2) VQK_CASE(128, 4) VQK_CASE(128, 8)
    VQK_CASE(256, 2) VQK_CASE(256, 4) VQK_CASE(256, 8)
    { return cudaErrorInvalidValue; }
#undef VQK_CASE
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_combine(geo, pl, args, tab, st);
}

cudaError_t launch_combine(const Geometry &geo, const Planes &pl,
                           const DecodeArgs &args, const DecodeTable &tab,
                           cudaStream_t st) {
  cudaError_t e = launch_pdl(k_combine, dim3(geo.B * geo.H_q), dim3(kCombineThreads),
                             sizeof(float) * (geo.max_items + 1 + kCombineWarps * geo.D), st,
                             geo, pl, args, tab);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace vqk
