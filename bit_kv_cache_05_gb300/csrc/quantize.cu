// KIVI group quantization (prefill and append flush), residual-ring writes
// and the residual export.
//
// Method: VeloxQuant-MLX changelog v0.8.0 "New" (KIVI: keys per channel over
// g tokens, values per token over g channels, fp16 residual window) and
// v0.42.0 "Added" (codes plus a per-group (scale, zero) from the group's
// min/max).  Formula, in IEEE fp32 with explicit round-to-nearest
// intrinsics so that no contraction or fast-math can change a code:
//   scale = (max - min) / (2^b - 1)
//   code  = scale == 0 ? 0 : clamp(rint((x - min) / scale), 0, 2^b - 1)
//   stored scale = fp16_rn(scale), stored zero = min (exact in fp16; a
//   minimum of -0.0 is stored as +0.0).
// Packing: code of channel e at byte e*b/8, bit (e*b) mod 8, LSB first.
#include "vqk_internal.cuh"

namespace vqk {
namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ int find_seq(const int32_t *prefix, int B,
                                        int item) {
  // largest b with prefix[b] <= item (prefix non-decreasing, prefix[0] = 0)
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ uint32_t quant_code(float x, float mn, float scale,
                                               int levels) {
  if (scale == 0.0f) return 0u;
  float t = __fdiv_rn(__fsub_rn(x, mn), scale);
  float r = rintf(t);
  r = fminf(fmaxf(r, 0.0f), (float)levels);
  return (uint32_t)r;
}

__device__ __forceinline__ void load4(const __half *row, int c, float v[4]) {
  // 4 consecutive fp16 channels starting at c (c % 4 == 0): one 8-byte load
  uint2 raw = *reinterpret_cast<const uint2 *>(row + c);
  __half2 a = *reinterpret_cast<__half2 *>(&raw.x);
  __half2 b = *reinterpret_cast<__half2 *>(&raw.y);
  float2 fa = __half22float2(a), fb = __half22float2(b);
  v[0] = fa.x; v[1] = fa.y; v[2] = fb.x; v[3] = fb.y;
}

// Packs the g x D code tile in shared memory into rows of D*BITS/8 bytes and
// stores it with 16-byte vector stores (the tile is contiguous in global).
template <int BITS>
__device__ __forceinline__ void store_packed_tile(const uint8_t *codes, int g,
                                                  int D, uint8_t *dst) {
  const int row = D * BITS / 8;
  const int nchunks = g * row / 16;
  constexpr int kPerWord = 32 / BITS;
  for (int k = threadIdx.x; k < nchunks; k += blockDim.x) {
    const int byte0 = 16 * k;
    const int i = byte0 / row;
    const int e0 = (byte0 % row) * 8 / BITS;
    const uint8_t *src = codes + i * D + e0;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t acc = 0;
#pragma unroll
      for (int e = 0; e < kPerWord; ++e)
        acc |= (uint32_t)src[q * kPerWord + e] << (BITS * e);
      w[q] = acc;
    }
    *reinterpret_cast<uint4 *>(dst + byte0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// One block = one group of g tokens of one (b, h): key codes per channel,
// value codes per token.
template <int BITS>
__global__ void __launch_bounds__(kThreads)
k_flush(Geometry geo, Planes pl, const __half *__restrict__ Kin,
        const __half *__restrict__ Vin, int64_t in_stride, FlushTable tab) {
  constexpr int levels = (1 << BITS) - 1;
  __shared__ uint8_t codes[128 * kMaxD];  // g x D, g <= 128
  __shared__ float red_mn[kThreads * 4], red_mx[kThreads * 4];
  __shared__ float ch_mn[kMaxD], ch_scale[kMaxD];

  const int D = geo.D, g = geo.g, H = geo.H_kv;
  const int item = blockIdx.x, h = blockIdx.y;
  const int b = find_seq(tab.prefix, geo.B, item);
  const int P0 = tab.first_pos[b] + (item - tab.prefix[b]) * g;
  const int split = tab.src_split[b];
  const size_t bh = (size_t)b * H + h;

  const int qpr = D / 4;                 // channel quads per row
  const int cq = threadIdx.x % qpr;
  const int r = threadIdx.x / qpr;
  const int RP = kThreads / qpr;         // rows handled in parallel
  const int c0 = 4 * cq;

  auto key_row = [&](int i) -> const __half * {
    const int p = P0 + i;
    if (p < split) return pl.Kr + (bh * geo.Rcap + (p % geo.Rcap)) * D;
    return Kin + (bh * in_stride + (p - split)) * D;
  };
  auto val_row = [&](int i) -> const __half * {
    const int p = P0 + i;
    if (p < split) return pl.Vr + (bh * geo.Rcap + (p % geo.Rcap)) * D;
    return Vin + (bh * in_stride + (p - split)) * D;
  };

  // ---- keys: per channel over the g tokens ----
  float mn[4], mx[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) { mn[u] = INFINITY; mx[u] = -INFINITY; }
  for (int i = r; i < g; i += RP) {
    float v[4];
    load4(key_row(i), c0, v);
#pragma unroll
    for (int u = 0; u < 4; ++u) { mn[u] = fminf(mn[u], v[u]); mx[u] = fmaxf(mx[u], v[u]); }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    red_mn[r * D + c0 + u] = mn[u];
    red_mx[r * D + c0 + u] = mx[u];
  }
  __syncthreads();
  if (r == 0) {
    const size_t G = (size_t)(P0 / g);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float a = red_mn[c0 + u], z = red_mx[c0 + u];
      for (int k = 1; k < RP; ++k) {
        a = fminf(a, red_mn[k * D + c0 + u]);
        z = fmaxf(z, red_mx[k * D + c0 + u]);
      }
      a = __fadd_rn(a, 0.0f);  // a -0.0 minimum is stored as +0.0
      const float scale = __fdiv_rn(__fsub_rn(z, a), (float)levels);
      ch_mn[c0 + u] = a;
      ch_scale[c0 + u] = scale;
      const size_t idx = (bh * (geo.Tcap / g) + G) * D + c0 + u;
      pl.Ks[idx] = __float2half_rn(scale);
      pl.Kz[idx] = __float2half_rn(a);
    }
  }
  __syncthreads();
  for (int i = r; i < g; i += RP) {
    float v[4];
    load4(key_row(i), c0, v);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      codes[i * D + c0 + u] =
          (uint8_t)quant_code(v[u], ch_mn[c0 + u], ch_scale[c0 + u], levels);
  }
  __syncthreads();
  store_packed_tile<BITS>(codes, g, D, pl.Kc + (bh * geo.Tcap + P0) * geo.row);
  __syncthreads();

  // ---- values: per token over groups of g channels (warp shuffles) ----
  const int lanes_per_group = g / 4;     // consecutive, aligned in a warp
  const int ngroups = D / g;
  for (int i = r; i < g; i += RP) {
    float v[4];
    load4(val_row(i), c0, v);
    float a = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
    float z = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
    for (int off = 1; off < lanes_per_group; off <<= 1) {
      a = fminf(a, __shfl_xor_sync(0xffffffffu, a, off));
      z = fmaxf(z, __shfl_xor_sync(0xffffffffu, z, off));
    }
    a = __fadd_rn(a, 0.0f);  // a -0.0 minimum is stored as +0.0
    const float scale = __fdiv_rn(__fsub_rn(z, a), (float)levels);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      codes[i * D + c0 + u] = (uint8_t)quant_code(v[u], a, scale, levels);
    if (cq % lanes_per_group == 0) {
      const int j = c0 / g;
      const size_t idx = (bh * geo.Tcap + P0 + i) * ngroups + j;
      pl.Vs[idx] = __float2half_rn(scale);
      pl.Vz[idx] = __float2half_rn(a);
    }
  }
  __syncthreads();
  store_packed_tile<BITS>(codes, g, D, pl.Vc + (bh * geo.Tcap + P0) * geo.row);
}

// Residual ring writes: 16-byte chunks of fp16 rows.
__global__ void __launch_bounds__(kThreads)
k_tail(Geometry geo, Planes pl, const __half *__restrict__ Kin,
       const __half *__restrict__ Vin, int64_t in_stride, TailTable tab,
       int total) {
  const int D = geo.D;
  const int cpr = D / 8;                       // 16-byte chunks per row
  const int rows_per_block = kThreads / cpr;
  const int tok = blockIdx.x * rows_per_block + threadIdx.x / cpr;
  const int ch = (threadIdx.x % cpr) * 8;
  if (tok >= total) return;
  const int h = blockIdx.y;
  const int b = find_seq(tab.prefix, geo.B, tok);
  const int i = tok - tab.prefix[b];
  const size_t bh = (size_t)b * geo.H_kv + h;
  const int64_t src = (int64_t)(bh * in_stride + tab.row0[b] + i) * D + ch;
  const int slot = (tab.pos0[b] + i) % geo.Rcap;
  const size_t dst = (bh * geo.Rcap + slot) * D + ch;
  *reinterpret_cast<uint4 *>(pl.Kr + dst) =
      *reinterpret_cast<const uint4 *>(Kin + src);
  *reinterpret_cast<uint4 *>(pl.Vr + dst) =
      *reinterpret_cast<const uint4 *>(Vin + src);
}

struct LenTable {
  int32_t Tq[kMaxB];
  int32_t nres[kMaxB];
};

// Residual ring -> canonical linear layout (slot i = token T_q + i), zero
// beyond n_res.  One block per (slot, b*H_kv + h).
__global__ void k_export_residual(Geometry geo, const __half *__restrict__ ring,
                                  __half *__restrict__ dst, LenTable lens) {
  const int i = blockIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / geo.H_kv;
  const int D = geo.D;
  const bool valid = i < lens.nres[b];
  const int slot = valid ? (lens.Tq[b] + i) % geo.Rcap : 0;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    __half v = valid ? ring[((size_t)bh * geo.Rcap + slot) * D + c]
                     : __float2half_rn(0.0f);
    dst[((size_t)bh * geo.Rcap + i) * D + c] = v;
  }
}

}  // namespace

cudaError_t launch_flush(const Geometry &geo, const Planes &pl,
                         const __half *Kin, const __half *Vin,
                         int64_t in_stride, const FlushTable &tab,
                         int total_groups, cudaStream_t st) {
  if (total_groups <= 0) return cudaSuccess;
  dim3 grid(total_groups, geo.H_kv);
  switch (geo.bits) {
    case 2: k_flush<2><<<grid, kThreads, 0, st>>>(geo, pl, Kin, Vin, in_stride, tab); break;
    case 4: k_flush<4><<<grid, kThreads, 0, st>>>(geo, pl, Kin, Vin, in_stride, tab); break;
    case 8: k_flush<8><<<grid, kThreads, 0, st>>>(geo, pl, Kin, Vin, in_stride, tab); break;
    default: return cudaErrorInvalidValue;
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_tail(const Geometry &geo, const Planes &pl,
                        const __half *Kin, const __half *Vin,
                        int64_t in_stride, const TailTable &tab,
                        int total_tokens, cudaStream_t st) {
  if (total_tokens <= 0) return cudaSuccess;
  const int rows_per_block = kThreads / (geo.D / 8);
  dim3 grid((total_tokens + rows_per_block - 1) / rows_per_block, geo.H_kv);
  k_tail<<<grid, kThreads, 0, st>>>(geo, pl, Kin, Vin, in_stride, tab,
                                    total_tokens);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_export_residual(const Geometry &geo, const Planes &pl,
                                   int which, void *dst, const int32_t *Tq,
                                   const int32_t *nres, cudaStream_t st) {
  LenTable lens;
  for (int b = 0; b < geo.B; ++b) { lens.Tq[b] = Tq[b]; lens.nres[b] = nres[b]; }
  const __half *ring = which == 6 ? pl.Kr : pl.Vr;
  dim3 grid(geo.Rcap, geo.B * geo.H_kv);
  k_export_residual<<<grid, 128, 0, st>>>(geo, ring, (__half *)dst, lens);
  count_launch();
  return cudaGetLastError();
}

}  // namespace vqk
