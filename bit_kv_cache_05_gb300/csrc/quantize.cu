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
//   minimum of -0.0 is stored as +0.0, and a zero range as the scale +0.0).
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

// Kernels here are launched as programmatic dependents of the stream's
// previous kernel: wait for its writes, then let the next kernel be
// scheduled as this one's CTAs retire.
__device__ __forceinline__ void pdl_wait_and_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
}

__device__ __forceinline__ uint32_t quant_code(float x, float mn, float scale,
                                               int levels) {
  if (scale == 0.0f) return 0u;
  float t = __fdiv_rn(__fsub_rn(x, mn), scale);
  float r = rintf(t);
  r = fminf(fmaxf(r, 0.0f), (float)levels);
  return (uint32_t)r;
}

// The same code as quant_code, mostly without a division.  With
// r = RN(1/scale), t' = RN((x - min) * r) differs from the correctly
// rounded quotient t = RN((x - min) / scale) by at most 1.5 * 2^-23 * t'
// (two roundings of 2^-24 each against the exact quotient, one more for t).
// rint(t') and rint(t) can only differ if a half-integer lies within that
// distance of t' (or t is itself a half-integer), so whenever t' is further
// than 2^-20 * t' + 2^-30 from the nearest half-integer, rint(t') is the
// answer; otherwise the exact quotient decides.
__device__ __forceinline__ uint32_t quant_code_fast(float x, float mn,
                                                    float scale, float rcp,
                                                    int levels) {
  if (scale == 0.0f) return 0u;
  const float d = __fsub_rn(x, mn);
  float t = __fmul_rn(d, rcp);
  const float frac = t - floorf(t);
  if (fabsf(frac - 0.5f) <= fmaf(t, 9.5367431640625e-7f, 1e-9f))
    t = __fdiv_rn(d, scale);
  float r = rintf(t);
  r = fminf(fmaxf(r, 0.0f), (float)levels);
  return (uint32_t)r;
}

// quant_code_fast for two values of one group at once (f32x2 arithmetic).
// d = x - min is exact and >= 0, and t <= (max - min) / scale * (1 + 2^-21)
// stays below 2^b - 1 + 1/2, so no clamp is needed; scale == 0 gives rcp = 0,
// t = 0 and code 0 with no special case.  r = rint(t), f = t - r (exact):
// t is near a half-integer exactly when |f| >= 1/2 - bound, with the bound of
// quant_code_fast; then the correctly rounded quotient decides.
__device__ __forceinline__ void quant2(float2 x, float mn, float scale,
                                       float rcp, uint32_t &c0, uint32_t &c1) {
  const float2 d = __fadd2_rn(x, make_float2(-mn, -mn));
  const float2 t = __fmul2_rn(d, make_float2(rcp, rcp));
  float2 r = make_float2(rintf(t.x), rintf(t.y));
  const float2 f = __fadd2_rn(t, make_float2(-r.x, -r.y));
  const float2 lim = __fadd2_rn(make_float2(0.5f, 0.5f),
                                __ffma2_rn(t, make_float2(-9.5367431640625e-7f, -9.5367431640625e-7f),
                                           make_float2(-1e-9f, -1e-9f)));
  if (fabsf(f.x) >= lim.x) r.x = rintf(__fdiv_rn(d.x, scale));
  if (fabsf(f.y) >= lim.y) r.y = rintf(__fdiv_rn(d.y, scale));
  c0 = (uint32_t)r.x;
  c1 = (uint32_t)r.y;
}

// quant2's fast path only: the codes from the reciprocal, and whether each
// value is near a half-integer (where quant2 takes the correctly rounded
// quotient instead; the caller redoes those values with quant_exact).  No
// branch, so a loop over many pairs carries no divergence bookkeeping.
// The rounding adds 2^23: for 0 <= t < 2^22 the sum's low mantissa bits
// are rint(t) (round to nearest, ties to even, as rintf), so the code comes
// out of the float's bits with no conversion.  Within a group t stays below
// LEVELS + 1, so the band of quant2, 2^-20 t + 1e-9, is inside the constant
// band (LEVELS + 1) 2^-20: flagging that band flags every value quant2
// would send to the exact quotient (and a few more, about 2 (LEVELS + 1)
// 2^-20 of the values, which the exact quotient gives the same code).
template <int LEVELS>
__device__ __forceinline__ void quant2_flag(float2 x, float mn, float rcp,
                                            uint32_t &c0, uint32_t &c1,
                                            bool &n0, bool &n1) {
  constexpr float kLim = 0.5f - (LEVELS + 1) * 9.5367431640625e-7f;
  const float2 d = __fadd2_rn(x, make_float2(-mn, -mn));
  const float2 t = __fmul2_rn(d, make_float2(rcp, rcp));
  const float2 tm = __fadd2_rn(t, make_float2(8388608.f, 8388608.f));
  const float2 r = __fadd2_rn(tm, make_float2(-8388608.f, -8388608.f));
  const float2 f = __fadd2_rn(t, make_float2(-r.x, -r.y));
  n0 = fabsf(f.x) >= kLim;
  n1 = fabsf(f.y) >= kLim;
  c0 = __float_as_uint(tm.x) & 0xFFu;
  c1 = __float_as_uint(tm.y) & 0xFFu;
}

// 16-byte asynchronous global -> shared copy (completed by cp.async.wait_group)
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}

// quant2's near-tie path for one value: rint of the correctly rounded
// quotient
__device__ __noinline__ uint32_t quant_exact(float x, float mn, float scale) {
  return (uint32_t)rintf(__fdiv_rn(__fsub_rn(x, mn), scale));
}

// Packs the g x D code tile in shared memory (row stride cs bytes) into rows
// of D*BITS/8 bytes and stores it with 16-byte vector stores (the tile is
// contiguous in global).
template <int BITS>
__device__ __forceinline__ void store_packed_tile(const uint8_t *codes, int cs,
                                                  int g, int D, uint8_t *dst) {
  const int row = D * BITS / 8;
  const int nchunks = g * row / 16;
  constexpr int kPerWord = 32 / BITS;
  for (int k = threadIdx.x; k < nchunks; k += blockDim.x) {
    const int byte0 = 16 * k;
    const int i = byte0 / row;
    const int e0 = (byte0 % row) * 8 / BITS;
    const uint8_t *src = codes + i * cs + e0;
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

// The g x D code tile in kLayoutFrag order (2- or 4-bit codes): one thread
// per 32-bit word, whose fields are gathered from the tile.
template <int BITS>
__device__ __forceinline__ void store_frag_keys(const uint8_t *codes, int cs,
                                                int g, int D, uint8_t *dst) {
  constexpr int F = 16 / BITS, KPW = 8 / BITS;   // fields per half
  const int wpr = D * BITS / 32, nw = D * BITS / 128;
  for (int w = threadIdx.x; w < g * wpr; w += blockDim.x) {
    const int i = w / wpr, wi = w - i * wpr;
    const int tig = wi / nw, hw = wi - tig * nw;
    uint32_t acc = 0;
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int r = 0; r < F; ++r) {
        const int ks = KPW * hw + (r >> 1), e = 2 * (r & 1) + s;
        acc |= (uint32_t)codes[i * cs + 16 * ks + 4 * tig + e] << (16 * s + BITS * r);
      }
    reinterpret_cast<uint32_t *>(dst)[w] = acc;
  }
}

template <int BITS>
__device__ __forceinline__ void store_frag_values(const uint8_t *codes, int cs,
                                                  int g, int D, uint8_t *dst) {
  constexpr int F = 16 / BITS, KPW = 8 / BITS;
  const int nw = D * BITS / 128, wpb = D * BITS / 2;   // words per block
  for (int w = threadIdx.x; w < g * D * BITS / 32; w += blockDim.x) {
    const int kb = w / wpb, wb = w - kb * wpb;
    const int pi = wb / (8 * nw), rem = wb - pi * 8 * nw;
    const int j = rem / nw, hw = rem - j * nw;
    const int tA = 16 * kb + (pi < 4 ? pi : pi + 4);
    uint32_t acc = 0;
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int r = 0; r < F; ++r) {
        const int mv = KPW * hw + (r >> 1), rho = r & 1;
        acc |= (uint32_t)codes[(tA + 4 * s) * cs + 16 * mv + 2 * j + rho]
               << (16 * s + BITS * r);
      }
    reinterpret_cast<uint32_t *>(dst)[w] = acc;
  }
}

// Copies the g fp16 rows of one group (token positions P0 ... P0+g-1) into a
// shared tile [g][D] with 16-byte loads, all in flight at once.  Position p
// comes from the residual ring when p < split, else from input row p - split.
__device__ __forceinline__ void load_tile(__half *tile, const __half *ring,
                                          const __half *in, size_t bh,
                                          int64_t in_stride, int P0, int split,
                                          int g, int D, int Rcap) {
  const int cpr = D / 8;
  for (int idx = threadIdx.x; idx < g * cpr; idx += blockDim.x) {
    const int i = idx / cpr, c8 = (idx - i * cpr) * 8;
    const int p = P0 + i;
    const __half *src = p < split ? ring + (bh * Rcap + (p % Rcap)) * D
                                  : in + (bh * in_stride + (p - split)) * D;
    *reinterpret_cast<uint4 *>(tile + i * D + c8) =
        *reinterpret_cast<const uint4 *>(src + c8);
  }
}

// One block = one group of g tokens of one (b, h), one thread per channel
// (D threads).  Keys: the group's key rows are staged in a shared tile and
// quantized per channel (thread c walks column c: consecutive threads read
// consecutive halves).  Values: thread t takes (token t / (D/g), channel
// group t % (D/g)) — D/g groups of g tokens is D items — and reads its g
// values straight from global memory with 16-byte loads.  Codes go to a
// shared code tile whose rows are padded to D + 4 bytes, so that the
// threads of a warp writing (and the packers reading) different rows hit
// different banks; the tile is then packed and stored.
template <int BITS>
__global__ void __launch_bounds__(kMaxD)
k_flush(Geometry geo, Planes pl, const __half *__restrict__ Kin,
        const __half *__restrict__ Vin, int64_t in_stride, FlushTable tab) {
  pdl_wait_and_release();
  constexpr int levels = (1 << BITS) - 1;
  extern __shared__ __align__(16) unsigned char fsm[];
  const int D = geo.D, g = geo.g, H = geo.H_kv;
  const int CS = D + 4;                                           // code row stride
  __half *tile = reinterpret_cast<__half *>(fsm);                 // [g][D]
  uint8_t *codes = fsm + (size_t)g * D * sizeof(__half);         // [g][CS]

  const int item = blockIdx.x, h = blockIdx.y;
  const int b = find_seq(tab.prefix, geo.B, item);
  const int P0 = tab.first_pos[b] + (item - tab.prefix[b]) * g;
  const int split = tab.src_split[b];
  const size_t bh = (size_t)b * H + h;
  const int c = threadIdx.x;   // blockDim.x == D

  // KIVI-Sink: bit i of sinkm = token P0 + i is a sink (left out of every
  // min/max; its codes 0, its own value groups empty)
  __shared__ uint32_t sinkm[4];
  const bool sinks = geo.n_sink > 0;
  if (sinks) {
    if (c < 4) sinkm[c] = 0u;
    __syncthreads();
    if (c < geo.n_sink) {
      const int p = pl.sink_pos[bh * geo.n_sink + c];
      if (p >= P0 && p < P0 + g) atomicOr(&sinkm[(p - P0) >> 5], 1u << ((p - P0) & 31));
    }
  }
  auto is_sink = [&](int i) { return sinks && ((sinkm[i >> 5] >> (i & 31)) & 1u); };

  // ---- keys: per channel over the g tokens ----
  load_tile(tile, pl.Kr, Kin, bh, in_stride, P0, split, g, D, geo.Rcap);
  __syncthreads();
  if (sinks) {
    // the group's non-sink tokens only
    float mn = INFINITY, mx = -INFINITY;
    for (int i = 0; i < g; ++i) {
      if (is_sink(i)) continue;
      const float v = __half2float(tile[i * D + c]);
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
    }
    if (mn > mx) { mn = 0.f; mx = 0.f; }   // sinks only: scale and zero +0
    mn = __fadd_rn(mn, 0.0f);
    const float scale = __fdiv_rn(__fadd_rn(__fsub_rn(mx, mn), 0.0f), (float)levels);
    const float rcp = scale != 0.0f ? __frcp_rn(scale) : 0.0f;
    const size_t idx = (bh * (geo.Tcap / g) + P0 / g) * D + c;
    const __half sh = __float2half_rn(scale);
    pl.Ks[idx] = sh;
    pl.Kz[idx] = __float2half_rn(mn);
    if (pl.ksmax) {
      const unsigned m = __reduce_max_sync(0xffffffffu, (unsigned)__half_as_ushort(sh));
      if ((c & 31) == 0) atomicMax(pl.ksmax + bh, m);
    }
    for (int i = 0; i < g; i += 2) {
      uint32_t c0, c1;
      quant2(make_float2(__half2float(tile[i * D + c]), __half2float(tile[(i + 1) * D + c])),
             mn, scale, rcp, c0, c1);
      codes[i * CS + c] = is_sink(i) ? 0 : (uint8_t)c0;
      codes[(i + 1) * CS + c] = is_sink(i + 1) ? 0 : (uint8_t)c1;
    }
  } else {
    // column c, two tokens per step as an fp16 pair (min / max are exact)
    __half2 mn2 = __float2half2_rn(INFINITY), mx2 = __float2half2_rn(-INFINITY);
    for (int i = 0; i < g; i += 2) {
      const __half2 v = __halves2half2(tile[i * D + c], tile[(i + 1) * D + c]);
      mn2 = __hmin2(mn2, v);
      mx2 = __hmax2(mx2, v);
    }
    float mn = fminf(__low2float(mn2), __high2float(mn2));
    const float mx = fmaxf(__low2float(mx2), __high2float(mx2));
    mn = __fadd_rn(mn, 0.0f);  // a -0.0 minimum is stored as +0.0
    // a zero range is +0.0 (max - min is -0.0 when the max is -0.0)
    const float scale = __fdiv_rn(__fadd_rn(__fsub_rn(mx, mn), 0.0f), (float)levels);
    const float rcp = scale != 0.0f ? __frcp_rn(scale) : 0.0f;
    const size_t idx = (bh * (geo.Tcap / g) + P0 / g) * D + c;
    const __half sh = __float2half_rn(scale);
    pl.Ks[idx] = sh;
    pl.Kz[idx] = __float2half_rn(mn);
    // running bound of the head's key scales (non-negative fp16 values
    // order like their bit patterns)
    if (pl.ksmax) {
      const unsigned m = __reduce_max_sync(0xffffffffu, (unsigned)__half_as_ushort(sh));
      if ((c & 31) == 0) atomicMax(pl.ksmax + bh, m);
    }
    for (int i = 0; i < g; i += 2) {
      uint32_t c0, c1;
      quant2(make_float2(__half2float(tile[i * D + c]), __half2float(tile[(i + 1) * D + c])),
             mn, scale, rcp, c0, c1);
      codes[i * CS + c] = (uint8_t)c0;
      codes[(i + 1) * CS + c] = (uint8_t)c1;
    }
  }
  __syncthreads();
  if ((BITS == 2 || BITS == 4) && geo.layout == kLayoutFrag)
    store_frag_keys<BITS>(codes, CS, g, D, pl.Kc + (bh * geo.Tcap + P0) * geo.row);
  else
    store_packed_tile<BITS>(codes, CS, g, D, pl.Kc + (bh * geo.Tcap + P0) * geo.row);
  __syncthreads();

  // ---- values: per token over groups of g channels ----
  {
    const int ngroups = D / g;
    const int i = c / ngroups, j = c - i * ngroups;   // g * ngroups == D items
    const int p = P0 + i;
    const bool empty = is_sink(i);   // a sink's value groups have no member
    const __half *row = (p < split ? pl.Vr + (bh * geo.Rcap + (p % geo.Rcap)) * D
                                   : Vin + (bh * in_stride + (p - split)) * D) + j * g;
    __half2 mn2 = __float2half2_rn(INFINITY), mx2 = __float2half2_rn(-INFINITY);
    for (int k = 0; k < g; k += 8) {
      const uint4 u = *reinterpret_cast<const uint4 *>(row + k);
      const __half2 *h4 = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        mn2 = __hmin2(mn2, h4[e]);
        mx2 = __hmax2(mx2, h4[e]);
      }
    }
    float mn = fminf(__low2float(mn2), __high2float(mn2));
    const float mx = fmaxf(__low2float(mx2), __high2float(mx2));
    mn = empty ? 0.f : __fadd_rn(mn, 0.0f);  // a -0.0 minimum is stored as +0.0
    // a zero range is +0.0 (max - min is -0.0 when the max is -0.0)
    const float scale = empty ? 0.f : __fdiv_rn(__fadd_rn(__fsub_rn(mx, mn), 0.0f), (float)levels);
    const float rcp = scale != 0.0f ? __frcp_rn(scale) : 0.0f;
    uint32_t *crow = reinterpret_cast<uint32_t *>(codes + i * CS + j * g);
    for (int k = 0; k < g; k += 8) {
      const uint4 u = *reinterpret_cast<const uint4 *>(row + k);
      const __half2 *h4 = reinterpret_cast<const __half2 *>(&u);
      uint32_t w[2] = {0u, 0u};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t c0, c1;
        quant2(__half22float2(h4[e]), mn, scale, rcp, c0, c1);
        w[e >> 1] |= (c0 | (c1 << 8)) << (16 * (e & 1));
      }
      crow[k / 4] = w[0];
      crow[k / 4 + 1] = w[1];
    }
    const size_t vidx = (bh * geo.Tcap + P0 + i) * ngroups + j;
    pl.Vs[vidx] = __float2half_rn(scale);
    pl.Vz[vidx] = __float2half_rn(mn);
  }
  __syncthreads();
  if ((BITS == 2 || BITS == 4) && geo.layout == kLayoutFrag)
    store_frag_values<BITS>(codes, CS, g, D, pl.Vc + (bh * geo.Tcap + P0) * geo.row);
  else
    store_packed_tile<BITS>(codes, CS, g, D, pl.Vc + (bh * geo.Tcap + P0) * geo.row);
}

// The flush for the common shapes (D = 64 or 128, g = 32 or 64), with D,
// g and the code width known at compile time: every index of the tile, the
// code tile and the packers is a constant or a shift, the g source rows of
// the group are looked up once (the residual ring's slot arithmetic per
// token, not per 16-byte chunk), the key and value tiles arrive together
// by asynchronous copies, and the near-tie test flags values in one
// branch-free pass that a rare second pass redoes exactly.
// Same arithmetic as k_flush, bit for bit.
template <int BITS, int D, int G>
__device__ __forceinline__ void store_frag_keys_t(const uint8_t *codes, uint8_t *dst) {
  constexpr int F = 16 / BITS, KPW = 8 / BITS, CS = D + 4;
  constexpr int WPR = D * BITS / 32, NWD = D * BITS / 128;
#pragma unroll
  for (int k = 0; k < G * WPR / D; ++k) {
    const int w = threadIdx.x + k * D;
    const int i = w / WPR, wi = w % WPR;
    const int tig = wi / NWD, hw = wi % NWD;
    if constexpr (BITS == 4) {
      // the word's 8 fields are channels 16 ks + 4 tig + e, e = 0 ... 3, of
      // K-steps ks = 2 hw and 2 hw + 1: two 4-byte runs of the token's code
      // row.  Field (r, s) of the word (e = 2 (r & 1) + s) sits at bit
      // 16 s + 4 r: bytes e0, e1 of a run go to bits 0 and 16, bytes e2,
      // e3 to bits 4 and 20, the second run 8 bits higher.
      uint32_t acc = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t x = *reinterpret_cast<const uint32_t *>(
            codes + i * CS + 16 * (2 * hw + h) + 4 * tig);
        const uint32_t lo = __byte_perm(x, 0u, 0x4140);   // e0 | e1 << 16
        const uint32_t hi = __byte_perm(x, 0u, 0x4342);   // e2 | e3 << 16
        acc |= (lo | (hi << 4)) << (8 * h);
      }
      reinterpret_cast<uint32_t *>(dst)[w] = acc;
      continue;
    }
    uint32_t acc = 0;
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int r = 0; r < F; ++r) {
        const int ks = KPW * hw + (r >> 1), e = 2 * (r & 1) + s;
        acc |= (uint32_t)codes[i * CS + 16 * ks + 4 * tig + e] << (16 * s + BITS * r);
      }
    reinterpret_cast<uint32_t *>(dst)[w] = acc;
  }
}

template <int BITS, int D, int G>
__device__ __forceinline__ void store_frag_values_t(const uint8_t *codes, uint8_t *dst) {
  constexpr int F = 16 / BITS, KPW = 8 / BITS, CS = D + 4;
  constexpr int NWD = D * BITS / 128, WPB = D * BITS / 2;
#pragma unroll
  for (int k = 0; k < G * D * BITS / 32 / D; ++k) {
    const int w = threadIdx.x + k * D;
    const int kb = w / WPB, wb = w % WPB;
    const int pi = wb / (8 * NWD), rem = wb % (8 * NWD);
    const int j = rem / NWD, hw = rem % NWD;
    const int tA = 16 * kb + (pi < 4 ? pi : pi + 4);
    uint32_t acc = 0;
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int r = 0; r < F; ++r) {
        const int mv = KPW * hw + (r >> 1), rho = r & 1;
        acc |= (uint32_t)codes[(tA + 4 * s) * CS + 16 * mv + 2 * j + rho]
               << (16 * s + BITS * r);
      }
    reinterpret_cast<uint32_t *>(dst)[w] = acc;
  }
}

template <int BITS, int D, int G>
__device__ __forceinline__ void store_packed_tile_t(const uint8_t *codes, uint8_t *dst) {
  constexpr int ROW = D * BITS / 8, CS = D + 4, PER = 32 / BITS;
#pragma unroll
  for (int k = 0; k < (G * ROW / 16 + D - 1) / D; ++k) {
    const int q16 = threadIdx.x + k * D;
    if (q16 >= G * ROW / 16) break;
    const int byte0 = 16 * q16;
    const int i = byte0 / ROW, e0 = (byte0 % ROW) * 8 / BITS;
    const uint8_t *src = codes + i * CS + e0;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t acc = 0;
#pragma unroll
      for (int e = 0; e < PER; ++e) acc |= (uint32_t)src[q * PER + e] << (BITS * e);
      w[q] = acc;
    }
    *reinterpret_cast<uint4 *>(dst + byte0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// CTAs per SM the register budget is cut for: the shared memory of a
// 64-token group of 128 channels (41 KB with both staged tiles) leaves room
// for five, which at most 96 registers a thread allow (four at 100)
template <int D, int G>
constexpr int flush_min_ctas() { return D * G == 128 * 64 || D * G == 128 * 32 ? 5 : 1; }

template <int BITS, int D, int G>
__global__ void __launch_bounds__(D, flush_min_ctas<D, G>())
k_flush_t(Geometry geo, Planes pl, const __half *__restrict__ Kin,
          const __half *__restrict__ Vin, int64_t in_stride, FlushTable tab) {
  pdl_wait_and_release();
  constexpr int levels = (1 << BITS) - 1, CS = D + 4, ROW = D * BITS / 8;
  constexpr int NJ = D / G, CPR = D / 8;
  constexpr int VS = D + 8;   // value row stride (halves): 16 bytes of padding
  extern __shared__ __align__(16) unsigned char fsm[];
  __half *tile = reinterpret_cast<__half *>(fsm);                 // [G][D]
  uint8_t *codes = fsm + (size_t)G * D * sizeof(__half);         // [G][CS]
  __half *vtile = reinterpret_cast<__half *>(codes + G * CS);    // [G][VS]
  __shared__ const __half *sk[G], *sv[G];
  __shared__ uint32_t sinkm[4];
  const int c = threadIdx.x, item = blockIdx.x, h = blockIdx.y;
  const int b = find_seq(tab.prefix, geo.B, item);
  const int P0 = tab.first_pos[b] + (item - tab.prefix[b]) * G;
  const int split = tab.src_split[b];
  const size_t bh = (size_t)b * geo.H_kv + h;
  if (c < G) {
    // the source rows of the group's tokens: residual ring, then input
    const int p = P0 + c;
    if (p < split) {
      const size_t off = (bh * geo.Rcap + (p % geo.Rcap)) * D;
      sk[c] = pl.Kr + off;
      sv[c] = pl.Vr + off;
    } else {
      const size_t off = (bh * in_stride + (p - split)) * D;
      sk[c] = Kin + off;
      sv[c] = Vin + off;
    }
  }
  const bool sinks = geo.n_sink > 0;
  if (sinks && c < 4) sinkm[c] = 0u;
  __syncthreads();
  if (sinks && c < geo.n_sink) {
    const int p = pl.sink_pos[bh * geo.n_sink + c];
    if (p >= P0 && p < P0 + G) atomicOr(&sinkm[(p - P0) >> 5], 1u << ((p - P0) & 31));
  }
  // the key and value tiles (G rows of D fp16 values each) by 16-byte
  // asynchronous copies, all in flight together, in two groups: the keys
  // are quantized while the value tile still lands
#pragma unroll
  for (int k = 0; k < G * CPR / D; ++k) {
    const int idx = c + k * D, i = idx / CPR, c8 = (idx % CPR) * 8;
    cp_async16(tile + i * D + c8, sk[i] + c8);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
#pragma unroll
  for (int k = 0; k < G * CPR / D; ++k) {
    const int idx = c + k * D, i = idx / CPR, c8 = (idx % CPR) * 8;
    cp_async16(vtile + i * VS + c8, sv[i] + c8);
  }
  asm volatile("cp.async.commit_group;\n cp.async.wait_group 1;" ::: "memory");
  __syncthreads();
  auto is_sink = [&](int i) { return sinks && ((sinkm[i >> 5] >> (i & 31)) & 1u); };

  // ---- keys: channel c over the G tokens, held as fp16 pairs ----
  {
    __half2 col[G / 2];
#pragma unroll
    for (int k = 0; k < G / 2; ++k)
      col[k] = __halves2half2(tile[(2 * k) * D + c], tile[(2 * k + 1) * D + c]);
    float mn, mx;
    if (!sinks) {
      __half2 mn2 = col[0], mx2 = col[0];
#pragma unroll
      for (int k = 1; k < G / 2; ++k) {
        mn2 = __hmin2(mn2, col[k]);
        mx2 = __hmax2(mx2, col[k]);
      }
      mn = fminf(__low2float(mn2), __high2float(mn2));
      mx = fmaxf(__low2float(mx2), __high2float(mx2));
    } else {
      mn = INFINITY;
      mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < G / 2; ++k) {
        const float2 f = __half22float2(col[k]);
        if (!is_sink(2 * k)) { mn = fminf(mn, f.x); mx = fmaxf(mx, f.x); }
        if (!is_sink(2 * k + 1)) { mn = fminf(mn, f.y); mx = fmaxf(mx, f.y); }
      }
      if (mn > mx) { mn = 0.f; mx = 0.f; }   // sinks only: scale and zero +0
    }
    mn = __fadd_rn(mn, 0.0f);  // a -0.0 minimum is stored as +0.0
    // a zero range is +0.0 (max - min is -0.0 when the max is -0.0)
    const float scale = __fdiv_rn(__fadd_rn(__fsub_rn(mx, mn), 0.0f), (float)levels);
    const float rcp = scale != 0.0f ? __frcp_rn(scale) : 0.0f;
    const size_t idx = (bh * (geo.Tcap / G) + P0 / G) * D + c;
    const __half sh = __float2half_rn(scale);
    pl.Ks[idx] = sh;
    pl.Kz[idx] = __float2half_rn(mn);
    if (pl.ksmax) {
      const unsigned m = __reduce_max_sync(0xffffffffu, (unsigned)__half_as_ushort(sh));
      if ((c & 31) == 0) atomicMax(pl.ksmax + bh, m);
    }
    // bit k: a value of token pair k is near a half-integer (one bit per
    // pair: one select and one or per two values)
    uint32_t near = 0;
#pragma unroll
    for (int k = 0; k < G / 2; ++k) {
      uint32_t c0, c1;
      bool n0, n1;
      quant2_flag<levels>(__half22float2(col[k]), mn, rcp, c0, c1, n0, n1);
      near |= (uint32_t)(n0 | n1) << k;
      codes[(2 * k) * CS + c] = (uint8_t)c0;
      codes[(2 * k + 1) * CS + c] = (uint8_t)c1;
    }
    // the rare near-ties: the pair's flags again, and the correctly rounded
    // quotient for the flagged values (scale == 0 gives rcp = 0, t = 0 and
    // no near-tie)
    while (near) {
      const int k = __ffs(near) - 1;
      near &= near - 1;
      const __half2 x2 = __halves2half2(tile[(2 * k) * D + c], tile[(2 * k + 1) * D + c]);
      uint32_t c0, c1;
      bool n0, n1;
      quant2_flag<levels>(__half22float2(x2), mn, rcp, c0, c1, n0, n1);
      if (n0) codes[(2 * k) * CS + c] = (uint8_t)quant_exact(__low2float(x2), mn, scale);
      if (n1) codes[(2 * k + 1) * CS + c] = (uint8_t)quant_exact(__high2float(x2), mn, scale);
    }
    // sink tokens hold code 0 (their rows are kept in fp16)
    if (sinks) {
#pragma unroll
      for (int w = 0; w < (G + 31) / 32; ++w) {
        uint32_t m = sinkm[w];
        while (m) {
          const int i = 32 * w + __ffs(m) - 1;
          m &= m - 1;
          codes[i * CS + c] = 0;
        }
      }
    }
  }
  __syncthreads();
  if constexpr (BITS == 2 || BITS == 4) {
    if (geo.layout == kLayoutFrag)
      store_frag_keys_t<BITS, D, G>(codes, pl.Kc + (bh * geo.Tcap + P0) * ROW);
    else
      store_packed_tile_t<BITS, D, G>(codes, pl.Kc + (bh * geo.Tcap + P0) * ROW);
  } else {
    store_packed_tile_t<BITS, D, G>(codes, pl.Kc + (bh * geo.Tcap + P0) * ROW);
  }
  // this thread's value copies complete, then every thread's
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  // ---- values: token i over channels j*G ... j*G+G-1, in registers ----
  {
    const int i = c / NJ, j = c % NJ;
    const bool empty = is_sink(i);   // a sink's value groups have no member
    const uint4 *row = reinterpret_cast<const uint4 *>(vtile + i * VS + j * G);
    uint4 u[G / 8];
#pragma unroll
    for (int k = 0; k < G / 8; ++k) u[k] = row[k];
    __half2 mn2 = *reinterpret_cast<const __half2 *>(&u[0].x), mx2 = mn2;
#pragma unroll
    for (int k = 0; k < G / 8; ++k) {
      const __half2 *h4 = reinterpret_cast<const __half2 *>(&u[k]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        mn2 = __hmin2(mn2, h4[e]);
        mx2 = __hmax2(mx2, h4[e]);
      }
    }
    float mn = fminf(__low2float(mn2), __high2float(mn2));
    const float mx = fmaxf(__low2float(mx2), __high2float(mx2));
    mn = empty ? 0.f : __fadd_rn(mn, 0.0f);
    const float scale = empty ? 0.f : __fdiv_rn(__fadd_rn(__fsub_rn(mx, mn), 0.0f), (float)levels);
    const float rcp = scale != 0.0f ? __frcp_rn(scale) : 0.0f;
    uint32_t *crow = reinterpret_cast<uint32_t *>(codes + i * CS + j * G);
    uint32_t near = 0;   // bit v: a value of pair v of the group is near a half-integer
#pragma unroll
    for (int k = 0; k < G / 8; ++k) {
      const __half2 *h4 = reinterpret_cast<const __half2 *>(&u[k]);
      uint32_t w[2] = {0u, 0u};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t c0, c1;
        bool n0, n1;
        quant2_flag<levels>(__half22float2(h4[e]), mn, rcp, c0, c1, n0, n1);
        near |= (uint32_t)(n0 | n1) << (4 * k + e);
        w[e >> 1] |= (c0 | (c1 << 8)) << (16 * (e & 1));
      }
      crow[2 * k] = w[0];
      crow[2 * k + 1] = w[1];
    }
    // the rare near-ties: the pair's flags again
    while (near) {
      const int v = __ffs(near) - 1;
      near &= near - 1;
      const __half2 x2 = reinterpret_cast<const __half2 *>(vtile + i * VS + j * G)[v];
      uint32_t c0, c1;
      bool n0, n1;
      quant2_flag<levels>(__half22float2(x2), mn, rcp, c0, c1, n0, n1);
      uint8_t *cv = codes + i * CS + j * G + 2 * v;
      if (n0) cv[0] = (uint8_t)quant_exact(__low2float(x2), mn, scale);
      if (n1) cv[1] = (uint8_t)quant_exact(__high2float(x2), mn, scale);
    }
    const size_t vidx = (bh * geo.Tcap + P0 + i) * NJ + j;
    pl.Vs[vidx] = __float2half_rn(scale);
    pl.Vz[vidx] = __float2half_rn(mn);
  }
  __syncthreads();
  if constexpr (BITS == 2 || BITS == 4) {
    if (geo.layout == kLayoutFrag)
      store_frag_values_t<BITS, D, G>(codes, pl.Vc + (bh * geo.Tcap + P0) * ROW);
    else
      store_packed_tile_t<BITS, D, G>(codes, pl.Vc + (bh * geo.Tcap + P0) * ROW);
  } else {
    store_packed_tile_t<BITS, D, G>(codes, pl.Vc + (bh * geo.Tcap + P0) * ROW);
  }
}

// Residual ring writes: 16-byte chunks of fp16 rows.  The ring slots they
// go to may still be read by the kernel before this one in the stream (a
// flush reads the old residual rows, a merge the window), so the stores
// follow the programmatic wait.  When the input was complete before the
// append's first kernel (input_ready: that kernel releases this grid only
// after its own wait), each thread loads its chunks before the wait, and
// the loads overlap the previous kernel's end; otherwise (the kernel
// before wrote the input) after it.
__global__ void __launch_bounds__(kThreads)
k_tail(Geometry geo, Planes pl, const __half *__restrict__ Kin,
       const __half *__restrict__ Vin, int64_t in_stride, TailTable tab,
       int total, int input_ready) {
  if (!input_ready) asm volatile("griddepcontrol.wait;" ::: "memory");
  const int D = geo.D;
  const int cpr = D / 8;                       // 16-byte chunks per row
  const int rows_per_block = kThreads / cpr;
  const int tok = blockIdx.x * rows_per_block + threadIdx.x / cpr;
  const int ch = (threadIdx.x % cpr) * 8;
  const bool ok = tok < total;
  uint4 kx = make_uint4(0u, 0u, 0u, 0u), vx = kx;
  size_t dst = 0;
  if (ok) {
    const int h = blockIdx.y;
    const int b = find_seq(tab.prefix, geo.B, tok);
    const int i = tok - tab.prefix[b];
    const size_t bh = (size_t)b * geo.H_kv + h;
    const int64_t src = (int64_t)(bh * in_stride + tab.row0[b] + i) * D + ch;
    const int slot = (tab.pos0[b] + i) % geo.Rcap;
    dst = (bh * geo.Rcap + slot) * D + ch;
    kx = *reinterpret_cast<const uint4 *>(Kin + src);
    vx = *reinterpret_cast<const uint4 *>(Vin + src);
  }
  pdl_wait_and_release();
  if (!ok) return;
  *reinterpret_cast<uint4 *>(pl.Kr + dst) = kx;
  *reinterpret_cast<uint4 *>(pl.Vr + dst) = vx;
}

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
  const size_t smem = (size_t)geo.g * (geo.D * sizeof(__half) + geo.D + 4);
  // the specialised flush also stages the value tile (rows padded by 8 halves)
  const size_t smem_t = smem + (size_t)geo.g * (geo.D + 8) * sizeof(__half);
  // the common shapes: the compile-time specialised flush
#define VQK_FT(BB, DD, GG)                                                     \
  if (geo.bits == BB && geo.D == DD && geo.g == GG) {                          \
    const cudaError_t e2 = launch_pdl(k_flush_t<BB, DD, GG>, grid, dim3(DD),   \
                                      smem_t, st, geo, pl, Kin, Vin, in_stride, \
                                      tab);                                    \
    count_launch();                                                            \
    return e2;                                                                 \
  }
#define VQK_FT_B(BB) VQK_FT(BB, 64, 32) VQK_FT(BB, 64, 64) VQK_FT(BB, 128, 32) \
  VQK_FT(BB, 128, 64)
  VQK_FT_B(2) VQK_FT_B(4) VQK_FT_B(8)
#undef VQK_FT_B
#undef VQK_FT
  void *fn = nullptr;
  switch (geo.bits) {
    case 2: fn = (void *)k_flush<2>; break;
    case 4: fn = (void *)k_flush<4>; break;
    case 8: fn = (void *)k_flush<8>; break;
    default: return cudaErrorInvalidValue;
  }
  // tiles above the default 48 KB (g = 128 with D = 256) need the opt-in
  // limit, which belongs to the current device's context: set it on every
  // such launch (no process-wide flag to race on or to carry across devices)
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaSuccess;
  switch (geo.bits) {
    case 2: e = launch_pdl(k_flush<2>, grid, dim3(geo.D), smem, st, geo, pl, Kin, Vin, in_stride, tab); break;
    case 4: e = launch_pdl(k_flush<4>, grid, dim3(geo.D), smem, st, geo, pl, Kin, Vin, in_stride, tab); break;
    case 8: e = launch_pdl(k_flush<8>, grid, dim3(geo.D), smem, st, geo, pl, Kin, Vin, in_stride, tab); break;
  }
  count_launch();
  return e;
}

cudaError_t launch_tail(const Geometry &geo, const Planes &pl,
                        const __half *Kin, const __half *Vin,
                        int64_t in_stride, const TailTable &tab,
                        int total_tokens, bool input_ready, cudaStream_t st) {
  if (total_tokens <= 0) return cudaSuccess;
  const int rows_per_block = kThreads / (geo.D / 8);
  dim3 grid((total_tokens + rows_per_block - 1) / rows_per_block, geo.H_kv);
  const cudaError_t e = launch_pdl(k_tail, grid, dim3(kThreads), 0, st, geo, pl,
                                  Kin, Vin, in_stride, tab, total_tokens,
                                  input_ready ? 1 : 0);
  count_launch();
  return e;
}

// kLayoutFrag plane -> packed order: one thread per packed 32-bit word
// (32/b codes of one token row), each field gathered from its
// fragment-order position.  Covers all Tcap rows of every (b, h).
__global__ void k_export_frag(Geometry geo, const uint8_t *__restrict__ src,
                              bool values, uint32_t *__restrict__ dst) {
  const int D = geo.D, b = geo.bits, cpw = 32 / b, wpr = D * b / 32;
  const uint32_t mask = (1u << b) - 1u;
  const size_t total = (size_t)geo.B * geo.H_kv * geo.Tcap * wpr;
  for (size_t w = blockIdx.x * (size_t)blockDim.x + threadIdx.x; w < total;
       w += (size_t)gridDim.x * blockDim.x) {
    const size_t row = w / wpr;                 // (b, h, t)
    const int wr = (int)(w - row * wpr);
    const int t = (int)(row % geo.Tcap);
    const uint32_t *rw = reinterpret_cast<const uint32_t *>(src) + row * wpr;
    const uint32_t *blk = reinterpret_cast<const uint32_t *>(src) +
                          (row - (t & 15)) * wpr;   // the token's 16-row block
    uint32_t acc = 0;
    for (int f = 0; f < cpw; ++f) {
      const int c = cpw * wr + f;
      const FragPos pos = values ? frag_value(D, b, t & 15, c) : frag_key(D, b, c);
      const uint32_t word = values ? blk[pos.word] : rw[pos.word];
      acc |= ((word >> pos.bit) & mask) << (b * f);
    }
    dst[w] = acc;
  }
}

cudaError_t launch_export_frag(const Geometry &geo, const uint8_t *src,
                               bool values, void *dst, cudaStream_t st) {
  k_export_frag<<<1024, 256, 0, st>>>(geo, src, values, (uint32_t *)dst);
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

// ---- dequantized copy of the cache (the unfused baseline) ------------------
//
// Per (sequence, kv head): tokens t < T_q are rebuilt as fp16_rn(code * s +
// z) (fp32 fma of the fp16 scale and zero), tokens T_q <= t < S copied from
// the residual ring (slot t mod Rcap).  One thread per (token, 8 channels
// c0 ... c0+7), one 16-byte store per plane.  The codes are read in the
// cache's own order: packed (the 8 codes are b consecutive bytes) or
// MMA-fragment (2 words for keys, 4 for values, by the position functions
// specialised to 8 channels of one 16-channel step).
__global__ void k_dequantize(Geometry geo, Planes pl, LenTable lens,
                             __half *__restrict__ Kh, __half *__restrict__ Vh,
                             int64_t s_stride) {
  const int hd = blockIdx.y, bq = hd / geo.H_kv;
  const int D = geo.D, g = geo.g, NJ = D / g, c8 = D / 8;
  const int Tq = lens.Tq[bq], S = Tq + lens.nres[bq];
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
       i < (int64_t)S * c8; i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / c8), c0 = (int)(i - (int64_t)t * c8) * 8;
    uint4 ko, vo;
    int slot = -1;   // KIVI-Sink: a sink of the quantized region is exact
    for (int j = 0; j < geo.n_sink && t < Tq; ++j)
      if (pl.sink_pos[(size_t)hd * geo.n_sink + j] == t) slot = j;
    if (slot >= 0) {
      const size_t sr = ((size_t)hd * geo.n_sink + slot) * D + c0;
      ko = *reinterpret_cast<const uint4 *>(pl.sink_k + sr);
      vo = *reinterpret_cast<const uint4 *>(pl.sink_v + sr);
    } else if (t < Tq) {
      const size_t r = (size_t)hd * geo.Tcap + t;
      uint32_t kc[8], vc[8];
      codes8(geo, pl.Kc + r * geo.row, pl.Vc + (r - (t & 15)) * geo.row, t & 15,
             c0, kc, vc);
      const size_t kg = ((size_t)hd * (geo.Tcap / g) + t / g) * D + c0;
      const uint4 ksr = *reinterpret_cast<const uint4 *>(pl.Ks + kg);
      const uint4 kzr = *reinterpret_cast<const uint4 *>(pl.Kz + kg);
      const __half *ksh = reinterpret_cast<const __half *>(&ksr);
      const __half *kzh = reinterpret_cast<const __half *>(&kzr);
      const float vs = __half2float(pl.Vs[r * NJ + c0 / g]);
      const float vz = __half2float(pl.Vz[r * NJ + c0 / g]);
      __half kx[8], vx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        kx[e] = __float2half_rn(__fmaf_rn((float)kc[e], __half2float(ksh[e]),
                                          __half2float(kzh[e])));
        vx[e] = __float2half_rn(__fmaf_rn((float)vc[e], vs, vz));
      }
      ko = *reinterpret_cast<const uint4 *>(kx);
      vo = *reinterpret_cast<const uint4 *>(vx);
    } else {
      const size_t slot = ((size_t)hd * geo.Rcap + t % geo.Rcap) * D + c0;
      ko = *reinterpret_cast<const uint4 *>(pl.Kr + slot);
      vo = *reinterpret_cast<const uint4 *>(pl.Vr + slot);
    }
    const size_t o = ((size_t)hd * s_stride + t) * D + c0;
    *reinterpret_cast<uint4 *>(Kh + o) = ko;
    *reinterpret_cast<uint4 *>(Vh + o) = vo;
  }
}

cudaError_t launch_dequantize(const Geometry &geo, const Planes &pl,
                              const int32_t *Tq, const int32_t *nres,
                              __half *Kh, __half *Vh, int64_t s_stride,
                              cudaStream_t st) {
  LenTable lens;
  int64_t smax = 0;
  for (int b = 0; b < geo.B; ++b) {
    lens.Tq[b] = Tq[b];
    lens.nres[b] = nres[b];
    if (Tq[b] + nres[b] > smax) smax = Tq[b] + nres[b];
  }
  if (smax == 0) return cudaSuccess;
  const int64_t items = smax * (geo.D / 8);
  int64_t bx = (items + 255) / 256;
  if (bx > 4096) bx = 4096;
  dim3 grid((unsigned)bx, geo.B * geo.H_kv);
  k_dequantize<<<grid, 256, 0, st>>>(geo, pl, lens, Kh, Vh, s_stride);
  count_launch();
  return cudaGetLastError();
}

}  // namespace vqk
