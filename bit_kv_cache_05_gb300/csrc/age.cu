// AgeTieredKV: quantization width by token age (three tiers of the KIVI
// group quantizer): its flush (quantize and demote), the export of its code
// planes and the launch of its fused decode (age_decode.cuh).
//
// Method: VeloxQuant-MLX method overview, AgeTieredKV entry (three tiers,
// default 8 / 4 / 2 bits, chosen by current position minus token position
// against two boundaries, default 128 and 1024 tokens; the shared min/max
// group quantizer of KIVI), on the KIVI cache of changelog v0.8.0 (keys per
// channel over g tokens, values per token over g channels).  A group's age
// counts from its newest token; a group enters at the top tier and moves
// down one tier at a time, re-quantized from its values rebuilt in fp32
// (code * scale rounded, then + zero rounded), so that a prefill and any
// chunking of appends give the same cache.  A group owns g * D bytes of
// each code plane; at width w its rows (D * w / 8 bytes, codes LSB first)
// are packed densely from the start of that block, so that a decode reads
// only the group's bytes (rows of D bytes with the codes in their leading
// bytes made DRAM fetch every row's whole line: 2.9x the bytes at 2 bits).
// The export expands the rows to D bytes.
#include "age_decode.cuh"

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
    const int w = age_width(geo, t);
    const uint32_t m = (1u << w) - 1u;
    for (int idx = c; idx < g * D; idx += blockDim.x) {
      const int i = idx / D, ch = idx - i * D;
      const int bit = ch * w;
      const size_t ro = age_row_off(geo, bh, G, i, w) + (bit >> 3);
      const uint8_t kb = pl.Kc[ro];
      const uint8_t vb = pl.Vc[ro];
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
    const int levels = (1 << age_width(geo, t)) - 1;
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
  // rows packed densely at the final width (the group block's leading
  // g * D * w / 8 bytes); every read of the old rows is behind the
  // barriers above, so the block is rewritten in place
  const int w = age_width(geo, t_to);
  const int per = 32 / w, wpr = D * w / 32;                // fields, words per row
  for (int idx = c; idx < g * wpr; idx += blockDim.x) {
    const int i = idx / wpr, k = idx - i * wpr;
    uint32_t ak = 0, av = 0;
    for (int e = 0; e < per; ++e) {
      ak |= (uint32_t)ck[i * D + k * per + e] << (w * e);
      av |= (uint32_t)cv[i * D + k * per + e] << (w * e);
    }
    const size_t wo = age_row_off(geo, bh, G, i, w) / 4 + k;
    reinterpret_cast<uint32_t *>(pl.Kc)[wo] = ak;
    reinterpret_cast<uint32_t *>(pl.Vc)[wo] = av;
  }
  if (c == 0) pl.tier[bh * (geo.Tcap / g) + G] = (int8_t)t_to;
}

// D-byte rows of an AgeTieredKV code plane (the packed row order the oracle
// and the export use): one thread per 32-bit word of the output.
__global__ void k_age_export(Geometry geo, const uint8_t *__restrict__ src,
                             const int8_t *__restrict__ tier, LenTable lens,
                             uint32_t *__restrict__ dst) {
  const int D = geo.D, wrow = D / 4;
  const size_t words = (size_t)geo.B * geo.H_kv * geo.Tcap * wrow;
  for (size_t x = (size_t)blockIdx.x * blockDim.x + threadIdx.x; x < words;
       x += (size_t)gridDim.x * blockDim.x) {
    const size_t r = x / wrow;
    const int k = (int)(x - r * wrow);
    const size_t bh = r / geo.Tcap;
    const int t = (int)(r - bh * geo.Tcap);
    const int b = (int)(bh / geo.H_kv);
    uint32_t v = 0;
    if (t < lens.Tq[b]) {
      const int G = t / geo.g, i = t - G * geo.g;
      const int w = age_width(geo, tier[bh * (geo.Tcap / geo.g) + G]);
      if (k < D * w / 32)
        v = reinterpret_cast<const uint32_t *>(src + age_row_off(geo, bh, G, i, w))[k];
    }
    dst[x] = v;
  }
}

}  // namespace

using agedec::AgeKernel;

static AgeKernel pick_age_kernel(const Geometry &geo) {
  const int gq = geo.H_q / geo.H_kv;
  if (geo.D == 64) return agedec::pick_d64(gq);
  if (geo.D == 128) return agedec::pick_d128(gq);
  return {};
}

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

cudaError_t launch_age_export(const Geometry &geo, const Planes &pl, bool values,
                              void *dst, const int32_t *Tq, cudaStream_t st) {
  LenTable lens;
  for (int b = 0; b < geo.B; ++b) { lens.Tq[b] = Tq[b]; lens.nres[b] = 0; }
  k_age_export<<<1024, 256, 0, st>>>(geo, values ? pl.Vc : pl.Kc, pl.tier, lens,
                                     (uint32_t *)dst);
  count_launch();
  return cudaGetLastError();
}

int age_decode_ctas_per_sm(const Geometry &geo) {
  const AgeKernel kf = pick_age_kernel(geo);
  return kf.occ > 0 ? kf.occ : 1;
}

// The split is planned for one wave: a launch of fewer CTAs than the SMs
// hold would let the block scheduler stack some SMs fuller than others, so
// the dynamic shared memory request is padded until an SM holds at most
// ceil(CTAs / SMs) of them.
cudaError_t launch_decode_age(const Geometry &geo, const Planes &pl,
                              const DecodeArgs &args, const DecodeTable &tab,
                              cudaStream_t st) {
  if (args.total_items > 0) {
    const AgeKernel kf = pick_age_kernel(geo);
    if (!kf.f) return cudaErrorInvalidValue;
    int dev = 0, sms = 0, smem_sm = 0, reserved = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess) return e;
    const int64_t ctas = (int64_t)args.total_items * geo.H_kv;
    const int64_t occ = (ctas + sms - 1) / (sms > 0 ? sms : 1);
    size_t smem = (size_t)kf.smem;
    if (occ >= 1 && occ < kf.occ) {
      const int64_t per = ((int64_t)smem_sm / occ - reserved - kf.smem_static) / 128 * 128;
      if (per > (int64_t)smem) smem = (size_t)per;
    }
    Geometry g2 = geo;
    Planes p2 = pl;
    DecodeArgs a2 = args;
    DecodeTable t2 = tab;
    void *params[] = {&g2, &p2, &a2, &t2};
    e = cudaLaunchKernel(kf.f, dim3(args.total_items, geo.H_kv),
                         dim3(agedec::kDecodeThreads), params, smem, st);
    count_launch();
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_combine(geo, pl, args, tab, st);
}

}  // namespace vqk
