// Kitty: channel-wise mixed-precision keys (4-bit channels of high running
// variance, 2-bit for the rest) and fp16 values: its flush and the launch
// of its fused decode (kitty_decode.cuh).
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
#include "kitty_decode.cuh"
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

// The ranking is a scan over a flush's groups (a group's ranking uses the
// running sums through its last token), cut into C chunks per (sequence,
// kv head) so that it spreads over the GPU: k_kitty_chunk_sums sums each
// chunk's keys, k_kitty_rank ranks each chunk's groups from the running
// sums before the chunk (the cache's sums plus the earlier chunks' totals),
// k_kitty_sums_update adds every chunk's total to the cache's sums.  The
// totals (int64 sum m, 128-bit sum m^2 as two words, per channel) sit in a
// scratch area of 3 * D words per (sequence, kv head, chunk).
constexpr int kRankThreads = 1024;

// groups [k0, k1) of chunk ch of sequence b's n groups
__device__ __forceinline__ void chunk_range(int n, int C, int ch, int &k0, int &k1) {
  k0 = (int)((int64_t)n * ch / C);
  k1 = (int)((int64_t)n * (ch + 1) / C);
}

// One CTA of kRankThreads per (chunk, kv head, sequence): NS = kRankThreads
// / D slices of one thread per channel take the chunk's groups NS apart and
// sum their keys (the rows' loads in flight together); the slices' sums are
// added in shared memory.
__global__ void __launch_bounds__(kRankThreads)
k_kitty_chunk_sums(Geometry geo, Planes pl, const __half *__restrict__ Kin,
                   int64_t in_stride, FlushTable tab, int C,
                   unsigned long long *__restrict__ scratch) {
  __shared__ unsigned long long r1[kRankThreads], r2lo[kRankThreads], r2hi[kRankThreads];
  const int D = geo.D, g = geo.g, NS = kRankThreads / D;
  const int c = threadIdx.x % D, sl = threadIdx.x / D;
  const int ch = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int n = tab.prefix[b + 1] - tab.prefix[b];
  int k0, k1;
  chunk_range(n, C, ch, k0, k1);
  const size_t bh = (size_t)b * geo.H_kv + h;
  const int split = tab.src_split[b];
  long long s1 = 0;
  u128 s2 = 0;
  for (int k = k0 + sl; k < k1; k += NS) {
    const int P0 = tab.first_pos[b] + k * g;
#pragma unroll 8
    for (int i = 0; i < g; ++i) {
      const __half *row = src_row(geo, pl, Kin, in_stride, bh, P0 + i, split);
      const long long m = f16_units(__half_as_ushort(row[c]));
      s1 += m;
      s2 += (u128)((__int128)m * m);
    }
  }
  r1[threadIdx.x] = (unsigned long long)s1;
  r2lo[threadIdx.x] = (unsigned long long)s2;
  r2hi[threadIdx.x] = (unsigned long long)(s2 >> 64);
  __syncthreads();
  if (sl == 0) {
    for (int j = 1; j < NS; ++j) {
      s1 += (long long)r1[j * D + c];
      s2 += ((u128)r2hi[j * D + c] << 64) | r2lo[j * D + c];
    }
    unsigned long long *dst = scratch + ((bh * C + ch) * 3) * D;
    dst[c] = (unsigned long long)s1;
    dst[D + c] = (unsigned long long)s2;
    dst[2 * D + c] = (unsigned long long)(s2 >> 64);
  }
}

// One CTA of kRankThreads per (chunk, kv head, sequence): the running sums
// before the chunk, then its groups NS at a time: each slice sums its
// group's keys, the slices' sums are carried in shared memory (slice j adds
// slices 0 ... j to the running sums), and every slice ranks its channels by
// the running variance through its group's last token.
__global__ void __launch_bounds__(kRankThreads)
k_kitty_rank(Geometry geo, Planes pl, const __half *__restrict__ Kin,
             int64_t in_stride, FlushTable tab, int C,
             const unsigned long long *__restrict__ scratch) {
  extern __shared__ unsigned long long rsm[];
  const int D = geo.D, g = geo.g, NS = kRankThreads / D;
  const int c = threadIdx.x % D, sl = threadIdx.x / D;
  // per (slice, channel): the group's sums, then the running variance
  unsigned long long *q1 = rsm, *q2lo = q1 + NS * D, *q2hi = q2lo + NS * D;
  unsigned long long *vlo = q2hi + NS * D, *vhi = vlo + NS * D;
  const int ch = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int n = tab.prefix[b + 1] - tab.prefix[b];
  int kb, ke;
  chunk_range(n, C, ch, kb, ke);
  if (kb >= ke) return;
  const size_t bh = (size_t)b * geo.H_kv + h;
  long long s1 = pl.ksum[bh * D + c];
  u128 s2 = ((u128)pl.ksq[(bh * D + c) * 2 + 1] << 64) | pl.ksq[(bh * D + c) * 2];
  for (int j = 0; j < ch; ++j) {
    const unsigned long long *t = scratch + ((bh * C + j) * 3) * D;
    s1 += (long long)t[c];
    s2 += ((u128)t[2 * D + c] << 64) | t[D + c];
  }
  const int split = tab.src_split[b];
  for (int k0 = kb; k0 < ke; k0 += NS) {
    const int k = k0 + sl;
    const int P0 = tab.first_pos[b] + k * g;
    long long g1 = 0;
    u128 g2 = 0;
    if (k < ke) {
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
    if (k < ke) {
      const u128 N = (u128)(P0 + g);
      const u128 a = (u128)(r1 < 0 ? -r1 : r1);
      var = N * r2 - a * a;
    }
    vlo[sl * D + c] = (unsigned long long)var;
    vhi[sl * D + c] = (unsigned long long)(var >> 64);
    __syncthreads();
    if (k < ke) {
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
}

// The cache's running sums += every chunk's total: one thread per (channel,
// kv head, sequence).
__global__ void k_kitty_sums_update(Geometry geo, Planes pl, FlushTable tab, int C,
                                    const unsigned long long *__restrict__ scratch) {
  const int D = geo.D;
  const int c = threadIdx.x, h = blockIdx.x, b = blockIdx.y;
  if (tab.prefix[b + 1] == tab.prefix[b]) return;
  const size_t bh = (size_t)b * geo.H_kv + h;
  long long s1 = pl.ksum[bh * D + c];
  u128 s2 = ((u128)pl.ksq[(bh * D + c) * 2 + 1] << 64) | pl.ksq[(bh * D + c) * 2];
  for (int j = 0; j < C; ++j) {
    const unsigned long long *t = scratch + ((bh * C + j) * 3) * D;
    s1 += (long long)t[c];
    s2 += ((u128)t[2 * D + c] << 64) | t[D + c];
  }
  pl.ksum[bh * D + c] = s1;
  pl.ksq[(bh * D + c) * 2] = (unsigned long long)s2;
  pl.ksq[(bh * D + c) * 2 + 1] = (unsigned long long)(s2 >> 64);
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

}  // namespace

static kitdec::KitKernel pick_kitty_kernel(const Geometry &geo) {
  const int gq = geo.H_q / geo.H_kv;
  if (geo.D == 64) return kitdec::pick_d64(gq);
  if (geo.D == 128) return kitdec::pick_d128(gq);
  return {};
}

cudaError_t launch_flush_kitty(const Geometry &geo, const Planes &pl,
                               const __half *Kin, const __half *Vin,
                               int64_t in_stride, const FlushTable &tab,
                               int total_groups, cudaStream_t st) {
  if (total_groups <= 0) return cudaSuccess;
  // chunks per (sequence, kv head): enough CTAs to spread over the GPU,
  // each chunk at least a step of NS groups, the totals within the decode's
  // partial buffer (idle during a flush; part_floats(geo) floats, at least
  // one chunk's totals)
  const int NS = kRankThreads / geo.D;
  int n_max = 0;
  for (int b = 0; b < geo.B; ++b) {
    const int n = tab.prefix[b + 1] - tab.prefix[b];
    if (n > n_max) n_max = n;
  }
  const size_t part_words = part_floats(geo) / 2;
  const size_t per_chunk = kitty_chunk_words(geo);
  int C = n_max / NS;
  if (C > 16) C = 16;
  if ((size_t)C * per_chunk > part_words) C = (int)(part_words / per_chunk);
  if (C < 1) C = 1;
  unsigned long long *scratch = reinterpret_cast<unsigned long long *>(pl.part);
  const dim3 grid(C, geo.H_kv, geo.B);
  k_kitty_chunk_sums<<<grid, kRankThreads, 0, st>>>(geo, pl, Kin, in_stride, tab, C, scratch);
  count_launch();
  const size_t rsmem = (size_t)5 * kRankThreads * sizeof(unsigned long long);
  if (rsmem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_kitty_rank, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)rsmem);
    if (e != cudaSuccess) return e;
  }
  k_kitty_rank<<<grid, kRankThreads, rsmem, st>>>(geo, pl, Kin, in_stride, tab, C, scratch);
  count_launch();
  k_kitty_sums_update<<<dim3(geo.H_kv, geo.B), geo.D, 0, st>>>(geo, pl, tab, C, scratch);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)geo.g * (geo.D + geo.kitty_hi) / 4;
  k_flush_kitty<<<dim3(total_groups, geo.H_kv), geo.D, smem, st>>>(geo, pl, Kin, Vin,
                                                                   in_stride, tab);
  count_launch();
  return cudaGetLastError();
}

int kitty_decode_ctas_per_sm(const Geometry &geo) {
  const kitdec::KitKernel kf = pick_kitty_kernel(geo);
  return kf.occ > 0 ? kf.occ : 1;
}

// The split is planned for one wave (as the AgeTieredKV decode's): the
// dynamic shared memory request is padded until an SM holds at most
// ceil(CTAs / SMs) CTAs, so that the block scheduler cannot stack some SMs
// fuller than others.
cudaError_t launch_decode_kitty(const Geometry &geo, const Planes &pl,
                                const DecodeArgs &args, const DecodeTable &tab,
                                cudaStream_t st) {
  if (args.total_items > 0) {
    const kitdec::KitKernel kf = pick_kitty_kernel(geo);
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
                         dim3(kitdec::kThreads), params, smem, st);
    count_launch();
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_combine(geo, pl, args, tab, st);
}

}  // namespace vqk
