// KIVI-Sink: choice of the sink tokens of each (sequence, kv head) at
// prefill.
//
// Method: VeloxQuant-MLX changelog v0.9.0 "New" (KIVI-Sink): tokens with
// anomalously large key L2 norms are kept in fp16 and left out of the
// quantization groups' min/max.  Here: the min(n_sink, S) prefill tokens
// with the largest squared key norms, computed in fp32 as a running sum of
// the squares in channel order (each square of an fp16 value is exact in
// fp32; the sums round to nearest), the earlier token first among equal
// norms.  The flush, decode and dequantize kernels read the positions
// (ascending, -1 in unused slots) and the copied fp16 rows.
#include "vqk_internal.cuh"

namespace vqk {
namespace {

constexpr int kPickThreads = 1024;

// (norm, position) order: a larger norm first, then the earlier position
__device__ __forceinline__ bool before(float na, int pa, float nb, int pb) {
  return na > nb || (na == nb && pa < pb);
}

// One CTA per (kv head, sequence).  Each thread keeps the best n of its
// tokens (t = tid, tid + blockDim, ...) in a sorted list; n rounds of a
// block-wide arg-best then pop the overall best n.
__global__ void __launch_bounds__(kPickThreads)
k_pick_sinks(Geometry geo, Planes pl, const __half *__restrict__ K,
             const __half *__restrict__ V, int64_t s_stride, SinkTable tab) {
  __shared__ float red_n[kPickThreads / 32];
  __shared__ int red_p[kPickThreads / 32];
  __shared__ int chosen[kMaxSink];
  const int h = blockIdx.x, b = blockIdx.y;
  const int D = geo.D, n = geo.n_sink, S = tab.S[b];
  const size_t bh = (size_t)b * geo.H_kv + h;
  const __half *Kbh = K + bh * s_stride * D;
  const __half *Vbh = V + bh * s_stride * D;

  float ln[kMaxSink];
  int lp[kMaxSink];
  int cnt = 0;
  for (int t = threadIdx.x; t < S; t += blockDim.x) {
    const uint4 *row = reinterpret_cast<const uint4 *>(Kbh + (size_t)t * D);
    float acc = 0.f;
    for (int q = 0; q < D / 8; ++q) {
      const uint4 u = __ldg(row + q);
      const __half *hv = reinterpret_cast<const __half *>(&u);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x = __half2float(hv[e]);
        acc = __fadd_rn(acc, __fmul_rn(x, x));
      }
    }
    // insert (acc, t) into the sorted list, keeping at most n entries
    if (cnt < n || before(acc, t, ln[cnt - 1], lp[cnt - 1])) {
      int i = cnt < n ? cnt++ : n - 1;
      while (i > 0 && before(acc, t, ln[i - 1], lp[i - 1])) {
        ln[i] = ln[i - 1];
        lp[i] = lp[i - 1];
        --i;
      }
      ln[i] = acc;
      lp[i] = t;
    }
  }

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int head = 0;   // next entry of this thread's list
  for (int r = 0; r < n; ++r) {
    float bn = head < cnt ? ln[head] : -1.f;   // norms are >= 0
    int bp = head < cnt ? lp[head] : 0x7fffffff;
    for (int off = 16; off > 0; off >>= 1) {
      const float on = __shfl_xor_sync(0xffffffffu, bn, off);
      const int op = __shfl_xor_sync(0xffffffffu, bp, off);
      if (before(on, op, bn, bp)) { bn = on; bp = op; }
    }
    if (lane == 0) { red_n[warp] = bn; red_p[warp] = bp; }
    __syncthreads();
    if (warp == 0) {
      bn = lane < nwarps ? red_n[lane] : -1.f;
      bp = lane < nwarps ? red_p[lane] : 0x7fffffff;
      for (int off = 16; off > 0; off >>= 1) {
        const float on = __shfl_xor_sync(0xffffffffu, bn, off);
        const int op = __shfl_xor_sync(0xffffffffu, bp, off);
        if (before(on, op, bn, bp)) { bn = on; bp = op; }
      }
      if (lane == 0) chosen[r] = bn >= 0.f ? bp : -1;
    }
    __syncthreads();
    // the owner of the chosen token moves past it (positions are unique)
    if (head < cnt && lp[head] == chosen[r]) ++head;
  }

  if (threadIdx.x == 0) {
    // ascending positions, unused slots (-1) last
    int m = 0;
    int sorted[kMaxSink];
    for (int r = 0; r < n; ++r)
      if (chosen[r] >= 0) sorted[m++] = chosen[r];
    for (int i = 1; i < m; ++i)
      for (int j = i; j > 0 && sorted[j - 1] > sorted[j]; --j) {
        const int x = sorted[j]; sorted[j] = sorted[j - 1]; sorted[j - 1] = x;
      }
    for (int r = 0; r < n; ++r) {
      const int p = r < m ? sorted[r] : -1;
      chosen[r] = p;
      pl.sink_pos[bh * n + r] = p;
    }
  }
  __syncthreads();
  // copy the sinks' rows (unused slots are zero)
  for (int i = threadIdx.x; i < n * D; i += blockDim.x) {
    const int r = i / D, c = i - r * D;
    const int p = chosen[r];
    const __half zero = __float2half_rn(0.f);
    pl.sink_k[(bh * n + r) * D + c] = p >= 0 ? Kbh[(size_t)p * D + c] : zero;
    pl.sink_v[(bh * n + r) * D + c] = p >= 0 ? Vbh[(size_t)p * D + c] : zero;
  }
}

}  // namespace

cudaError_t launch_pick_sinks(const Geometry &geo, const Planes &pl,
                              const __half *K, const __half *V,
                              int64_t s_stride, const SinkTable &tab,
                              cudaStream_t st) {
  if (geo.n_sink <= 0) return cudaSuccess;
  dim3 grid(geo.H_kv, geo.B);
  k_pick_sinks<<<grid, kPickThreads, 0, st>>>(geo, pl, K, V, s_stride, tab);
  count_launch();
  return cudaGetLastError();
}

}  // namespace vqk
