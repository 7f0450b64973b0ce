// Host side of the tensor-core decode: kernel choice, launch plan (stages,
// persistent grid size), launch, and the log-sum-exp merge of the partials.
// The kernel itself is in decode_mma.cuh.
#include "decode_mma.cuh"

namespace vqk {
namespace {

using mma::kNW;

bool pick(const Geometry &geo, int GQp, mma::KernelInfo *ki) {
  switch (geo.bits) {
    case 2: return mma::kernel_b2(geo.D, GQp, geo.g, ki);
    case 4: return mma::kernel_b4(geo.D, GQp, geo.g, ki);
    case 8: return mma::kernel_b8(geo.D, GQp, geo.g, ki);
    default: return false;
  }
}

// out[b][hq] = sum_w 2^(m_w - M) o_w / sum_w 2^(m_w - M) l_w over the warps w
// whose chunk range touches head hd = b*H_kv + hq/GQ (partial slot w + hd)
__global__ void k_combine_mma(Geometry geo, MmaArgs args, MmaTable tab) {
  const int b = blockIdx.x / geo.H_q, hq = blockIdx.x % geo.H_q;
  const int D = geo.D, GQ = args.GQ;
  const int h = hq / GQ, hh = hq % GQ;
  const int hd = b * geo.H_kv + h;
  const int nc = tab.nc[b];
  float *out = args.out + ((size_t)b * geo.H_q + hq) * D;
  if (nc == 0) {
    for (int c = threadIdx.x; c < D; c += blockDim.x) out[c] = 0.f;
    return;
  }
  const int64_t N = args.N, W = args.W;
  const int64_t cs = tab.bprefix[b] + (int64_t)h * nc, ce = cs + nc;
  const int w0 = (int)(((cs + 1) * W - 1) / N);
  const int w1 = (int)((ce * W - 1) / N);
  auto entry = [&](int w) {
    return args.part + ((size_t)(w + hd) * args.GQp + hh) * (D + 2);
  };
  float M = -INFINITY;
  for (int w = w0; w <= w1; ++w) M = fmaxf(M, entry(w)[D]);
  float Lsum = 0.f;
  for (int w = w0; w <= w1; ++w) Lsum += exp2f(entry(w)[D] - M) * entry(w)[D + 1];
  const float inv = 1.0f / Lsum;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float acc = 0.f;
    for (int w = w0; w <= w1; ++w) acc += exp2f(entry(w)[D] - M) * entry(w)[c];
    out[c] = acc * inv;
  }
}

}  // namespace

bool mma_plan(const Geometry &geo, int sm_count, MmaPlan *plan) {
  const int GQ = geo.H_q / geo.H_kv;
  int GQp = 1;
  while (GQp < GQ) GQp *= 2;
  if (GQp > 4 || (geo.D != 64 && geo.D != 128)) return false;
  mma::KernelInfo ki;
  if (!pick(geo, GQp, &ki)) return false;
  // as many stages (2..4) as keep two CTAs per SM, else fewer CTAs
  int ST = mma::kMaxStages;
  const uint32_t budget2 = 110 * 1024;
  while (ST > 2 && kNW * (ki.stage0 + ST * ki.stage_bytes) > budget2) --ST;
  const uint32_t smem = kNW * (ki.stage0 + ST * ki.stage_bytes);
  if (smem > 227 * 1024) return false;
  if (cudaFuncSetAttribute((const void *)ki.fn,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, ki.fn, kNW * 32,
                                                    smem) != cudaSuccess ||
      occ < 1) {
    cudaGetLastError();
    return false;
  }
  plan->GQ = GQ;
  plan->GQp = GQp;
  plan->KG = 0;
  plan->ST = ST;
  plan->smem = smem;
  plan->warps_max = sm_count * occ * kNW;
  plan->chunk = mma::kC;
  return true;
}

size_t mma_part_floats(const Geometry &geo, const MmaPlan &plan) {
  return ((size_t)plan.warps_max + (size_t)geo.B * geo.H_kv) * plan.GQp *
         (geo.D + 2);
}

cudaError_t launch_decode_mma(const Geometry &geo, const Planes &pl,
                              const MmaPlan &plan, MmaArgs args,
                              const MmaTable &tab, cudaStream_t st) {
  args.GQ = plan.GQ;
  args.GQp = plan.GQp;
  args.KG = plan.KG;
  args.ST = plan.ST;
  if (args.N > 0) {
    mma::KernelInfo ki;
    if (!pick(geo, plan.GQp, &ki)) return cudaErrorInvalidValue;
    int64_t W = plan.warps_max;
    if (W > args.N) W = args.N;
    args.W = (int)W;
    const int grid = (int)((W + kNW - 1) / kNW);
    ki.fn<<<grid, kNW * 32, plan.smem, st>>>(geo, pl, args, tab);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  } else {
    args.W = 1;
  }
  k_combine_mma<<<geo.B * geo.H_q, geo.D, 0, st>>>(geo, args, tab);
  count_launch();
  return cudaGetLastError();
}

}  // namespace vqk
