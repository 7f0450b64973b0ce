// Host side of the tensor-core decode: kernel choice, launch plan (stages,
// persistent grid size) and launch of the decode kernel and of the
// log-sum-exp merge of its per-warp partials (both in decode_mma.cuh).
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

}  // namespace

bool mma_plan(const Geometry &geo, int sm_count, MmaPlan *plan) {
  const int GQ = geo.H_q / geo.H_kv;
  int GQp = 1;
  while (GQp < GQ) GQp *= 2;
  if (GQp > 4 || (geo.D != 64 && geo.D != 128)) return false;
  mma::KernelInfo ki;
  if (!pick(geo, GQp, &ki)) return false;
  // the stage count (2..4) that keeps the most warps resident, and among
  // those the deepest pipeline
  if (cudaFuncSetAttribute((const void *)ki.fn,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           227 * 1024) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  int best_occ = 0, ST = 0;
  uint32_t smem = 0;
  for (int st = 2; st <= mma::kMaxStages; ++st) {
    const uint32_t sm = kNW * (ki.stage0 + st * ki.stage_bytes);
    if (sm > 227 * 1024) break;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, ki.fn, kNW * 32,
                                                      sm) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (occ >= 1 && occ >= best_occ) {
      best_occ = occ;
      ST = st;
      smem = sm;
    }
  }
  if (best_occ < 1) return false;
  const int occ = best_occ;
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
         (geo.D == 64 ? mma::part_stride<64>() : mma::part_stride<128>());
}

cudaError_t launch_decode_mma(const Geometry &geo, const Planes &pl,
                              const MmaPlan &plan, MmaArgs args,
                              const MmaTable &tab, cudaStream_t st) {
  args.GQ = plan.GQ;
  args.GQp = plan.GQp;
  args.KG = plan.KG;
  args.ST = plan.ST;
  // sequences without tokens get an all-zero output (the kernel never
  // visits them)
  for (int b = 0; b < geo.B; ++b) {
    if (tab.nc[b] == 0) {
      cudaError_t e = cudaMemsetAsync(args.out + (size_t)b * geo.H_q * geo.D, 0,
                                      sizeof(float) * geo.H_q * geo.D, st);
      if (e != cudaSuccess) return e;
    }
  }
  if (args.N <= 0) return cudaSuccess;
  mma::KernelInfo ki;
  if (!pick(geo, plan.GQp, &ki)) return cudaErrorInvalidValue;
  int64_t W = plan.warps_max;
  if (W > args.N) W = args.N;
  args.W = (int)W;
  const int grid = (int)((W + kNW - 1) / kNW);
  // both kernels are programmatic dependents of the kernel before them in
  // the stream (they wait for its writes with griddepcontrol.wait), so a
  // launch's set-up overlaps the end of the previous kernel
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kNW * 32);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = st;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, ki.fn, geo, pl, args, tab);
  count_launch();
  if (e != cudaSuccess) return e;
  mma::MergeFn mf = nullptr;
  switch (geo.D * 8 + plan.GQp) {
    case 64 * 8 + 1: mf = mma::merge_fn<64, 1>(); break;
    case 64 * 8 + 2: mf = mma::merge_fn<64, 2>(); break;
    case 64 * 8 + 4: mf = mma::merge_fn<64, 4>(); break;
    case 128 * 8 + 1: mf = mma::merge_fn<128, 1>(); break;
    case 128 * 8 + 2: mf = mma::merge_fn<128, 2>(); break;
    case 128 * 8 + 4: mf = mma::merge_fn<128, 4>(); break;
    default: return cudaErrorInvalidValue;
  }
  // merge warps per CTA: enough for the largest partial count of a head to
  // be read in one round
  int64_t n_max = 1;
  for (int b = 0; b < geo.B; ++b) {
    if (tab.nc[b] == 0) continue;
    for (int h = 0; h < geo.H_kv; ++h) {
      const int64_t cs = tab.bprefix[b] + (int64_t)h * tab.nc[b];
      const int64_t ce = cs + tab.nc[b];
      const int64_t n = (ce * W - 1) / args.N - ((cs + 1) * W - 1) / args.N + 1;
      if (n > n_max) n_max = n;
    }
  }
  int64_t nw = (n_max + mma::kMergeU - 1) / mma::kMergeU;
  if (nw > mma::kMergeWarps) nw = mma::kMergeWarps;
  cfg.gridDim = dim3(geo.B * geo.H_q, geo.D / 32);
  cfg.blockDim = dim3((unsigned)nw * 32);
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, mf, geo, args, tab);
  count_launch();
  return e;
}

}  // namespace vqk
