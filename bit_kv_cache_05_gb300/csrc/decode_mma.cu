// Host side of the tensor-core decode: kernel choice, launch plan (stages,
// persistent grid size) and launch of the decode kernel and of the
// log-sum-exp merge of its per-warp partials (both in decode_mma.cuh).
#include <mutex>

#include "decode_mma.cuh"

namespace vqk {
namespace {

using mma::kNW;

bool pick(const Geometry &geo, int GQp, mma::KernelInfo *ki) {
  const bool sink = geo.n_sink > 0;   // KIVI-Sink: the masking instantiation
  switch (geo.bits) {
    case 2: return sink ? mma::kernel_sink_b2(geo.D, GQp, geo.g, ki)
                        : mma::kernel_b2(geo.D, GQp, geo.g, ki);
    case 4: return sink ? mma::kernel_sink_b4(geo.D, GQp, geo.g, ki)
                        : mma::kernel_b4(geo.D, GQp, geo.g, ki);
    case 8: return sink ? mma::kernel_sink_b8(geo.D, GQp, geo.g, ki)
                        : mma::kernel_b8(geo.D, GQp, geo.g, ki);
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
  // the stage count (1..4) that keeps the most warps resident, and among
  // those the deepest pipeline (one stage per warp still streams: the other
  // resident warps' copies hide a warp's own copy latency, and for wide
  // codes it is what lets 16 warps share an SM's shared memory)
  if (cudaFuncSetAttribute((const void *)ki.fn,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           227 * 1024) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  int best_occ = 0, ST = 0;
  uint32_t smem = 0;
  for (int st = 1; st <= mma::kMaxStages; ++st) {
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
  plan->sm_count = sm_count;
  plan->chunk = mma::kC;
  return true;
}

// resident CTAs per SM of a merge kernel at nw warps per CTA (cached; the
// cache is shared by every thread of the process)
static int merge_ctas_per_sm(mma::MergeFn mf, int nw) {
  struct Entry { mma::MergeFn fn; int nw, occ; };
  static Entry cache[64];
  static int used = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].fn == mf && cache[i].nw == nw) return cache[i].occ;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, (const void *)mf, nw * 32, 0) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (used < 64) cache[used++] = Entry{mf, nw, occ};
  return occ;
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
  // sequences without any token get an all-zero output (no kernel writes it)
  for (int b = 0; b < geo.B; ++b) {
    if (tab.nq[b] == 0 && tab.nres[b] == 0) {
      cudaError_t e = cudaMemsetAsync(args.out + (size_t)b * geo.H_q * geo.D, 0,
                                      sizeof(float) * geo.H_q * geo.D, st);
      if (e != cudaSuccess) return e;
    }
  }
  // both kernels are programmatic dependents of the kernel before them in
  // the stream (they wait for its writes with griddepcontrol.wait), so a
  // launch's set-up overlaps the end of the previous kernel
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = st;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t e = cudaSuccess;
  int64_t W = 1;
  if (args.N > 0) {
    mma::KernelInfo ki;
    if (!pick(geo, plan.GQp, &ki)) return cudaErrorInvalidValue;
    W = plan.warps_max;
    if (W > args.N) W = args.N;
    args.W = (int)W;
    cfg.gridDim = dim3((unsigned)((W + kNW - 1) / kNW));
    cfg.blockDim = dim3(kNW * 32);
    cfg.dynamicSmemBytes = plan.smem;
    e = cudaLaunchKernelEx(&cfg, ki.fn, geo, pl, args, tab);
    count_launch();
    if (e != cudaSuccess) return e;
  } else {
    args.W = 1;
  }
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
  // merge warps per CTA (one query head, one channel slice): enough for the
  // largest partial count of a head to be read in one round, and more, up
  // to what reads the longest residual window in one round, only while
  // every CTA of the grid still fits on the device at once (a second wave
  // costs more than a second round of the window)
  const int GQ = plan.GQ;
  int64_t per = 1, nr = 1;
  bool any = false;
  for (int b = 0; b < geo.B; ++b) {
    if (tab.nq[b] == 0 && tab.nres[b] == 0) continue;
    any = true;
    const int64_t wr = (tab.nres[b] + mma::kMergeRT - 1) / mma::kMergeRT;
    if (wr > nr) nr = wr;
    if (tab.nq[b] == 0) continue;
    for (int h = 0; h < geo.H_kv; ++h) {
      const int64_t cs = tab.bprefix[b] + (int64_t)h * tab.nc[b];
      const int64_t ce = cs + tab.nc[b];
      const int64_t n = (ce * W - 1) / args.N - ((cs + 1) * W - 1) / args.N + 1;
      const int64_t wn = (n + mma::kMergeU - 1) / mma::kMergeU;
      if (wn > per) per = wn;
    }
  }
  if (!any) return cudaSuccess;
  const int64_t per_max = mma::kMergeWarps;
  if (per > per_max) per = per_max;
  if (nr > per_max) nr = per_max;
  const int nsl = geo.D == 64 ? (plan.GQp == 4 ? 1 : 2) : 4 / plan.GQp;
  const int64_t ctas = (int64_t)geo.B * geo.H_kv * GQ * nsl;
  for (int64_t pr = nr; pr > per; --pr) {
    if ((int64_t)merge_ctas_per_sm(mf, (int)pr) * plan.sm_count >= ctas) {
      per = pr;
      break;
    }
  }
  cfg.gridDim = dim3(geo.B * geo.H_kv, GQ, nsl);
  cfg.blockDim = dim3((unsigned)per * 32);
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, mf, geo, pl, args, tab);
  count_launch();
  return e;
}

}  // namespace vqk
