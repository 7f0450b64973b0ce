// Decode entry point that allocates nothing: vq_kivi_decode_attend_static.
//
// Who needs it: programs that are not allowed to call cudaMalloc once they
// are running -- inference engines that reserve all device memory at
// start-up and hand out only their own pool, plugins whose host forbids
// allocations, and latency-critical loops where cudaMalloc would
// synchronize the device.  They keep the cache planes in memory they own and
// call this entry point with plain pointers.  Its only scratch (the split-KV
// partial results) lives in the fixed-size device array below, which every
// GPU that loads this library holds until the process exits.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "vqk_internal.cuh"

namespace vqk {
namespace {

constexpr size_t kScratchBytes = VQ_KIVI_STATIC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep alignment");

// The scratch.  Host code must not pass `g_scratch` itself to a kernel: on the
// host that name is only a stand-in; the device address comes from
// cudaGetSymbolAddress (per device, in scratch_address below).
__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

int fail_static(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  set_last_error(buf);  // read back with vq_kivi_last_error()
  return code;
}

// Device address of the scratch array on `dev` (which must be current):
// looked up once per device, on that device's first call.
cudaError_t scratch_address(int dev, void **out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace vqk

using namespace vqk;

extern "C" int vq_kivi_decode_attend_static(
    const vq_kivi_params *p, const vq_kivi_planes *planes,
    const int32_t *seq_lens, const void *q, float *out, float softmax_scale,
    void *stream) {
  if (!p || !planes || !seq_lens || !q || !out)
    return fail_static(VQ_ERR_ARG, "NULL argument");
  if (p->B < 1 || p->B > kMaxB || p->H_kv < 1 || p->H_q < 1 ||
      p->H_q % p->H_kv != 0 || p->H_q / p->H_kv > kMaxGroupHeads ||
      (p->D != 64 && p->D != 128 && p->D != 256) ||
      (p->bits != 2 && p->bits != 4 && p->bits != 8) ||
      (p->group != 16 && p->group != 32 && p->group != 64 &&
       p->group != 128) ||
      p->D % p->group != 0 || p->residual < 0 || p->residual > 4096 ||
      p->max_seq < 0 || p->max_seq > (1 << 24))
    return fail_static(VQ_ERR_UNSUPPORTED, "unsupported parameters");
  if (!std::isfinite(softmax_scale))
    return fail_static(VQ_ERR_ARG, "softmax_scale is not finite");
  const void *ptrs[8] = {planes->Kc, planes->Ks, planes->Kz, planes->Vc,
                         planes->Vs, planes->Vz, planes->Kr, planes->Vr};
  for (const void *ptr : ptrs)
    if (!ptr || !aligned16(ptr))
      return fail_static(VQ_ERR_ARG, "plane pointers must be non-NULL and "
                         "16-byte aligned");
  if (!aligned16(q) || !aligned16(out))
    return fail_static(VQ_ERR_ARG, "q and out must be 16-byte aligned");

  const int g = p->group;
  Geometry geo;
  geo.B = p->B; geo.H_q = p->H_q; geo.H_kv = p->H_kv; geo.D = p->D;
  geo.bits = p->bits; geo.g = g; geo.R = p->residual;
  geo.Tcap = ((p->max_seq > 0 ? p->max_seq : 1) + g - 1) / g * g;
  geo.Rcap = p->residual + g;
  geo.row = p->D * p->bits / 8;

  // Split size: as many work items per sequence as the scratch holds.
  const size_t per_item = (size_t)p->B * p->H_q * (p->D + 2) * sizeof(float);
  const int64_t max_items = (int64_t)(kScratchBytes / per_item);
  if (max_items < 2)
    return fail_static(VQ_ERR_CAPACITY, "B*H_q*(D+2)*4 = %zu bytes exceeds "
                       "the static scratch (%zu bytes) for two work items",
                       per_item, kScratchBytes);
  int64_t total_tq = 0;
  int32_t Tq[kMaxB], nres[kMaxB];
  for (int b = 0; b < p->B; ++b) {
    const int32_t S = seq_lens[b];
    if (S < 0 || S > p->max_seq)
      return fail_static(VQ_ERR_CAPACITY, "seq_lens[%d]=%d outside [0, %d]",
                         b, S, p->max_seq);
    Tq[b] = S < p->residual ? 0 : g * ((S - p->residual) / g);
    nres[b] = S - Tq[b];
    total_tq += Tq[b];
  }
  int dev = -1, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess)
    return fail_static(VQ_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fail_static(VQ_ERR_UNSUPPORTED, "device index %d >= %d", dev,
                       kMaxDevices);
  const int32_t unit = g > 64 ? g : 64;
  int64_t tps = (total_tq * p->H_kv + 4LL * sms - 1) / (4LL * sms);
  tps = (tps + unit - 1) / unit * unit;
  if (tps < 256) tps = 256;
  int32_t tq_max = 0;
  for (int b = 0; b < p->B; ++b) tq_max = Tq[b] > tq_max ? Tq[b] : tq_max;
  const int64_t q_items_cap = max_items - 1;  // one item left for the residual
  const int64_t tps_floor = (tq_max + q_items_cap - 1) / q_items_cap;
  if (tps < tps_floor) tps = (tps_floor + unit - 1) / unit * unit;
  geo.max_items = (int)max_items;

  void *scratch = nullptr;
  e = scratch_address(dev, &scratch);
  if (e != cudaSuccess)
    return fail_static(VQ_ERR_CUDA, "cudaGetSymbolAddress: %s",
                       cudaGetErrorString(e));

  Planes pl;
  pl.Kc = (uint8_t *)planes->Kc;
  pl.Ks = (__half *)planes->Ks;
  pl.Kz = (__half *)planes->Kz;
  pl.Vc = (uint8_t *)planes->Vc;
  pl.Vs = (__half *)planes->Vs;
  pl.Vz = (__half *)planes->Vz;
  pl.Kr = (__half *)planes->Kr;
  pl.Vr = (__half *)planes->Vr;
  pl.part = (float *)scratch;
  pl.ksmax = nullptr;   // only the tensor-core decode reads it

  DecodeTable tab;
  tab.prefix[0] = 0;
  for (int b = 0; b < p->B; ++b) {
    tab.Tq[b] = Tq[b];
    tab.nres[b] = nres[b];
    tab.nq[b] = (int32_t)((Tq[b] + tps - 1) / tps);
    tab.prefix[b + 1] = tab.prefix[b] + tab.nq[b] + (nres[b] > 0 ? 1 : 0);
  }
  DecodeArgs args;
  args.q = (const __half *)q;
  args.out = out;
  const float scale = softmax_scale > 0.f ? softmax_scale
                                          : 1.0f / std::sqrt((float)p->D);
  args.scale_log2 = scale * 1.4426950408889634f;
  args.tps = (int)tps;
  args.total_items = tab.prefix[p->B];
  e = launch_decode(geo, pl, args, tab, (cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail_static(VQ_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return VQ_OK;
}
