// C ABI of the KIVI cache: argument checks, the cache handle, device memory
// and the launch sequence of each call.  See include/vq_kivi.h.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "vqk_internal.cuh"

using namespace vqk;

// vq_kivi_step_host's state: the device slot for a step's inputs (the
// token's K and V at 0 and off_v, the query at off_q).
struct StepIO {
  void *slot = nullptr;
  std::vector<int32_t> ones;
  size_t off_v = 0, off_q = 0;
};

static void free_step_io(StepIO *io) {
  if (!io) return;
  if (io->slot) cudaFree(io->slot);   // waits for the kernels using it
  delete io;
}

struct vq_kivi_cache {
  vq_kivi_params p;
  Geometry geo;
  Planes pl;
  void *block;
  size_t block_bytes;
  int device;
  int sm_count;
  cudaStream_t last_stream;
  int32_t split_tokens;   // 0 = automatic
  int32_t tps_min;        // smallest split the workspace allows
  bool use_mma;           // tensor-core decode kernel for this shape
  int32_t fail_chunk;     // testing hook, -1 = off
  bool flush_last;        // the last kernel launched for this cache is a
                          // k_flush (it may still be writing planes when a
                          // programmatic dependent starts)
  MmaPlan plan;
  unsigned *err;          // device word set by a kernel whose wait gave up
  int32_t S[kMaxB], Tq[kMaxB], nres[kMaxB];
  // AgeTieredKV and Kitty: the automatic split last planned and the T_q it was
  // planned for (the plan is a search, redone when a flush moves T_q)
  int32_t age_tps;
  int32_t age_Tq[kMaxB];
  StepIO *io;             // vq_kivi_step_host's slots (first call)
  // the multi-query attend's key-range partials (grown on demand)
  void *mq_scratch;
  size_t mq_scratch_bytes;
};

namespace {

thread_local std::string g_err;
std::atomic<uint64_t> g_launches{0};

int fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char *what) {
  return fail(VQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

int32_t n_quantized(int32_t S, int32_t R, int32_t g) {
  if (S < R) return 0;
  return g * ((S - R) / g);
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int check_params(const vq_kivi_params *p) {
  if (!p) return fail(VQ_ERR_ARG, "params is NULL");
  if (p->B < 1 || p->H_q < 1 || p->H_kv < 1 || p->D < 1 || p->group < 1 ||
      p->residual < 0 || p->max_seq < 0)
    return fail(VQ_ERR_ARG, "params: sizes must be positive (B=%d H_q=%d "
                "H_kv=%d D=%d group=%d residual=%d max_seq=%d)", p->B, p->H_q,
                p->H_kv, p->D, p->group, p->residual, p->max_seq);
  if (p->B > kMaxB) return fail(VQ_ERR_UNSUPPORTED, "B=%d > %d", p->B, kMaxB);
  if (p->H_q % p->H_kv != 0)
    return fail(VQ_ERR_UNSUPPORTED, "H_q=%d is not a multiple of H_kv=%d",
                p->H_q, p->H_kv);
  if (p->H_q / p->H_kv > kMaxGroupHeads)
    return fail(VQ_ERR_UNSUPPORTED, "H_q/H_kv=%d > %d", p->H_q / p->H_kv,
                kMaxGroupHeads);
  if (p->D != 64 && p->D != 128 && p->D != 256)
    return fail(VQ_ERR_UNSUPPORTED, "D=%d (supported: 64, 128, 256)", p->D);
  if (p->bits != 2 && p->bits != 4 && p->bits != 8)
    return fail(VQ_ERR_UNSUPPORTED, "bits=%d (supported: 2, 4, 8)", p->bits);
  if (p->group != 16 && p->group != 32 && p->group != 64 && p->group != 128)
    return fail(VQ_ERR_UNSUPPORTED, "group=%d (supported: 16, 32, 64, 128)",
                p->group);
  if (p->D % p->group != 0)
    return fail(VQ_ERR_UNSUPPORTED, "group=%d does not divide D=%d", p->group,
                p->D);
  if (p->residual > 4096)
    return fail(VQ_ERR_UNSUPPORTED, "residual=%d > 4096", p->residual);
  if (p->max_seq > (1 << 24))
    return fail(VQ_ERR_UNSUPPORTED, "max_seq=%d > 2^24", p->max_seq);
  return VQ_OK;
}

int check_cache(const vq_kivi_cache *c) {
  if (!c) return fail(VQ_ERR_ARG, "cache is NULL");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != c->device)
    return fail(VQ_ERR_ARG, "cache lives on device %d, current device is %d",
                c->device, dev);
  return VQ_OK;
}

// Split unit: a multiple of the key group and of 64 tokens.
int32_t split_unit(int g) { return g > 64 ? g : 64; }

}  // namespace

namespace vqk {
void count_launch(int n) { g_launches.fetch_add((uint64_t)n); }

// vq_kivi_step_host's inputs into the cache's slot: 16-byte chunks of the
// token's K and V (nkv chunks each) and of the query (nq), read through the
// pinned buffers' device mappings before the programmatic wait (the host
// wrote them before the call) and stored after it, when every earlier
// kernel of the stream (the previous step's readers of the slot among
// them) has completed.
__global__ void k_stage_inputs(const uint4 *__restrict__ hk, const uint4 *__restrict__ hv,
                               const uint4 *__restrict__ hq, uint4 *__restrict__ dk,
                               uint4 *__restrict__ dv, uint4 *__restrict__ dq, int nkv,
                               int nq) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a, q = a;
  if (i < nkv) {
    a = hk[i];
    b = hv[i];
  }
  if (i < nq) q = hq[i];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  if (i < nkv) {
    dk[i] = a;
    dv[i] = b;
  }
  if (i < nq) dq[i] = q;
}
void set_last_error(const char *msg) { g_err = msg; }
}  // namespace vqk

extern "C" {

const char *vq_kivi_last_error(void) { return g_err.c_str(); }

uint64_t vq_kivi_launch_count(void) { return g_launches.load(); }

int vq_kivi_quantize(const vq_kivi_params *p, const void *K, const void *V,
                     int64_t s_stride, const int32_t *seq_lens, void *stream,
                     vq_kivi_cache **out) {
  return vq_kivi_quantize_ex(p, nullptr, K, V, s_stride, seq_lens, stream, out);
}

int vq_kivi_quantize_ex(const vq_kivi_params *p, const vq_kivi_options *opt,
                        const void *K, const void *V, int64_t s_stride,
                        const int32_t *seq_lens, void *stream,
                        vq_kivi_cache **out) {
  int rc = check_params(p);
  if (rc) return rc;
  const vq_kivi_options o = opt ? *opt : vq_kivi_options{0, 0, 0, 0, 0, 0, 0, 0};
  if (o.n_sink < 0 || o.n_sink > kMaxSink)
    return fail(VQ_ERR_ARG, "n_sink=%d outside [0, %d]", o.n_sink, kMaxSink);
  if (o.kitty) {
    if (p->bits != 2 || o.n_sink != 0 || (p->D != 64 && p->D != 128))
      return fail(VQ_ERR_UNSUPPORTED, "Kitty needs bits=2, n_sink=0 and D = 64 "
                  "or 128");
    if (o.kitty_hi < 0 || o.kitty_hi > p->D || o.kitty_hi % 16 != 0)
      return fail(VQ_ERR_ARG, "kitty_hi=%d: a multiple of 16 in [0, D=%d]",
                  o.kitty_hi, p->D);
    if (p->max_seq > (1 << 20))
      return fail(VQ_ERR_UNSUPPORTED, "Kitty: max_seq=%d > 2^20", p->max_seq);
  }
  if (o.age_recent > 0) {
    if (p->bits != 8 || o.n_sink != 0 || o.kitty || (p->D != 64 && p->D != 128))
      return fail(VQ_ERR_UNSUPPORTED, "AgeTieredKV needs bits=8 (the row "
                  "capacity), no sinks, no Kitty and D = 64 or 128");
    const int wb[3] = {o.age_bits_recent, o.age_bits_mid, o.age_bits_old};
    for (int i = 0; i < 3; ++i)
      if ((wb[i] != 2 && wb[i] != 4 && wb[i] != 8) || (i && wb[i] > wb[i - 1]))
        return fail(VQ_ERR_ARG, "AgeTieredKV widths %d/%d/%d: each of 2, 4, 8, "
                    "non-increasing", wb[0], wb[1], wb[2]);
    if (o.age_mid <= o.age_recent || o.age_recent % p->group || o.age_mid % p->group)
      return fail(VQ_ERR_ARG, "AgeTieredKV boundaries %d < %d, multiples of g=%d",
                  o.age_recent, o.age_mid, p->group);
  }
  if (!out) return fail(VQ_ERR_ARG, "out is NULL");
  if (!seq_lens) return fail(VQ_ERR_ARG, "seq_lens is NULL");
  int32_t smax = 0;
  for (int b = 0; b < p->B; ++b) {
    if (seq_lens[b] < 0 || seq_lens[b] > p->max_seq)
      return fail(seq_lens[b] < 0 ? VQ_ERR_ARG : VQ_ERR_CAPACITY,
                  "seq_lens[%d]=%d outside [0, max_seq=%d]", b, seq_lens[b],
                  p->max_seq);
    smax = seq_lens[b] > smax ? seq_lens[b] : smax;
  }
  if (smax > 0) {
    if (!K || !V) return fail(VQ_ERR_ARG, "K or V is NULL");
    if (s_stride < smax)
      return fail(VQ_ERR_ARG, "s_stride=%lld < longest sequence %d",
                  (long long)s_stride, smax);
    if (!aligned(K, 16) || !aligned(V, 16))
      return fail(VQ_ERR_ARG, "K and V must be 16-byte aligned");
  }
  cudaStream_t st = (cudaStream_t)stream;

  vq_kivi_cache *c = new (std::nothrow) vq_kivi_cache();
  if (!c) return fail(VQ_ERR_OOM, "host allocation of the cache handle failed");
  c->p = *p;
  c->fail_chunk = -1;
  cudaError_t e = cudaGetDevice(&c->device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount,
                               c->device);
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e, "device query");
  }

  Geometry &geo = c->geo;
  const int g = p->group;
  geo.B = p->B; geo.H_q = p->H_q; geo.H_kv = p->H_kv; geo.D = p->D;
  geo.bits = p->bits; geo.g = g; geo.R = p->residual;
  geo.Tcap = (int)round_up(p->max_seq > 0 ? p->max_seq : 1, g);
  geo.Rcap = p->residual + g;
  geo.row = p->D * p->bits / 8;
  geo.n_sink = o.n_sink;
  geo.kitty = o.kitty ? 1 : 0;
  geo.kitty_hi = o.kitty ? o.kitty_hi : 0;
  if (o.age_recent > 0) {
    geo.age_b1 = o.age_recent;
    geo.age_b2 = o.age_mid;
    geo.age_bits[0] = o.age_bits_recent;
    geo.age_bits[1] = o.age_bits_mid;
    geo.age_bits[2] = o.age_bits_old;
  }
  const bool aged = geo.age_b1 > 0;
  const int32_t unit = split_unit(g);
  const int32_t tps_for_cap = (int32_t)round_up((geo.Tcap + 1023) / 1024, unit);
  c->tps_min = tps_for_cap > 256 ? tps_for_cap : 256;
  geo.max_items = (geo.Tcap + c->tps_min - 1) / c->tps_min + 1;

  const size_t BH = (size_t)p->B * p->H_kv;
  const bool kitty = geo.kitty != 0;
  const size_t krow = (size_t)(p->D + geo.kitty_hi) / 4;
  const size_t sz_codes = BH * geo.Tcap * geo.row;
  const size_t sz_kcodes = kitty ? BH * geo.Tcap * krow : sz_codes;
  const size_t sz_vcodes = kitty ? 0 : sz_codes;
  const size_t sz_kmeta = BH * (geo.Tcap / g) * p->D * sizeof(__half);
  const size_t sz_vmeta = kitty ? 0 : BH * geo.Tcap * (p->D / g) * sizeof(__half);
  const size_t sz_res = BH * geo.Rcap * p->D * sizeof(__half);
  // Kitty: the CUDA-core decode over mixed-width key rows
  c->use_mma = !kitty && !aged && mma_plan(geo, c->sm_count, &c->plan);
  // 2- and 4-bit caches decoded on the tensor cores keep their codes in the
  // order the MMA fragments consume them
  geo.layout = c->use_mma && (p->bits == 2 || p->bits == 4) ? kLayoutFrag : kLayoutPacked;
  size_t n_part = part_floats(geo);
  if (c->use_mma) {
    const size_t n_mma = mma_part_floats(geo, c->plan);
    if (n_mma > n_part) n_part = n_mma;
  }
  const size_t sz_part = n_part * sizeof(float);
  const size_t A = 256;
  size_t off = 0;
  size_t o_Kc = off; off += round_up(sz_kcodes, A);
  size_t o_Vc = off; off += round_up(sz_vcodes, A);
  size_t o_Ks = off; off += round_up(sz_kmeta, A);
  size_t o_Kz = off; off += round_up(sz_kmeta, A);
  size_t o_Vs = off; off += round_up(sz_vmeta, A);
  size_t o_Vz = off; off += round_up(sz_vmeta, A);
  size_t o_Kr = off; off += round_up(sz_res, A);
  size_t o_Vr = off; off += round_up(sz_res, A);
  size_t o_part = off; off += round_up(sz_part, A);
  size_t o_err = off; off += A;
  size_t o_ksmax = off; off += round_up(BH * sizeof(uint32_t), A);
  size_t o_spos = off; off += round_up(BH * o.n_sink * sizeof(int32_t), A);
  size_t o_sk = off; off += round_up(BH * o.n_sink * p->D * sizeof(__half), A);
  size_t o_sv = off; off += round_up(BH * o.n_sink * p->D * sizeof(__half), A);
  size_t o_kmask = off; off += round_up(kitty ? BH * (geo.Tcap / g) * (p->D / 32) * 4 : 0, A);
  size_t o_vf = off; off += round_up(kitty ? BH * geo.Tcap * p->D * sizeof(__half) : 0, A);
  size_t o_ksum = off; off += round_up(kitty ? BH * p->D * 8 : 0, A);
  size_t o_ksq = off; off += round_up(kitty ? BH * p->D * 16 : 0, A);
  size_t o_tier = off; off += round_up(aged ? BH * (geo.Tcap / g) : 0, A);
  c->block_bytes = off;

  e = cudaMallocAsync(&c->block, c->block_bytes, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    delete c;
    return fail(VQ_ERR_OOM, "cudaMallocAsync(%zu bytes): %s", off,
                cudaGetErrorString(e));
  }
  uint8_t *base = (uint8_t *)c->block;
  Planes &pl = c->pl;
  pl.Kc = base + o_Kc;
  pl.Vc = base + o_Vc;
  pl.Ks = (__half *)(base + o_Ks);
  pl.Kz = (__half *)(base + o_Kz);
  pl.Vs = (__half *)(base + o_Vs);
  pl.Vz = (__half *)(base + o_Vz);
  pl.Kr = (__half *)(base + o_Kr);
  pl.Vr = (__half *)(base + o_Vr);
  pl.part = (float *)(base + o_part);
  c->err = (unsigned *)(base + o_err);
  pl.ksmax = (uint32_t *)(base + o_ksmax);
  if (o.n_sink > 0) {
    pl.sink_pos = (int32_t *)(base + o_spos);
    pl.sink_k = (__half *)(base + o_sk);
    pl.sink_v = (__half *)(base + o_sv);
  }
  if (aged) pl.tier = (int8_t *)(base + o_tier);
  if (kitty) {
    pl.kmask = (uint32_t *)(base + o_kmask);
    pl.Vf = (__half *)(base + o_vf);
    pl.ksum = (long long *)(base + o_ksum);
    pl.ksq = (unsigned long long *)(base + o_ksq);
  }
  c->last_stream = st;

  auto abort_create = [&](cudaError_t err, const char *what) {
    cudaFreeAsync(c->block, st);
    cudaStreamSynchronize(st);
    delete c;
    return cuda_fail(err, what);
  };

  // planes start zeroed so that exported padding is deterministic
  e = cudaMemsetAsync(c->block, 0, o_part, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->err, 0, off - o_err, st);
  if (e != cudaSuccess) return abort_create(e, "cudaMemsetAsync");

  FlushTable ft;
  TailTable tt;
  ft.prefix[0] = 0;
  tt.prefix[0] = 0;
  for (int b = 0; b < p->B; ++b) {
    const int32_t S = seq_lens[b];
    const int32_t Tq = n_quantized(S, p->residual, g);
    c->S[b] = S; c->Tq[b] = Tq; c->nres[b] = S - Tq;
    ft.prefix[b + 1] = ft.prefix[b] + Tq / g;
    ft.first_pos[b] = 0;
    ft.src_split[b] = 0;
    tt.prefix[b + 1] = tt.prefix[b] + (S - Tq);
    tt.row0[b] = Tq;
    tt.pos0[b] = Tq;
  }
  if (geo.n_sink > 0) {
    SinkTable sk;
    for (int b = 0; b < p->B; ++b) sk.S[b] = seq_lens[b];
    e = launch_pick_sinks(geo, pl, (const __half *)K, (const __half *)V, s_stride,
                          sk, st);
    if (e != cudaSuccess) return abort_create(e, "sink selection launch");
  }
  if (aged) {
    AgeTable at;
    at.prefix[0] = 0;
    for (int b = 0; b < p->B; ++b) {
      at.gn0[b] = 0;
      at.gn1[b] = c->Tq[b] / g;
      at.gd0[b] = at.gd1[b] = 0;
      at.src_split[b] = 0;
      at.S_old[b] = 0;
      at.S_new[b] = c->S[b];
      at.prefix[b + 1] = at.prefix[b] + at.gn1[b];
    }
    e = launch_age_flush(geo, pl, (const __half *)K, (const __half *)V, s_stride, at, st);
  } else {
    e = kitty ? launch_flush_kitty(geo, pl, (const __half *)K, (const __half *)V,
                                   s_stride, ft, ft.prefix[p->B], st)
              : launch_flush(geo, pl, (const __half *)K, (const __half *)V, s_stride, ft,
                             ft.prefix[p->B], st);
  }
  if (e != cudaSuccess) return abort_create(e, "quantize kernel launch");
  e = launch_tail(geo, pl, (const __half *)K, (const __half *)V, s_stride, tt,
                  tt.prefix[p->B], true, st);
  if (e != cudaSuccess) return abort_create(e, "residual kernel launch");
  c->flush_last = ft.prefix[p->B] > 0 && tt.prefix[p->B] == 0;
  *out = c;
  return VQ_OK;
}

// vq_kivi_append; input_ready: K_new / V_new were written before the call
// (not by the stream's last kernel), so the ring append may load them
// before its programmatic wait
static int append_impl(vq_kivi_cache *c, const void *K_new, const void *V_new,
                       int64_t n_stride, const int32_t *n_new, void *stream,
                       bool input_ready);

int vq_kivi_append(vq_kivi_cache *c, const void *K_new, const void *V_new,
                   int64_t n_stride, const int32_t *n_new, void *stream) {
  return append_impl(c, K_new, V_new, n_stride, n_new, stream, true);
}

static int append_impl(vq_kivi_cache *c, const void *K_new, const void *V_new,
                       int64_t n_stride, const int32_t *n_new, void *stream,
                       bool input_ready) {
  int rc = check_cache(c);
  if (rc) return rc;
  if (!n_new) return fail(VQ_ERR_ARG, "n_new is NULL");
  const vq_kivi_params &p = c->p;
  int32_t nmax = 0;
  for (int b = 0; b < p.B; ++b) {
    if (n_new[b] < 0) return fail(VQ_ERR_ARG, "n_new[%d]=%d < 0", b, n_new[b]);
    if ((int64_t)c->S[b] + n_new[b] > p.max_seq)
      return fail(VQ_ERR_CAPACITY, "sequence %d: %d + %d tokens > max_seq=%d",
                  b, c->S[b], n_new[b], p.max_seq);
    nmax = n_new[b] > nmax ? n_new[b] : nmax;
  }
  if (nmax == 0) return VQ_OK;
  if (!K_new || !V_new) return fail(VQ_ERR_ARG, "K_new or V_new is NULL");
  if (n_stride < nmax)
    return fail(VQ_ERR_ARG, "n_stride=%lld < largest n_new %d",
                (long long)n_stride, nmax);
  if (!aligned(K_new, 16) || !aligned(V_new, 16))
    return fail(VQ_ERR_ARG, "K_new and V_new must be 16-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  const int g = p.group;

  FlushTable ft;
  TailTable tt;
  int32_t Tq_new[kMaxB];
  ft.prefix[0] = 0;
  tt.prefix[0] = 0;
  for (int b = 0; b < p.B; ++b) {
    const int32_t S_old = c->S[b], S_new = S_old + n_new[b];
    Tq_new[b] = n_quantized(S_new, p.residual, g);
    ft.prefix[b + 1] = ft.prefix[b] + (Tq_new[b] - c->Tq[b]) / g;
    ft.first_pos[b] = c->Tq[b];
    ft.src_split[b] = S_old;
    const int32_t keep0 = S_old > Tq_new[b] ? S_old : Tq_new[b];
    tt.prefix[b + 1] = tt.prefix[b] + (S_new - keep0);
    tt.row0[b] = keep0 - S_old;
    tt.pos0[b] = keep0;
  }
  cudaError_t e;
  if (c->geo.age_b1 > 0) {
    // AgeTieredKV: new groups, and the stored groups whose age crossed a
    // boundary: for boundary x the groups G with S_old - (G+1) g < x <=
    // S_new - (G+1) g, i.e. floor((S_old - x)/g) <= G < floor((S_new - x)/g)
    auto floordiv = [](int64_t a, int64_t d) { return a >= 0 ? a / d : -((-a + d - 1) / d); };
    AgeTable at;
    at.prefix[0] = 0;
    for (int b = 0; b < p.B; ++b) {
      const int32_t S_old = c->S[b], S_new = S_old + n_new[b];
      at.gn0[b] = c->Tq[b] / g;
      at.gn1[b] = Tq_new[b] / g;
      int64_t lo = INT32_MAX, hi = 0;
      for (int x : {c->geo.age_b1, c->geo.age_b2}) {
        const int64_t l = floordiv(S_old - x, g), u = floordiv(S_new - x, g);
        if (u > l) { lo = l < lo ? l : lo; hi = u > hi ? u : hi; }
      }
      if (lo < 0) lo = 0;
      if (hi > c->Tq[b] / g) hi = c->Tq[b] / g;
      if (hi < lo) hi = lo;
      at.gd0[b] = (int32_t)(hi > lo ? lo : 0);
      at.gd1[b] = (int32_t)(hi > lo ? hi : 0);
      at.src_split[b] = S_old;
      at.S_old[b] = S_old;
      at.S_new[b] = S_new;
      at.prefix[b + 1] = at.prefix[b] + (at.gn1[b] - at.gn0[b]) + (at.gd1[b] - at.gd0[b]);
    }
    e = launch_age_flush(c->geo, c->pl, (const __half *)K_new, (const __half *)V_new,
                         n_stride, at, st);
  } else {
    e = c->geo.kitty
        ? launch_flush_kitty(c->geo, c->pl, (const __half *)K_new, (const __half *)V_new,
                             n_stride, ft, ft.prefix[p.B], st)
        : launch_flush(c->geo, c->pl, (const __half *)K_new,
                       (const __half *)V_new, n_stride, ft,
                       ft.prefix[p.B], st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "flush kernel launch");
  e = launch_tail(c->geo, c->pl, (const __half *)K_new, (const __half *)V_new,
                  n_stride, tt, tt.prefix[p.B], input_ready, st);
  if (e != cudaSuccess) return cuda_fail(e, "residual kernel launch");
  if (tt.prefix[p.B] > 0)
    c->flush_last = false;
  else if (ft.prefix[p.B] > 0)
    c->flush_last = true;
  for (int b = 0; b < p.B; ++b) {
    c->S[b] += n_new[b];
    c->Tq[b] = Tq_new[b];
    c->nres[b] = c->S[b] - Tq_new[b];
  }
  c->last_stream = st;
  return VQ_OK;
}

int vq_kivi_decode_attend(vq_kivi_cache *c, const void *q, float *out,
                          float softmax_scale, void *stream) {
  int rc = check_cache(c);
  if (rc) return rc;
  if (!q || !out) return fail(VQ_ERR_ARG, "q or out is NULL");
  if (!aligned(q, 16) || !aligned(out, 16))
    return fail(VQ_ERR_ARG, "q and out must be 16-byte aligned");
  if (!std::isfinite(softmax_scale))
    return fail(VQ_ERR_ARG, "softmax_scale is not finite");
  const vq_kivi_params &p = c->p;
  cudaStream_t st = (cudaStream_t)stream;

  const float scale = softmax_scale > 0.f ? softmax_scale
                                          : 1.0f / std::sqrt((float)p.D);
  if (c->use_mma) {
    MmaTable tab;
    tab.bprefix[0] = 0;
    for (int b = 0; b < p.B; ++b) {
      tab.Tq[b] = c->Tq[b];
      tab.nres[b] = c->nres[b];
      tab.nq[b] = (c->Tq[b] + c->plan.chunk - 1) / c->plan.chunk;
      tab.nc[b] = tab.nq[b];
      tab.bprefix[b + 1] = tab.bprefix[b] + p.H_kv * tab.nc[b];
    }
    MmaArgs args;
    args.q = (const __half *)q;
    args.out = out;
    args.part = c->pl.part;
    args.err = c->err;
    args.scale_log2 = scale * 1.4426950408889634f;
    args.N = tab.bprefix[p.B];
    args.fail_chunk = c->fail_chunk;
    c->fail_chunk = -1;
    args.early = c->flush_last ? 0 : 1;
    MmaPlan plan = c->plan;
    if (c->split_tokens > 0) {
      // a fixed partition: about split_tokens quantized tokens per warp
      const int64_t w = ((int64_t)args.N * plan.chunk + c->split_tokens - 1) /
                        c->split_tokens;
      if (w < plan.warps_max) plan.warps_max = (int)(w > 0 ? w : 1);
    }
    cudaError_t e = launch_decode_mma(c->geo, c->pl, plan, args, tab, st);
    c->flush_last = false;
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
    c->last_stream = st;
    return VQ_OK;
  }

  int64_t total_tq = 0;
  for (int b = 0; b < p.B; ++b) total_tq += c->Tq[b];
  int32_t tps = c->split_tokens;
  const int32_t unit = split_unit(p.group);
  const bool one_wave = c->geo.age_b1 > 0 || c->geo.kitty;
  if (tps == 0 && one_wave) {
    // AgeTieredKV and Kitty: one wave of CTAs, each streaming its groups through
    // per-warp pipelines (a CTA's start costs a pipeline fill, so items are
    // long); a sequence's last item also takes its residual window.  Among
    // the splits whose items fit one wave, take the one whose busiest SM
    // (ceil(items / SMs) items of tps tokens; the launcher caps the CTAs per
    // SM at that count) finishes first by the cost below.
    if (c->age_tps > 0 && !memcmp(c->age_Tq, c->Tq, sizeof(int32_t) * p.B)) {
      tps = c->age_tps;
    } else {
      const int64_t sms = c->sm_count;
      const int64_t cap = (int64_t)(c->geo.kitty ? kitty_decode_ctas_per_sm(c->geo)
                                                 : age_decode_ctas_per_sm(c->geo)) * sms;
      auto items = [&](int64_t t) {
        int64_t n = 0;
        for (int b = 0; b < p.B; ++b) {
          const int64_t nq = (c->Tq[b] + t - 1) / t;
          n += nq > 0 ? nq : (c->nres[b] > 0 ? 1 : 0);
        }
        return n * p.H_kv;
      };
      int32_t tq_max = 1;
      for (int b = 0; b < p.B; ++b) tq_max = c->Tq[b] > tq_max ? c->Tq[b] : tq_max;
      const int64_t t_top = (int64_t)round_up((size_t)tq_max, unit);
      int64_t t = (total_tq * p.H_kv + cap - 1) / (cap > 0 ? cap : 1);
      t = (int64_t)round_up((size_t)(t > 1 ? t : 1), unit);
      // more (sequence, head) pairs than CTA slots: one item each
      while (items(t) > cap && t < t_top) t += unit;
      // the busiest SM holds k = ceil(items / SMs) CTAs of t tokens (plus a
      // pipeline fill each); an SM's throughput grows with its CTAs (their
      // warps hide one another's latency: per-CTA timestamps of the
      // AgeTieredKV decode, two CTAs on an SM 1.7 times one alone), taken
      // here as k^0.75, so the cost is k^0.25 (t + 64)
      int64_t best = t;
      double best_cost = -1.0;
      for (int i = 0; i < 64; ++i, t += unit) {
        const int64_t n = items(t);
        const double k = (double)((n + sms - 1) / sms);
        const double cost = std::pow(k, 0.25) * (double)(t + 64);
        if (best_cost < 0 || cost < best_cost) { best = t; best_cost = cost; }
        if (n <= p.H_kv) break;   // one item per sequence and head
      }
      tps = (int32_t)best;
      c->age_tps = tps;
      memcpy(c->age_Tq, c->Tq, sizeof(int32_t) * p.B);
    }
  } else if (tps == 0) {
    const int64_t target_items = 4LL * c->sm_count;
    int64_t t = (total_tq * p.H_kv + target_items - 1) / target_items;
    tps = (int32_t)round_up((size_t)(t > 1 ? t : 1), unit);
  }
  if (tps < c->tps_min) tps = c->tps_min;

  DecodeTable tab;
  tab.prefix[0] = 0;
  for (int b = 0; b < p.B; ++b) {
    tab.Tq[b] = c->Tq[b];
    tab.nres[b] = c->nres[b];
    tab.nq[b] = (c->Tq[b] + tps - 1) / tps;
    if (one_wave) {
      // the last quantized item takes the residual window (an item of its
      // own when there is no quantized token)
      if (tab.nq[b] == 0 && c->nres[b] > 0) tab.nq[b] = 1;
      tab.prefix[b + 1] = tab.prefix[b] + tab.nq[b];
    } else {
      tab.prefix[b + 1] = tab.prefix[b] + tab.nq[b] + (c->nres[b] > 0 ? 1 : 0);
    }
  }
  DecodeArgs args;
  args.q = (const __half *)q;
  args.out = out;
  args.scale_log2 = scale * 1.4426950408889634f;
  args.tps = tps;
  args.total_items = tab.prefix[p.B];
  args.err = c->err;
  cudaError_t e = launch_decode(c->geo, c->pl, args, tab, st);
  if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
  c->last_stream = st;
  return VQ_OK;
}

namespace {
// the device address of pinned host memory, or nullptr when `p` is not
// pinned host memory
void *pinned_device_ptr(const void *p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}
}  // namespace

int vq_kivi_step_host(vq_kivi_cache *c, const void *h_k_new, const void *h_v_new,
                      const void *h_q, float *h_out, float softmax_scale,
                      void *stream) {
  int rc = check_cache(c);
  if (rc) return rc;
  if (!h_k_new || !h_v_new || !h_q || !h_out)
    return fail(VQ_ERR_ARG, "step_host: NULL argument");
  const void *d_k = pinned_device_ptr(h_k_new), *d_v = pinned_device_ptr(h_v_new),
             *d_q = pinned_device_ptr(h_q);
  if (!d_k || !d_v || !d_q)
    return fail(VQ_ERR_ARG, "step_host: the inputs must be pinned host memory");
  float *d_out = static_cast<float *>(pinned_device_ptr(h_out));
  if (!d_out) return fail(VQ_ERR_ARG, "step_host: h_out must be pinned host memory");
  if (!aligned(d_k, 16) || !aligned(d_v, 16) || !aligned(d_q, 16))
    return fail(VQ_ERR_ARG, "step_host: the inputs must be 16-byte aligned");
  const vq_kivi_params &p = c->p;
  const size_t kv_bytes = (size_t)p.B * p.H_kv * p.D * sizeof(__half);
  const size_t q_bytes = (size_t)p.B * p.H_q * p.D * sizeof(__half);
  cudaError_t e;
  if (!c->io) {
    StepIO *io = new (std::nothrow) StepIO();
    if (!io) return fail(VQ_ERR_OOM, "step_host: host allocation failed");
    io->off_v = round_up(kv_bytes, 256);
    io->off_q = io->off_v + round_up(kv_bytes, 256);
    io->ones.assign(p.B, 1);
    e = cudaMalloc(&io->slot, io->off_q + q_bytes);
    if (e != cudaSuccess) {
      io->slot = nullptr;
      free_step_io(io);
      return cuda_fail(e, "step_host: slot allocation");
    }
    c->io = io;
  }
  StepIO *io = c->io;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t *slot = static_cast<uint8_t *>(io->slot);
  // A step that flushes no group (and no AgeTieredKV tier) only copies the
  // token's rows into the residual ring: the ring append reads them, and
  // the decode kernels q, through the pinned buffers' device mappings (the
  // host wrote them before this call, so the loads may precede the kernels'
  // programmatic waits), and no staging kernel runs.
  bool flushes = c->geo.age_b1 > 0;
  for (int b = 0; b < p.B && !flushes; ++b)
    flushes = n_quantized(c->S[b] + 1, p.residual, p.group) > c->Tq[b];
  if (!flushes) {
    rc = append_impl(c, d_k, d_v, 1, io->ones.data(), stream, true);
    if (rc == VQ_OK) rc = vq_kivi_decode_attend(c, d_q, d_out, softmax_scale, stream);
    return rc;
  }
  // Otherwise the inputs go into the slot first: a programmatic dependent
  // of the stream's last kernel (the previous step's merge), then the
  // append (the flush and the ring copy read the slot after their waits)
  // and the decode.
  const int nkv = (int)(kv_bytes / 16), nq = (int)(q_bytes / 16);
  const int n = nkv > nq ? nkv : nq;
  e = launch_pdl(k_stage_inputs, dim3((n + 255) / 256), dim3(256), 0, st,
                 static_cast<const uint4 *>(d_k), static_cast<const uint4 *>(d_v),
                 static_cast<const uint4 *>(d_q), reinterpret_cast<uint4 *>(slot),
                 reinterpret_cast<uint4 *>(slot + io->off_v),
                 reinterpret_cast<uint4 *>(slot + io->off_q), nkv, nq);
  count_launch();
  if (e != cudaSuccess) return cuda_fail(e, "step_host: input staging launch");
  rc = append_impl(c, slot, slot + io->off_v, 1, io->ones.data(), stream, false);
  if (rc == VQ_OK) rc = vq_kivi_decode_attend(c, slot + io->off_q, d_out, softmax_scale, stream);
  return rc;
}

int vq_kivi_attend_multi(vq_kivi_cache *c, const void *q, int32_t S_q,
                         float *out, float softmax_scale, void *stream) {
  int rc = check_cache(c);
  if (rc) return rc;
  if (!q || !out) return fail(VQ_ERR_ARG, "q or out is NULL");
  if (!aligned(q, 16) || !aligned(out, 16))
    return fail(VQ_ERR_ARG, "q and out must be 16-byte aligned");
  if (!std::isfinite(softmax_scale))
    return fail(VQ_ERR_ARG, "softmax_scale is not finite");
  const vq_kivi_params &p = c->p;
  if (S_q < 1) return fail(VQ_ERR_ARG, "S_q=%d < 1", S_q);
  for (int b = 0; b < p.B; ++b)
    if (c->S[b] < S_q)
      return fail(VQ_ERR_ARG, "sequence %d holds %d tokens, fewer than S_q=%d",
                  b, c->S[b], S_q);
  const int GQ = p.H_q / p.H_kv;
  if (c->geo.kitty || c->geo.age_b1 > 0)
    return fail(VQ_ERR_UNSUPPORTED, "multi-query attend: not for Kitty or "
                "AgeTieredKV caches");
  if (p.D != 64 && p.D != 128)
    return fail(VQ_ERR_UNSUPPORTED, "multi-query attend: D=%d (supported: 64, 128)", p.D);
  if (GQ != 1 && GQ != 2 && GQ != 4 && GQ != 8)
    return fail(VQ_ERR_UNSUPPORTED, "multi-query attend: H_q/H_kv=%d (supported: "
                "1, 2, 4, 8)", GQ);
  if ((int64_t)S_q * p.D * 2 * p.H_q * p.B > ((int64_t)1 << 40))
    return fail(VQ_ERR_UNSUPPORTED, "multi-query attend: q too large");
  const float scale = softmax_scale > 0.f ? softmax_scale
                                          : 1.0f / std::sqrt((float)p.D);
  MultiTable tab;
  for (int b = 0; b < p.B; ++b) {
    tab.S[b] = c->S[b];
    tab.Tq[b] = c->Tq[b];
  }
  MultiArgs args;
  args.q = (const __half *)q;
  args.out = out;
  args.err = c->err;
  args.scale_log2 = scale * 1.4426950408889634f;
  args.S_q = S_q;
  args.GQ = GQ;
  cudaStream_t st = (cudaStream_t)stream;
  // key-range splits: the partials of all but the first range and every
  // range's (max, sum) rows live in the cache's scratch
  args.splits = multi_splits(c->geo, args, tab, c->sm_count, c->split_tokens);
  if (args.splits > 1) {
    const size_t rows = (size_t)p.B * p.H_q * S_q;
    const size_t o_bytes = round_up((size_t)(args.splits - 1) * rows * p.D * sizeof(float), 256);
    const size_t need = o_bytes + (size_t)args.splits * rows * sizeof(float2);
    if (need > c->mq_scratch_bytes) {
      if (c->mq_scratch) cudaFree(c->mq_scratch);   // waits for its last users
      c->mq_scratch = nullptr;
      c->mq_scratch_bytes = 0;
      cudaError_t ea = cudaMalloc(&c->mq_scratch, need);
      if (ea != cudaSuccess) {
        cudaGetLastError();
        c->mq_scratch = nullptr;
        return fail(VQ_ERR_OOM, "multi-query attend: scratch of %zu bytes", need);
      }
      c->mq_scratch_bytes = need;
    }
    args.part_o = static_cast<float *>(c->mq_scratch);
    args.part_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(c->mq_scratch) + o_bytes);
  }
  cudaError_t e = launch_attend_multi(c->geo, c->pl, args, tab, st);
  if (e == cudaErrorNotSupported)
    return fail(VQ_ERR_UNSUPPORTED, "multi-query attend: the driver offers no "
                "tensor-map encoder");
  if (e != cudaSuccess) return cuda_fail(e, "multi-query attend launch");
  c->flush_last = false;
  c->last_stream = st;
  return VQ_OK;
}

int vq_kivi_free(vq_kivi_cache *c) {
  if (!c) return VQ_OK;
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != c->device) cudaSetDevice(c->device);
  free_step_io(c->io);
  c->io = nullptr;
  if (c->mq_scratch) cudaFree(c->mq_scratch);
  c->mq_scratch = nullptr;
  cudaError_t e = cudaFreeAsync(c->block, c->last_stream);
  cudaError_t e2 = cudaStreamSynchronize(c->last_stream);
  if (dev != c->device && dev >= 0) cudaSetDevice(dev);
  delete c;
  if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync");
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaStreamSynchronize");
  return VQ_OK;
}

int vq_kivi_lengths(const vq_kivi_cache *c, int32_t *S, int32_t *T_q,
                    int32_t *n_res) {
  if (!c) return fail(VQ_ERR_ARG, "cache is NULL");
  const size_t n = sizeof(int32_t) * c->p.B;
  if (S) memcpy(S, c->S, n);
  if (T_q) memcpy(T_q, c->Tq, n);
  if (n_res) memcpy(n_res, c->nres, n);
  return VQ_OK;
}

int vq_kivi_get_params(const vq_kivi_cache *c, vq_kivi_params *p) {
  if (!c || !p) return fail(VQ_ERR_ARG, "NULL argument");
  *p = c->p;
  return VQ_OK;
}

size_t vq_kivi_plane_bytes(const vq_kivi_cache *c, int which) {
  if (!c) return 0;
  const Geometry &geo = c->geo;
  const size_t BH = (size_t)geo.B * geo.H_kv;
  const bool kitty = geo.kitty != 0;
  switch (which) {
    case 0: return BH * geo.Tcap * (kitty ? (size_t)(geo.D + geo.kitty_hi) / 4 : geo.row);
    case 3: return kitty ? 0 : BH * geo.Tcap * geo.row;
    case 1: case 2: return BH * (geo.Tcap / geo.g) * geo.D * sizeof(__half);
    case 4: case 5: return kitty ? 0 : BH * geo.Tcap * (geo.D / geo.g) * sizeof(__half);
    case 11: return kitty ? BH * (geo.Tcap / geo.g) * (geo.D / 32) * 4 : 0;
    case 12: return kitty ? BH * geo.Tcap * geo.D * sizeof(__half) : 0;
    case 13: return geo.age_b1 > 0 ? BH * (geo.Tcap / geo.g) : 0;
    case 6: case 7: return BH * geo.Rcap * geo.D * sizeof(__half);
    case 8: return BH * geo.n_sink * sizeof(int32_t);
    case 9: case 10: return BH * geo.n_sink * geo.D * sizeof(__half);
    default: return 0;
  }
}

int vq_kivi_export(const vq_kivi_cache *c, int which, void *dst,
                   size_t dst_bytes, void *stream) {
  int rc = check_cache(c);
  if (rc) return rc;
  const size_t need = vq_kivi_plane_bytes(c, which);
  // an empty plane (no sinks, no Kitty, or a Kitty cache's value codes)
  if (need == 0 && which >= 0 && which <= 13 && which != 1 && which != 2 &&
      which != 6 && which != 7)
    return VQ_OK;
  if (need == 0) return fail(VQ_ERR_ARG, "which=%d is not a plane", which);
  if (!dst) return fail(VQ_ERR_ARG, "dst is NULL");
  if (dst_bytes < need)
    return fail(VQ_ERR_ARG, "dst holds %zu bytes, plane needs %zu", dst_bytes,
                need);
  cudaStream_t st = (cudaStream_t)stream;
  const void *src = nullptr;
  switch (which) {
    case 0: src = c->pl.Kc; break;
    case 1: src = c->pl.Ks; break;
    case 2: src = c->pl.Kz; break;
    case 3: src = c->pl.Vc; break;
    case 4: src = c->pl.Vs; break;
    case 5: src = c->pl.Vz; break;
    case 8: src = c->pl.sink_pos; break;
    case 9: src = c->pl.sink_k; break;
    case 10: src = c->pl.sink_v; break;
    case 11: src = c->pl.kmask; break;
    case 12: src = c->pl.Vf; break;
    case 13: src = c->pl.tier; break;
    default: break;
  }
  cudaError_t e;
  if ((which == 0 || which == 3) && c->geo.age_b1 > 0) {
    e = launch_age_export(c->geo, c->pl, which == 3, dst, c->Tq, st);
  } else if ((which == 0 || which == 3) && c->geo.layout == kLayoutFrag && !c->geo.kitty) {
    e = launch_export_frag(c->geo, (const uint8_t *)src, which == 3, dst, st);
  } else if (src) {
    e = cudaMemcpyAsync(dst, src, need, cudaMemcpyDeviceToDevice, st);
  } else {
    e = launch_export_residual(c->geo, c->pl, which, dst, c->Tq, c->nres, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "export");
  return VQ_OK;
}

int vq_kivi_dequantize(const vq_kivi_cache *c, void *K_hat, void *V_hat,
                       int64_t s_stride, void *stream) {
  int rc = check_cache(c);
  if (rc) return rc;
  if (c->geo.kitty || c->geo.age_b1 > 0)
    return fail(VQ_ERR_UNSUPPORTED, "dequantize: not for Kitty or AgeTieredKV caches");
  if (!K_hat || !V_hat) return fail(VQ_ERR_ARG, "K_hat or V_hat is NULL");
  if (((uintptr_t)K_hat | (uintptr_t)V_hat) & 15u)
    return fail(VQ_ERR_ARG, "K_hat and V_hat must be 16-byte aligned");
  int32_t smax = 0;
  for (int b = 0; b < c->p.B; ++b)
    if (c->S[b] > smax) smax = c->S[b];
  if (s_stride < smax)
    return fail(VQ_ERR_ARG, "s_stride=%lld < longest sequence %d",
                (long long)s_stride, smax);
  cudaError_t e = launch_dequantize(c->geo, c->pl, c->Tq, c->nres,
                                    (__half *)K_hat, (__half *)V_hat, s_stride,
                                    (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "dequantize");
  return VQ_OK;
}

int vq_kivi_cache_bytes(const vq_kivi_cache *c, vq_kivi_bytes *out) {
  if (!c || !out) return fail(VQ_ERR_ARG, "NULL argument");
  const vq_kivi_params &p = c->p;
  const uint64_t row = (uint64_t)c->geo.row;
  vq_kivi_bytes r = {0, 0, 0, 0, 0, 0};
  const bool kitty = c->geo.kitty != 0;
  for (int b = 0; b < p.B; ++b) {
    const uint64_t Tq = (uint64_t)c->Tq[b], H = (uint64_t)p.H_kv;
    if (kitty) {
      // mixed-width key rows, key scale/zero and the 4-bit channel masks,
      // fp16 values
      r.code_bytes += H * Tq * (uint64_t)((p.D + c->geo.kitty_hi) / 4);
      r.meta_bytes += H * ((Tq / p.group) * p.D * 4 + (Tq / p.group) * (p.D / 8));
      r.value_fp16_bytes += H * Tq * p.D * 2;
      r.residual_bytes += H * (uint64_t)c->nres[b] * p.D * 4;
      r.fp16_bytes += H * (uint64_t)c->S[b] * p.D * 4;
      continue;
    }
    if (c->geo.age_b1 > 0) {
      // codes at each group's tier width (a row's capacity is D bytes)
      for (int G = 0; G < (int)(Tq / p.group); ++G)
        r.code_bytes += 2 * H * (uint64_t)p.group * p.D *
                        c->geo.age_bits[age_tier(c->geo, c->S[b], G)] / 8;
    } else {
      r.code_bytes += 2 * H * Tq * row;
    }
    r.meta_bytes += H * ((Tq / p.group) * p.D * 4 + Tq * (p.D / p.group) * 4);
    r.residual_bytes += H * (uint64_t)c->nres[b] * p.D * 4;
    r.fp16_bytes += H * (uint64_t)c->S[b] * p.D * 4;
  }
  r.sink_bytes = 0;
  if (c->geo.n_sink > 0) {
    // sinks of the quantized region (their positions live on the device)
    const size_t n = (size_t)p.B * p.H_kv * c->geo.n_sink;
    int32_t *pos = new (std::nothrow) int32_t[n];
    if (!pos) return fail(VQ_ERR_OOM, "host allocation failed");
    cudaError_t e = cudaMemcpyAsync(pos, c->pl.sink_pos, n * sizeof(int32_t),
                                    cudaMemcpyDeviceToHost, c->last_stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->last_stream);
    if (e != cudaSuccess) {
      delete[] pos;
      return cuda_fail(e, "reading the sink positions");
    }
    for (size_t i = 0; i < n; ++i) {
      const int b = (int)(i / ((size_t)p.H_kv * c->geo.n_sink));
      if (pos[i] >= 0 && pos[i] < c->Tq[b]) r.sink_bytes += (uint64_t)p.D * 4;
    }
    delete[] pos;
  }
  *out = r;
  return VQ_OK;
}

int vq_kivi_device_status(vq_kivi_cache *c) {
  int rc = check_cache(c);
  if (rc) return rc;
  unsigned flag = 0;
  cudaError_t e = cudaMemcpyAsync(&flag, c->err, sizeof flag,
                                  cudaMemcpyDeviceToHost, c->last_stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->last_stream);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status");
  if (flag) {
    cudaMemsetAsync(c->err, 0, sizeof flag, c->last_stream);
    return fail(VQ_ERR_CUDA, "a decode kernel gave up waiting for its "
                "shared-memory copies; its outputs are not valid");
  }
  return VQ_OK;
}

int vq_kivi_debug_fail_chunk(vq_kivi_cache *c, int32_t chunk) {
  if (!c) return fail(VQ_ERR_ARG, "cache is NULL");
  c->fail_chunk = chunk < 0 ? -1 : chunk;
  return VQ_OK;
}

int vq_kivi_decode_kernel(const vq_kivi_cache *c) {
  if (!c) return fail(VQ_ERR_ARG, "cache is NULL");
  return c->use_mma ? 1 : 0;
}

int vq_kivi_set_split_tokens(vq_kivi_cache *c, int32_t tokens_per_split) {
  if (!c) return fail(VQ_ERR_ARG, "cache is NULL");
  if (tokens_per_split != 0) {
    const int32_t unit = split_unit(c->p.group);
    if (tokens_per_split < 64 || tokens_per_split % unit != 0)
      return fail(VQ_ERR_ARG, "tokens_per_split=%d must be a positive "
                  "multiple of %d", tokens_per_split, unit);
    if (tokens_per_split < c->tps_min)
      return fail(VQ_ERR_ARG, "tokens_per_split=%d below the workspace "
                  "minimum %d for this capacity", tokens_per_split, c->tps_min);
  }
  c->split_tokens = tokens_per_split;
  return VQ_OK;
}

}  // extern "C"
