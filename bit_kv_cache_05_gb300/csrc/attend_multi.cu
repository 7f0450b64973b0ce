// Several query tokens per sequence over the quantized cache, on the
// Blackwell tensor cores: tcgen05.mma with its accumulators in tensor memory
// (TMEM), the query tile brought in by a TMA tensor copy.
//
// Method: attention over the group-affine cache of VeloxQuant-MLX changelog
// v0.42.0 "Added" (k_hat / v_hat rebuilt from codes and per-group (scale,
// zero), never written to global memory), for S_q query tokens at once --
// speculative multi-token decode, or a chunked prefill whose tokens were
// just appended -- with a causal mask: query i of sequence b is the cache's
// token S_b - S_q + i and sees the tokens up to its own position.  The pages
// ship a matrix-tiled prefill / cross-attention companion for large S_q
// (changelog v0.40.0 "Added"); that is prior art for the shape of the work,
// not for this kernel.
//
// One CTA of 128 threads serves 128 rows of one (sequence, kv head); the
// rows are (query head of the kv head, query) pairs, row r = hh * QPT + i
// with QPT = 128 / GQ queries per tile, and thread r owns row r.  Key tiles
// of 64 tokens stream through; a tile's codes, scales and zeros arrive in a
// shared-memory stage by bulk copies (cp.async.bulk, one mbarrier), issued
// for the next tile as soon as this tile's rebuild has read the stage, so
// that they land while the products and the softmax run:
//   1. the threads rebuild the tile: k_hat and v_hat of every token in fp32
//      (code * scale + zero; residual-window rows are fp16 already), each
//      split into fp16 hi = RN(x) and lo = RN(x - hi), stored in shared
//      memory in the tensor cores' 128-byte-swizzled K-major layout: k_hat
//      as [token][channel], v_hat transposed as [channel][token];
//   2. one thread issues S = Q k_hat^T as Q K_hi^T + Q K_lo^T into TMEM
//      (M = 128, N = 64, K = D; q is fp16, hence exact as an operand);
//   3. each thread loads its row of S from TMEM, masks it causally and
//      updates an online softmax in fp32 (base 2), writing p as fp16 hi + lo,
//      the A operand of the next product;
//   4. one thread issues O += P v_hat as P_hi V_hi + P_hi V_lo + P_lo V_hi
//      into the TMEM accumulator O (N = D).
// The running maximum of a row is raised lazily: O is rescaled in TMEM only
// when a row's maximum grows by more than 8 (base 2), so p <= 2^8 stays in
// fp16 range; the final O / l does not depend on which maximum was used.
// Every wait on an mbarrier is bounded; a wait that gives up sets the
// cache's error word (read by vq_kivi_device_status) and the CTA returns
// after freeing its tensor memory.
#include <cuda.h>   // CUtensorMap and its enums; the encoder is looked up at run time

#include <cmath>
#include <mutex>

#include "bulk_pipe.cuh"
#include "vqk_internal.cuh"

namespace vqk {
namespace multi {

constexpr int kRows = 128;     // M: rows per CTA (one per thread)
constexpr int kTok = 64;       // tokens per key tile
constexpr int kThreads = 128;
constexpr uint32_t kTmemCols = 256;   // S in columns [0, 64), O in [128, 128 + D)
constexpr uint32_t kOCol = 128;
constexpr float kLazy = 8.f;   // rescale O when a row maximum grows by more

__device__ __forceinline__ uint32_t saddr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(bar)));
}

__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(saddr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// bounded wait (~0.5 s); false when it gives up
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  while (!mbar_try(bar, parity))
    if (now_ns() - t0 > 500000000ull) return false;
  return true;
}

// ---- tcgen05 ---------------------------------------------------------------

// Shared-memory matrix descriptor of a 128-byte-swizzled K-major tile whose
// 8-row swizzle atoms (1024 B, 1024-byte aligned) follow one another: start
// address >> 4 (bits 0-13), leading-dimension offset 16 B (unused by this
// layout), stride between 8-row groups 1024 B (bits 32-45), descriptor
// version 1 (bits 46-47), swizzle mode 128 B (value 2 in bits 61-63).
// Moving 16 fp16 along K inside the atom adds 32 B to the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A
// and B fp16 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3
// in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t f16_idesc(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b,
                                     uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          saddr(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (the warp reads
// its 32 lanes); the load is complete when this returns
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
        "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]),
      "f"(v[7]), "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]),
      "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]),
      "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]),
      "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// hi = RN(x), lo = RN(x - hi) as two packed fp16 pairs
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}

// ---- shared-memory plan ------------------------------------------------------

// P (128 rows x 64 tokens, hi and lo) is written only after the S product
// that read K_hat has completed, and K_hat of the next tile only after the O
// product that read P has completed, so at D = 128 P takes K_hat's place
// (16 KB each for hi and lo); the CTA then needs 96 KB and two fit on an SM
// (their tensor memory, 256 columns each, fills the SM's 512).
// The stage (the tile's quantized rows as stored, bulk-copied) follows:
// key codes and value codes (64 rows each), the key scale and zero rows of
// the tile's groups (up to 4, at g = 16), the value scale and zero rows of
// its tokens.
template <int D, int BITS>
struct Smem {
  static constexpr int KB = D / 64;                       // 64-channel K-blocks
  static constexpr int ROW = D * BITS / 8;                // code bytes per token
  static constexpr uint32_t Q = 0;                        // [KB][128 rows][128 B]
  static constexpr uint32_t KH = Q + KB * 16384;          // [KB][64 rows][128 B]
  static constexpr uint32_t KL = KH + KB * 8192;
  static constexpr uint32_t VH = KL + KB * 8192;          // [D rows][128 B]
  static constexpr uint32_t VL = VH + D * 128;
  static constexpr bool ALIAS = KB * 8192 >= 16384;
  static constexpr uint32_t PH = ALIAS ? KH : VL + D * 128;   // [128 rows][128 B]
  static constexpr uint32_t PL = ALIAS ? KL : PH + 16384;
  static constexpr uint32_t BAR = ALIAS ? VL + D * 128 : PL + 16384;  // 4 mbarriers + TMEM slot
  static constexpr uint32_t SKC = BAR + 64;               // stage
  static constexpr uint32_t SVC = SKC + 64 * ROW;
  // value codes per 16-token block, 16 bytes of padding between blocks (a
  // warp's reads of different blocks then fall in different banks)
  static constexpr uint32_t VBS = 16 * ROW + 16;
  static constexpr uint32_t SKS = SVC + 4 * VBS;
  static constexpr uint32_t SKZ = SKS + 8 * D;
  static constexpr uint32_t SVS = SKZ + 8 * D;
  static constexpr uint32_t SVZ = SVS + 8 * D;
  static constexpr uint32_t BYTES = SVZ + 8 * D;
  static constexpr uint32_t ALLOC = BYTES + 1024;         // room to align the base
};

// byte offset of the 16-byte chunk `chunk` of row `row` in a 128-byte-row
// swizzled tile
__device__ __forceinline__ uint32_t sw_off(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// ---- codes of the cache, per bit width and code order ----------------------
//
// FRAG: the MMA-fragment order of 2- and 4-bit caches decoded on the tensor
// cores (a 32-bit word holds two 16-bit halves of 16/b fields; keys: channel
// c = 16 ks + 4 tig + e of a token row in word NW tig + ks/KPW, half e mod
// 2, field 2 (ks mod KPW) + e/2; values: the tokens of a 16-token block pair
// up as (tl, tl + 4), and channel c = 16 mv + 2 j + rho of pair pi sits in
// word (8 pi + j) NW + mv/KPW, field 2 (mv mod KPW) + rho, the first token
// in the low half).  Otherwise the packed order: code of channel c of a
// token row at byte c b / 8, bit (c b) mod 8.
template <int D, int BITS, bool FRAG>
struct Codes {
  static constexpr uint32_t M = (1u << BITS) - 1u;
  static constexpr int ROW = D * BITS / 8;

  // the 16 codes of channels 16 ks ... 16 ks + 15 of a key row (a row of
  // the shared-memory stage)
  static __device__ __forceinline__ void key16(const uint8_t *krow, int ks,
                                               uint32_t (&c)[16]) {
    if constexpr (FRAG) {
      constexpr int KPW = 8 / BITS, NW = D * BITS / 128;
      const uint32_t *w = reinterpret_cast<const uint32_t *>(krow);
      const int r0 = 2 * (ks % KPW);
#pragma unroll
      for (int tig = 0; tig < 4; ++tig) {
        const uint32_t x = w[NW * tig + ks / KPW];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          c[4 * tig + e] = (x >> (16 * (e & 1) + BITS * (r0 + (e >> 1)))) & M;
      }
    } else {
      // 16 codes = 2 BITS bytes at byte 2 BITS ks
      uint32_t w[BITS / 2];
      if constexpr (BITS == 2) {
        w[0] = *reinterpret_cast<const uint32_t *>(krow + 4 * ks);
      } else if constexpr (BITS == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(krow + 8 * ks);
        w[0] = v.x; w[1] = v.y;
      } else {
        const uint4 v = *reinterpret_cast<const uint4 *>(krow + 16 * ks);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
      }
      constexpr int PER = 32 / BITS;
#pragma unroll
      for (int e = 0; e < 16; ++e) c[e] = (w[e / PER] >> (BITS * (e % PER))) & M;
    }
  }

  // codes of channels c0 ... c0+7 (c0 a multiple of 8) of the 8 tokens
  // tb ... tb+7 (tb = 0 or 8) of the 16-token value block vblk: c[u][e] for
  // token tb + u, channel c0 + e
  static __device__ __forceinline__ void value8x8(const uint8_t *vblk, int tb, int c0,
                                                  uint32_t (&c)[8][8]) {
    if constexpr (FRAG) {
      constexpr int KPW = 8 / BITS, NW = D * BITS / 128;
      const uint32_t *w = reinterpret_cast<const uint32_t *>(vblk);
      const int mv = c0 >> 4, j0 = (c0 & 15) >> 1, r0 = 2 * (mv % KPW);
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const int pi = (tb >> 1) + pp;          // pairs (tb + pp, tb + pp + 4)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const uint32_t x = w[(8 * pi + j0 + jj) * NW + mv / KPW];
#pragma unroll
          for (int rho = 0; rho < 2; ++rho) {
            c[pp][2 * jj + rho] = (x >> (BITS * (r0 + rho))) & M;
            c[pp + 4][2 * jj + rho] = (x >> (16 + BITS * (r0 + rho))) & M;
          }
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint8_t *p = vblk + (size_t)(tb + u) * ROW + c0 * BITS / 8;
        uint32_t w0, w1 = 0;
        if constexpr (BITS == 2) {
          w0 = *reinterpret_cast<const uint16_t *>(p);
        } else if constexpr (BITS == 4) {
          w0 = *reinterpret_cast<const uint32_t *>(p);
        } else {
          const uint2 v = *reinterpret_cast<const uint2 *>(p);
          w0 = v.x; w1 = v.y;
        }
        constexpr int PER = 32 / BITS;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          c[u][e] = ((e < PER ? w0 : w1) >> (BITS * (e % PER))) & M;
      }
    }
  }
};

template <int D, int BITS, bool FRAG>
__global__ void __launch_bounds__(kThreads, 2)
k_attend_multi(const __grid_constant__ CUtensorMap qmap, Geometry geo,
               Planes pl, MultiArgs args, MultiTable tab) {
  using SM = Smem<D, BITS>;
  using CD = Codes<D, BITS, FRAG>;
  constexpr int KB = SM::KB, KS = D / 16, C8 = D / 8, ROW = CD::ROW;
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte aligned (the swizzle atoms); pointer arithmetic on the shared
  // array, so that accesses through it compile as shared-memory ones
  unsigned char *sm = smem_raw + ((1024u - (saddr(smem_raw) & 1023u)) & 1023u);
  uint64_t *bar_q = reinterpret_cast<uint64_t *>(sm + SM::BAR);
  uint64_t *bar_s = bar_q + 1, *bar_o = bar_q + 2, *bar_k = bar_q + 3;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bar_q + 4);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int b = blockIdx.z, h = blockIdx.y;
  const int GQ = args.GQ, QPT = kRows / GQ, S_q = args.S_q;
  const int S = tab.S[b], Tq = tab.Tq[b];
  const int g = geo.g, NJ = D / g;
  const size_t hd = (size_t)b * geo.H_kv + h;
  const int splits = args.splits;
  const int sp = blockIdx.x % splits;              // this CTA's key range
  const int i0 = (blockIdx.x / splits) * QPT;
  const int hh = tid / QPT, qi = i0 + tid % QPT;
  const bool valid = qi < S_q;
  const int pos = valid ? S - S_q + qi : -1;       // this row's own token
  const int last_i = min(S_q - 1, i0 + QPT - 1);
  const int max_pos = S - S_q + last_i;            // furthest token any row sees
  // key tiles [kt_lo, kt_hi) of the nkt the rows see: tokens t_lo ... t_hi - 1
  const int nkt = max_pos / kTok + 1;
  const int t_lo = (int)((int64_t)nkt * sp / splits) * kTok;
  const int t_hi = min((int)((int64_t)nkt * (sp + 1) / splits) * kTok, max_pos + 1);
  const uint8_t *kc_base = pl.Kc + hd * geo.Tcap * ROW;
  const uint8_t *vc_base = pl.Vc + hd * geo.Tcap * ROW;
  const __half *ks_base = pl.Ks + hd * (geo.Tcap / g) * D;
  const __half *kz_base = pl.Kz + hd * (geo.Tcap / g) * D;
  const __half *vs_base = pl.Vs + hd * geo.Tcap * NJ;
  const __half *vz_base = pl.Vz + hd * geo.Tcap * NJ;
  const __half *kr_base = pl.Kr + hd * geo.Rcap * D;
  const __half *vr_base = pl.Vr + hd * geo.Rcap * D;

  if (tid == 0) {
    mbar_init(bar_q);
    mbar_init(bar_s);
    mbar_init(bar_o);
    mbar_init(bar_k);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     saddr(tslot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t t_lane = tmem + ((uint32_t)(32 * warp) << 16);   // this warp's lanes

  // the query tile: KB boxes of 64 channels x QPT queries x GQ heads
  if (tid == 0) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar_q)),
                 "r"((uint32_t)(KB * 16384))
                 : "memory");
    for (int kb = 0; kb < KB; ++kb)
      asm volatile(
          "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
          "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(saddr(sm + SM::Q + kb * 16384)),
          "l"(reinterpret_cast<uint64_t>(&qmap)), "r"(64 * kb), "r"(i0), "r"(h * GQ), "r"(b),
          "r"(saddr(bar_q))
          : "memory");
  }
  // the quantized rows of the tile at ta (ta < Tq) into the stage
  auto stage_tile = [&](int ta) {
    const int nq = min(kTok, Tq - ta);        // a multiple of 16 (g >= 16)
    const int G0 = ta / g, ng = (ta + nq - 1) / g - G0 + 1;
    mbar_expect_tx(bar_k, 2u * (nq * ROW + ng * D * 2 + nq * NJ * 2));
    bulk_g2s(sm + SM::SKC, kc_base + (size_t)ta * ROW, nq * ROW, bar_k);
    for (int k = 0; k < nq / 16; ++k)
      bulk_g2s(sm + SM::SVC + k * SM::VBS, vc_base + (size_t)(ta + 16 * k) * ROW, 16 * ROW,
               bar_k);
    bulk_g2s(sm + SM::SKS, ks_base + (size_t)G0 * D, ng * D * 2, bar_k);
    bulk_g2s(sm + SM::SKZ, kz_base + (size_t)G0 * D, ng * D * 2, bar_k);
    bulk_g2s(sm + SM::SVS, vs_base + (size_t)ta * NJ, nq * NJ * 2, bar_k);
    bulk_g2s(sm + SM::SVZ, vz_base + (size_t)ta * NJ, nq * NJ * 2, bar_k);
  };
  uint32_t ph_k = 0;
  bool k_pending = false;       // a stage copy is in flight
  if (tid == 0 && t_lo < Tq && t_lo < t_hi) stage_tile(t_lo);
  k_pending = t_lo < Tq && t_lo < t_hi;
  // KIVI-Sink: the sinks of the quantized region (the rest are -1); their
  // k_hat / v_hat are their fp16 rows
  __shared__ int ssk[kMaxSink];
  const int nsk = geo.n_sink;
  if (tid < nsk) {
    const int p = pl.sink_pos[hd * nsk + tid];
    ssk[tid] = p < Tq ? p : -1;
  }
  bool failed = __syncthreads_or(!mbar_wait(bar_q, 0));
  auto sink_slot = [&](int t) {
    int slot = -1;
    for (int j = 0; j < nsk; ++j)
      if (ssk[j] == t) slot = j;
    return slot;
  };

  const float sl2 = args.scale_log2;
  // rows without a query see no token; a finite maximum keeps their
  // weights at exactly 0 (2^-inf) instead of NaN
  float m_run = valid ? -INFINITY : 0.f, l_run = 0.f;
  uint32_t ph_s = 0, ph_o = 0;
  bool o_started = false;       // an O product has been issued
  bool o_pending = false;       // the last O product is not yet waited for
  const uint32_t idesc_s = f16_idesc(kRows, kTok), idesc_o = f16_idesc(kRows, D);
  const uint32_t sbase = saddr(sm);

  for (int t0 = t_lo; t0 < t_hi && !failed; t0 += kTok) {
    // (a) the previous O product read P and V_hat: wait before rewriting them
    if (o_pending) {
      const bool ok = mbar_wait(bar_o, ph_o);
      ph_o ^= 1u;
      o_pending = false;
      if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    // the tile's quantized rows in the stage
    if (t0 < Tq) {
      const bool ok = mbar_wait(bar_k, ph_k);
      ph_k ^= 1u;
      k_pending = false;
      if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    const int G0t = t0 / g;
    // sinks in this tile: bit (t - t0)
    uint64_t tmask = 0;
    for (int j = 0; j < nsk; ++j) {
      const int d = ssk[j] - t0;
      if (ssk[j] >= 0 && d >= 0 && d < kTok) tmask |= 1ull << d;
    }
    // (b1) k_hat of tokens t0 ... t0+63, 16 channels per item, as fp16 hi + lo;
    // consecutive threads take a token's consecutive 16-channel steps, so a
    // warp reads few stage rows (and writes whole swizzled rows)
    for (int it = tid; it < kTok * KS; it += kThreads) {
      const int tl = it / KS, ks = it % KS;
      const int t = t0 + tl;
      float kf[16];
      if (t < Tq) {
        uint32_t c[16];
        CD::key16(sm + SM::SKC + tl * ROW, ks, c);
        const int gr = t / g - G0t;
        const __half *sp = reinterpret_cast<const __half *>(sm + SM::SKS) + gr * D + 16 * ks;
        const __half *zp = reinterpret_cast<const __half *>(sm + SM::SKZ) + gr * D + 16 * ks;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint4 sr = reinterpret_cast<const uint4 *>(sp)[q];
          const uint4 zr = reinterpret_cast<const uint4 *>(zp)[q];
          const __half2 *s2 = reinterpret_cast<const __half2 *>(&sr);
          const __half2 *z2 = reinterpret_cast<const __half2 *>(&zr);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 sf = __half22float2(s2[e]), zf = __half22float2(z2[e]);
            const float2 r = __ffma2_rn(make_float2((float)c[8 * q + 2 * e],
                                                    (float)c[8 * q + 2 * e + 1]), sf, zf);
            kf[8 * q + 2 * e] = r.x;
            kf[8 * q + 2 * e + 1] = r.y;
          }
        }
      } else if (t < S) {
        const uint4 *rp = reinterpret_cast<const uint4 *>(
            kr_base + (size_t)(t % geo.Rcap) * D + 16 * ks);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint4 r = __ldg(rp + q);
          const __half2 *r2 = reinterpret_cast<const __half2 *>(&r);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(r2[e]);
            kf[8 * q + 2 * e] = f.x;
            kf[8 * q + 2 * e + 1] = f.y;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) kf[e] = 0.f;
      }
      if ((tmask >> tl) & 1ull) {
        const uint4 *rp = reinterpret_cast<const uint4 *>(
            pl.sink_k + (hd * nsk + sink_slot(t)) * D + 16 * ks);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint4 r = __ldg(rp + q);
          const __half2 *r2 = reinterpret_cast<const __half2 *>(&r);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(r2[e]);
            kf[8 * q + 2 * e] = f.x;
            kf[8 * q + 2 * e + 1] = f.y;
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          split2(kf[8 * q + 2 * e], kf[8 * q + 2 * e + 1], hw[e], lw[e]);
        const int c0 = 16 * ks + 8 * q;
        const uint32_t ko = (c0 >> 6) * 8192 + sw_off(tl, (c0 & 63) >> 3);
        *reinterpret_cast<uint4 *>(sm + SM::KH + ko) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4 *>(sm + SM::KL + ko) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    }
    // (b2) v_hat transposed, 8 channels x 8 tokens per item: V^T rows are
    // channels, a 16-byte chunk holds 8 consecutive tokens
    for (int it = tid; it < C8 * (kTok / 8); it += kThreads) {
      const int t8 = it % (kTok / 8), c0 = 8 * (it / (kTok / 8));
      const int ta = t0 + 8 * t8;                 // first token of the octet
      float vf[8][8];
      if (ta < Tq) {
        // Tq is a multiple of g >= 16: the octet is wholly quantized
        uint32_t c[8][8];
        CD::value8x8(sm + SM::SVC + (((ta & ~15) - t0) >> 4) * SM::VBS, ta & 8, c0, c);
        const int j = c0 / g;
        const __half *svs = reinterpret_cast<const __half *>(sm + SM::SVS);
        const __half *svz = reinterpret_cast<const __half *>(sm + SM::SVZ);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float sv = __half2float(svs[(ta + u - t0) * NJ + j]);
          const float zv = __half2float(svz[(ta + u - t0) * NJ + j]);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float2 r = __ffma2_rn(make_float2((float)c[u][e], (float)c[u][e + 1]),
                                        make_float2(sv, sv), make_float2(zv, zv));
            vf[u][e] = r.x;
            vf[u][e + 1] = r.y;
          }
        }
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int t = ta + u;
          if (t < S) {
            const uint4 r = __ldg(reinterpret_cast<const uint4 *>(
                vr_base + (size_t)(t % geo.Rcap) * D + c0));
            const __half2 *r2 = reinterpret_cast<const __half2 *>(&r);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __half22float2(r2[e]);
              vf[u][2 * e] = f.x;
              vf[u][2 * e + 1] = f.y;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) vf[u][e] = 0.f;
          }
        }
      }
      if ((tmask >> (8 * t8)) & 0xffull) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (!((tmask >> (8 * t8 + u)) & 1ull)) continue;
          const uint4 r = __ldg(reinterpret_cast<const uint4 *>(
              pl.sink_v + (hd * nsk + sink_slot(ta + u)) * D + c0));
          const __half2 *r2 = reinterpret_cast<const __half2 *>(&r);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(r2[e]);
            vf[u][2 * e] = f.x;
            vf[u][2 * e + 1] = f.y;
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) split2(vf[2 * u][e], vf[2 * u + 1][e], hw[u], lw[u]);
        const uint32_t vo = sw_off(c0 + e, t8);
        *reinterpret_cast<uint4 *>(sm + SM::VH + vo) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4 *>(sm + SM::VL + vo) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();

    // every thread's reads of the stage are done: the next tile's copies
    const int tn = t0 + kTok;
    if (tn < t_hi && tn < Tq) {
      if (tid == 0) stage_tile(tn);
      k_pending = true;
    }

    // (c) S = Q K_hi^T + Q K_lo^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint32_t kbase = sbase + (part ? SM::KL : SM::KH);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma(tmem, sw128_desc(sbase + SM::Q + kb * 16384 + 32 * k),
                 sw128_desc(kbase + kb * 8192 + 32 * k), idesc_s,
                 (part | kb | k) != 0);
      }
      umma_commit(bar_s);
    }
    {
      const bool ok = mbar_wait(bar_s, ph_s);
      ph_s ^= 1u;
      if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    tc_fence_after();

    // (d) this row's scores: causal mask, online softmax, p as fp16 hi + lo
    float sc[kTok];
    {
      float tmp[32];
      tmem_ld32(t_lane, tmp);
#pragma unroll
      for (int j = 0; j < 32; ++j) sc[j] = tmp[j];
      tmem_ld32(t_lane + 32, tmp);
#pragma unroll
      for (int j = 0; j < 32; ++j) sc[32 + j] = tmp[j];
    }
    // the row maximum of the raw scores, then scaled (sl2 > 0: the same
    // value as the maximum of the scaled scores); the weights below scale
    // each score inside one packed fma
    float mt = -INFINITY;
    if (t0 + kTok - 1 <= pos) {          // the whole tile is visible to this row
#pragma unroll
      for (int j = 0; j < kTok; ++j) mt = fmaxf(mt, sc[j]);
    } else {
#pragma unroll
      for (int j = 0; j < kTok; ++j) {
        sc[j] = (t0 + j <= pos) ? sc[j] : -INFINITY;
        mt = fmaxf(mt, sc[j]);
      }
    }
    mt *= sl2;
    float alpha = 1.f;
    const bool raise = mt > m_run + kLazy;   // false while both are -inf
    if (raise) {
      alpha = ex2(m_run - mt);               // 2^-inf = 0 on the first raise
      m_run = mt;
    }
    if (o_started && __any_sync(0xffffffffu, raise)) {
      // rescale this warp's rows of O in TMEM (rows that did not raise
      // their maximum multiply by 1)
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        float o[32];
        tmem_ld32(t_lane + kOCol + c, o);
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] *= alpha;
        tmem_st32(t_lane + kOCol + c, o);
      }
      tmem_wait_st();
    }
    float2 psum2 = make_float2(0.f, 0.f);
    // a row that has seen no token of its key range yet keeps m_run = -inf:
    // subtract 0 there, so that its -inf scores give 0
    const float msub = m_run == -INFINITY ? 0.f : m_run;
#pragma unroll
    for (int j8 = 0; j8 < kTok / 8; ++j8) {
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        // p = 2^(s sl2 - m) for two scores: one packed fma
        const float2 x = __ffma2_rn(make_float2(sc[8 * j8 + 2 * e], sc[8 * j8 + 2 * e + 1]),
                                    make_float2(sl2, sl2), make_float2(-msub, -msub));
        const float pa = ex2(x.x);
        const float pc = ex2(x.y);
        psum2 = __fadd2_rn(psum2, make_float2(pa, pc));
        split2(pa, pc, hw[e], lw[e]);
      }
      const uint32_t po = sw_off(tid, j8);
      *reinterpret_cast<uint4 *>(sm + SM::PH + po) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4 *>(sm + SM::PL + po) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
    l_run = fmaf(l_run, alpha, psum2.x + psum2.y);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();

    // (e) O += P_hi V_hi + P_hi V_lo + P_lo V_hi
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int part = 0; part < 3; ++part) {
        const uint32_t pb = sbase + (part == 2 ? SM::PL : SM::PH);
        const uint32_t vb = sbase + (part == 1 ? SM::VL : SM::VH);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma(tmem + kOCol, sw128_desc(pb + 32 * k), sw128_desc(vb + 32 * k), idesc_o,
               (o_started || part || k) ? 1u : 0u);
      }
      umma_commit(bar_o);
    }
    o_started = true;
    o_pending = true;
  }

  if (!failed && o_pending) {
    const bool ok = mbar_wait(bar_o, ph_o);
    ph_o ^= 1u;
    o_pending = false;
    failed = __syncthreads_or(!ok);
  }
  // this row's result: normalised into out, or with several key ranges
  // unnormalised into this range's rows and its (max, sum) beside them
  const size_t row = ((size_t)b * geo.H_q + (size_t)h * GQ + hh) * S_q + (valid ? qi : 0);
  const size_t rows = (size_t)geo.B * geo.H_q * S_q;
  if (!failed && valid && splits > 1) args.part_ml[sp * rows + row] = make_float2(m_run, l_run);
  if (!failed && o_started) {
    tc_fence_after();
    const float inv = splits > 1 ? 1.f : (l_run > 0.f ? 1.f / l_run : 0.f);
    float *orow = (sp == 0 ? args.out : args.part_o + (sp - 1) * rows * D) + row * D;
#pragma unroll
    for (int c = 0; c < D; c += 32) {
      float o[32];
      tmem_ld32(t_lane + kOCol + c, o);
      if (valid) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          __stcs(reinterpret_cast<float4 *>(orow + c + j),
                 make_float4(o[j] * inv, o[j + 1] * inv, o[j + 2] * inv, o[j + 3] * inv));
      }
    }
  } else if (!failed && valid && splits > 1) {
    // a key range without any product (none of its tiles issued one)
    float *orow = (sp == 0 ? args.out : args.part_o + (sp - 1) * rows * D) + row * D;
    for (int c = 0; c < D; c += 4)
      __stcs(reinterpret_cast<float4 *>(orow + c), make_float4(0.f, 0.f, 0.f, 0.f));
  }
  if (failed) {
    if (tid == 0) atomicOr(args.err, 2u);
    // let an O product still in flight finish (bounded) before the tensor
    // memory is released, and a stage copy land before the CTA ends
    if (o_pending) mbar_wait(bar_o, ph_o);
    if (k_pending) mbar_wait(bar_k, ph_k);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols));
  }
}

// Merge of the key ranges of a split multi-query attend: one warp per row
// (sequence, query head, query), lanes over channels; the ranges' rows are
// weighted by 2^(m_k - M) with M their largest maximum and divided by the
// weighted sum of their sums.
template <int D>
__global__ void __launch_bounds__(256)
k_attend_combine(MultiArgs args, int64_t rows) {
  constexpr int CPL = D / 32;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const int splits = args.splits;
  float M = -INFINITY;
  for (int k = 0; k < splits; ++k) M = fmaxf(M, args.part_ml[k * rows + row].x);
  float L = 0.f, o[CPL];
#pragma unroll
  for (int u = 0; u < CPL; ++u) o[u] = 0.f;
  for (int k = 0; k < splits; ++k) {
    const float2 ml = args.part_ml[k * rows + row];
    const float f = ml.x == -INFINITY ? 0.f : ex2(ml.x - M);
    L = fmaf(f, ml.y, L);
    const float *src = (k == 0 ? args.out : args.part_o + (k - 1) * rows * D) + row * D +
                       lane * CPL;
    float v[CPL];
    if constexpr (CPL == 4) {
      const float4 x = __ldcs(reinterpret_cast<const float4 *>(src));
      v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else {
      const float2 x = __ldcs(reinterpret_cast<const float2 *>(src));
      v[0] = x.x; v[1] = x.y;
    }
#pragma unroll
    for (int u = 0; u < CPL; ++u) o[u] = fmaf(f, v[u], o[u]);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float *dst = args.out + row * D + lane * CPL;
  if constexpr (CPL == 4)
    *reinterpret_cast<float4 *>(dst) = make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
  else
    *reinterpret_cast<float2 *>(dst) = make_float2(o[0] * inv, o[1] * inv);
}

// ---- host ------------------------------------------------------------------

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
  static std::once_flag once;
  static EncodeTiled fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

template <int D, int BITS, bool FRAG>
cudaError_t launch_k(const Geometry &geo, const Planes &pl, const MultiArgs &args,
                     const MultiTable &tab, cudaStream_t st) {
  EncodeTiled enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  // q [B][H_q][S_q][D] fp16 as a 4-D tensor (channel, query, head, sequence);
  // one box = 64 channels x QPT queries x GQ heads of one sequence, 128-byte
  // swizzled (the tensor cores' K-major layout)
  const int QPT = kRows / args.GQ;
  CUtensorMap map;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)args.S_q, (cuuint64_t)geo.H_q,
                              (cuuint64_t)geo.B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)args.S_q * D * 2,
                                 (cuuint64_t)geo.H_q * args.S_q * D * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)QPT, (cuuint32_t)args.GQ, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<__half *>(args.q),
                   dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const size_t smem = Smem<D, BITS>::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(k_attend_multi<D, BITS, FRAG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((args.S_q + QPT - 1) / QPT * args.splits, geo.H_kv, geo.B);
  k_attend_multi<D, BITS, FRAG><<<grid, kThreads, smem, st>>>(map, geo, pl, args, tab);
  count_launch();
  e = cudaGetLastError();
  if (e != cudaSuccess || args.splits == 1) return e;
  const int64_t rows = (int64_t)geo.B * geo.H_q * args.S_q;
  k_attend_combine<D><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(args, rows);
  count_launch();
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const Geometry &geo, const Planes &pl, const MultiArgs &args,
                     const MultiTable &tab, cudaStream_t st) {
  const bool frag = geo.layout == kLayoutFrag;
  switch (geo.bits) {
    case 2: return frag ? launch_k<D, 2, true>(geo, pl, args, tab, st)
                        : launch_k<D, 2, false>(geo, pl, args, tab, st);
    case 4: return frag ? launch_k<D, 4, true>(geo, pl, args, tab, st)
                        : launch_k<D, 4, false>(geo, pl, args, tab, st);
    case 8: return launch_k<D, 8, false>(geo, pl, args, tab, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace multi

int multi_splits(const Geometry &geo, const MultiArgs &args, const MultiTable &tab,
                 int sm_count, int split_tokens) {
  const int QPT = multi::kRows / args.GQ;
  const int64_t tiles = (args.S_q + QPT - 1) / QPT;
  int S_max = 0;
  for (int b = 0; b < geo.B; ++b) S_max = tab.S[b] > S_max ? tab.S[b] : S_max;
  const int nkt = (S_max + multi::kTok - 1) / multi::kTok;
  if (split_tokens > 0) {
    int s = (S_max + split_tokens - 1) / split_tokens;
    if (s > 8) s = 8;
    if (s > nkt) s = nkt;
    return s < 1 ? 1 : s;
  }
  // about 16 waves of CTAs (two per SM): the tiles' CTAs differ in length,
  // and finer ones fill the last waves (measured on 1024 CTAs of 520 key
  // tiles: 1, 2, 4, 5 ranges: 10.49, 10.18, 9.78, 9.61 ms; 6 and 8 no
  // faster); at most 8 ranges, each at least 8 key tiles
  const int64_t ctas = tiles * geo.H_kv * geo.B, slots = 2 * (int64_t)sm_count;
  int64_t s = (16 * slots + ctas - 1) / ctas;
  if (s > 8) s = 8;
  while (s > 1 && nkt / s < 8) --s;
  return s < 1 ? 1 : (int)s;
}

cudaError_t launch_attend_multi(const Geometry &geo, const Planes &pl,
                                const MultiArgs &args, const MultiTable &tab,
                                cudaStream_t st) {
  switch (geo.D) {
    case 64: return multi::launch_d<64>(geo, pl, args, tab, st);
    case 128: return multi::launch_d<128>(geo, pl, args, tab, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace vqk
