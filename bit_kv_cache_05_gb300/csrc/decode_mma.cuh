// Fused decode step over the quantized cache on the tensor cores (mma.sync
// m16n8k16, fp16 operands, fp32 accumulation): the kernel template.  One
// instantiation per (D, bits, padded query heads per kv head, group size);
// decode_mma_b{2,4,8}.cu instantiate it, decode_mma.cu plans and launches.
//
// Method: VeloxQuant-MLX changelog v0.42.0 "Added", scalar_fused_decode_attend:
// SDP attention directly over the group-affine cache; k_hat / v_hat are
// never written to memory; online softmax accumulated in fp32.
//
// Algebra (base-2 scores, q' = q * softmax_scale * log2(e)):
//   key group G:    q'.k_hat_t = sum_c (q'_c s_Gc) code_tc + sum_c q'_c z_Gc
//   value token t:  o_c += p_t (s_t,j(c) code_tc + z_t,j(c))
// The code sums run on the tensor cores:
//   scores   S^T[tok][col]  = codes[tok][ch] . A[ch][col],  A = q' s  (hi + lo)
//   values   O^T[ch][col]  += codes^T[ch][tok] . W[tok][col], W = p s  (hi + lo)
// The codes enter as exact fp16 subnormals (the b-bit field masked out of the
// packed word, value = code * 2^(bit position - 24)); each factor enters as
// two fp16 operands hi and lo in adjacent columns, so products keep about 21
// bits: p s as hi = its top 11 bits and lo = the fp32 remainder rounded to
// fp16; q' s (2- and 4-bit caches) in fp16 pair arithmetic from a per-head
// fp16 split of q' (hi = RN(qh s), lo = RN(ql s + the exact error of hi)).
// The zero-point sums (sum_c q'_c z_Gc and sum_t p_t z_t,j) run on the CUDA
// cores in fp32.
//
// MMA columns.  Scores: 8 columns = 4 (query head, key group) pairs x (hi,
// lo): with GQP query heads per kv head, a "window" of 4/GQP consecutive key
// groups shares one B operand (for one head: four groups, so the operand is
// rebuilt once per 4g tokens).  Values: 8 columns = 4 (query head, value
// group) pairs x (hi, lo); an m16 channel tile uses the block that holds its
// value group.
//
// Work split: the (sequence, kv head, 64-token chunk) space of the quantized
// tokens is cut into W equal contiguous ranges, one per warp of a persistent
// grid.  A warp streams its chunks through its own cp.async.bulk pipeline
// (one mbarrier per stage, bounded waits), keeps (m, l, O) for the head it
// is in, and writes one partial per head segment.  k_merge_mma, launched
// behind the decode kernel, adds each head's fp16 residual window and merges
// the head's partials with a log-sum-exp.
#pragma once

#include <type_traits>

#include "bulk_pipe.cuh"
#include "vqk_internal.cuh"

namespace vqk {
namespace mma {

constexpr int kC = 64;          // tokens per chunk (4 m16 tiles)
// One warp per CTA: everything a warp computes about its chunks (cursor,
// stage and plane addresses, branch conditions) then derives from blockIdx
// and the kernel arguments alone, so the compiler keeps it in uniform
// registers and branches on it without divergence handling, and the bulk
// copies take their addresses from uniform registers directly.
constexpr int kNW = 1;          // warps per CTA
constexpr int kMaxStages = 4;
// a partial (o[D], m, l) per (warp segment, query head), padded to D + 4
// floats so that the o rows stay 16-byte aligned
template <int D> __host__ __device__ constexpr int part_stride() { return D + 4; }
constexpr unsigned kFull = 0xffffffffu;

// ---- PTX helpers (the bulk-copy pipeline ones are in bulk_pipe.cuh) ------

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0,
                                         uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^x for x <= 0 (softmax weights): the hardware approximation, flushing
// results below 2^-126 to zero.
__device__ __forceinline__ float exp2_neg(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// fp32 factors enter the MMAs as two fp16 operands in adjacent columns:
// "hi" keeps x's sign, exponent and top 10 mantissa bits (exact in fp16
// while |x| is in fp16's normal range), "lo" the exact fp32 remainder
// x - hi, rounded to fp16, so hi + lo carries ~21 bits of x.  A lane builds
// only its own column, with one and-xor and one fma per value:
//   hv = (x & 0xFFFFE000) ^ flip,  y = x * d + hv
// (hi lanes: flip = 0, d = 0 -> y = hi;  lo lanes: flip = sign bit, d = 1
// -> y = x - hi, exact).
struct HiLo {
  uint32_t flip;
  float d;
};

__device__ __forceinline__ float2 hilo2(float2 x, const HiLo &s) {
  const float2 hv = make_float2(
      __uint_as_float((__float_as_uint(x.x) & 0xFFFFE000u) ^ s.flip),
      __uint_as_float((__float_as_uint(x.y) & 0xFFFFE000u) ^ s.flip));
  return __ffma2_rn(x, make_float2(s.d, s.d), hv);
}

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// 2^e as a float, e in [-126, 127]
__device__ __forceinline__ float exp2i(int e) {
  return __int_as_float((127 + e) << 23);
}

// NJ consecutive fp16 values (NJ a power of two, naturally aligned) -> fp32
template <int NJ>
__device__ __forceinline__ void load_halves(const __half *p, float (&out)[NJ]) {
  if constexpr (NJ == 1) {
    out[0] = __half2float(p[0]);
  } else if constexpr (NJ == 2) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(p));
    out[0] = f.x; out[1] = f.y;
  } else {
#pragma unroll
    for (int q = 0; q < NJ / 4; ++q) {
      const uint2 r = reinterpret_cast<const uint2 *>(p)[q];
      const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
      out[4 * q] = a.x; out[4 * q + 1] = a.y;
      out[4 * q + 2] = b.x; out[4 * q + 3] = b.y;
    }
  }
}

// ---- per-bit-width code layout --------------------------------------------
//
// Score A fragment (rows = 16 tokens, K = 16 channels of K-step ks): lane
// (gid, tig) holds K slots 2tig, 2tig+1 (register "lo") and 2tig+8, 2tig+9
// ("hi") of tokens gid and gid+8; those four slots are channels 4tig ...
// 4tig+3 of the K-step, slot e (0..3) being channel 4tig + off(e).  The code
// of channel c arrives scaled by 2^(oexp(c) - 24); the score B operand
// carries 2^-oexp(c) (folded into a copy of q'), so every product carries
// exactly 2^-24.  8-bit codes use the packed order (a uint4 of a token row
// holds WPQ K-steps, bytes permuted into place); 2- and 4-bit codes use the
// fragment order, where masks alone place the codes.
//
// Value A fragment (rows = channels 2gid, 2gid+1 of an m16 tile, K = tokens
// of the K-step): in the packed order lane (gid, tig) permutes the bytes of
// two tokens' words (vsel) and masks channel 2gid (vmask0) and 2gid+1
// (vmask1), whose codes arrive scaled by 2^(vpos0 - 24) and 2^(vpos1 - 24);
// a uint4 of a token row covers VTPQ m16 tiles, tile u of it uses word
// vword(x, u, gid).  In the fragment order (2- and 4-bit codes) the two
// tokens of a register share a word and masks alone place them.  The output
// rows are scaled back at the end.
template <int BITS> struct Layout;

// Codes in kLayoutFrag order (2- and 4-bit): a 32-bit word holds two
// halves of 16/B fields, field r at bits B*r of each half.  Fields whose
// bits lie within 0..9 of the half (r < DIRECT) are masked in place
// (exponent B*r); the rest are masked after one shift of the word by SHIFT
// (exponent B*r - SHIFT): a field at bit p of a half is the fp16 subnormal
// code * 2^(p - 24).  A word covers KPW = 8/B K-steps (keys) or m16 tiles
// (values).  Score slot e of channel c (K-step ks = c/16, lane group
// (c/4) mod 4, e = c mod 4) is field 2 (ks mod KPW) + e/2 of half e mod 2.
template <int B, int DIRECT_, int SHIFT_>
struct FragLayout {
  static constexpr bool FRAG = true;
  static constexpr int KPW = 8 / B, DIRECT = DIRECT_, SHIFT = SHIFT_;
  static constexpr uint32_t M = ((1u << B) - 1u) * 0x00010001u;
  static __host__ __device__ constexpr int fexp(int r) {
    return r < DIRECT ? B * r : B * r - SHIFT;
  }
  static __device__ __forceinline__ uint32_t field(uint32_t w, uint32_t ws, int r) {
    return r < DIRECT ? (w & (M << (B * r))) : (ws & (M << (B * r - SHIFT)));
  }
  static __host__ __device__ constexpr int off(int e) { return e; }
  static __device__ __forceinline__ int oexp(int c) {
    return fexp(2 * ((c >> 4) % KPW) + ((c & 3) >> 1));
  }
  static __device__ __forceinline__ uint32_t score_sel(int) { return 0u; }
  static __device__ __forceinline__ uint32_t vsel(int) { return 0u; }
  static __device__ __forceinline__ int vpos0(int) { return 0; }
  static __device__ __forceinline__ int vpos1(int) { return 0; }
};

template <> struct Layout<2> : FragLayout<2, 5, 6> {};
template <> struct Layout<4> : FragLayout<4, 2, 8> {};

template <> struct Layout<8> {
  static constexpr int WPQ = 1;    // uint4 = one K-step (4 words, one per tig)
  static constexpr int VTPQ = 1;
  // channels 4tig..4tig+3 are the bytes of word 4ks + tig (sel carries tig)
  static __device__ __forceinline__ uint32_t score_sel(int tig) { return tig; }
  static __device__ __forceinline__ void score_a(const uint4 &q, int,
                                                 uint32_t tig, uint32_t &lo,
                                                 uint32_t &hi) {
    const uint32_t w = (tig & 2) ? ((tig & 1) ? q.w : q.z) : ((tig & 1) ? q.y : q.x);
    lo = w & 0x00FF00FFu;          // channels 4tig, 4tig+2
    hi = (w >> 8) & 0x00FF00FFu;   // channels 4tig+1, 4tig+3
  }
  static __host__ __device__ constexpr int off(int e) { return (e & 1) * 2 + (e >> 1); }
  static __host__ __device__ constexpr int sexp(int) { return 0; }
  static constexpr bool FRAG = false;
  static __device__ __forceinline__ int oexp(int) { return 0; }
  static __device__ __forceinline__ uint32_t vword(const uint4 &x, int, int gid) {
    // word gid/2: bit 1 of gid picks the odd word, bit 2 the upper pair
    return (gid & 4) ? ((gid & 2) ? x.w : x.z) : ((gid & 2) ? x.y : x.x);
  }
  static __device__ __forceinline__ uint32_t vsel(int gid) {
    const uint32_t b = 2 * (gid & 1);
    return b | ((b + 1) << 4) | ((4 + b) << 8) | ((5 + b) << 12);
  }
  static __device__ __forceinline__ int vpos0(int) { return 0; }
  static __device__ __forceinline__ int vpos1(int) { return 0; }
  static __device__ __forceinline__ void value_a(uint32_t x, int,
                                                 uint32_t &r0, uint32_t &r1) {
    r0 = x & 0x00FF00FFu;
    r1 = (x >> 8) & 0x00FF00FFu;
  }
};

// ---- compile-time configuration ---------------------------------------------

template <int D_, int BITS_, int GQP_, int G_, bool SINK_ = false>
struct Cfg {
  static constexpr int D = D_, BITS = BITS_, GQP = GQP_, G = G_;
  // KIVI-Sink caches: the instantiation that masks sink tokens' scores
  static constexpr bool SINK = SINK_;
  // CTAs per SM the register budget is cut for: 4-bit stages (10.75 KB at
  // D = 128) allow one stage per warp only, so those kernels take more
  // warps (16, at most 128 registers) in place of a deeper pipeline; the
  // others keep 12-14 warps with two stages each
  static constexpr int MINB = BITS == 4 && G >= 32 ? 16 : 12;
  static constexpr int KS = D / 16;            // score K-steps = value m16 tiles
  static constexpr int NJ = D / G;             // value groups per row
  static constexpr int WG = 4 / GQP;           // key groups per score window
  static constexpr int ROW = D * BITS / 8;     // bytes per token row
  static constexpr int ROWQ = ROW / 16;        // uint4 per token row
  static constexpr int NVB = (GQP * NJ + 3) / 4;         // value B blocks
  static constexpr int WT = WG * G;            // tokens per score window
  static constexpr int NWIN = WT >= kC ? 1 : kC / WT;    // windows per chunk
  static constexpr int MPW = 4 / NWIN;         // m16 tiles per window
  static constexpr int CG = G >= kC ? 1 : kC / G;        // key groups per chunk
  static constexpr int KG = WG > CG ? WG : CG;           // key groups staged
  // stage layout (bytes)
  static constexpr uint32_t S_KC = 0;
  static constexpr uint32_t S_VC = S_KC + kC * ROW;
  static constexpr uint32_t S_KS = S_VC + kC * ROW;
  static constexpr uint32_t S_KZ = S_KS + KG * D * 2;
  static constexpr uint32_t S_VS = S_KZ + KG * D * 2;
  static constexpr uint32_t S_VZ = S_VS + kC * NJ * 2;
  static constexpr uint32_t S_BYTES = (S_VZ + kC * NJ * 2 + 127) / 128 * 128;
  // per-warp layout: [mbarriers][q' GQP x D, channel c scaled by the
  // 2^-oexp of its score slot and the head's power of two: f32, or for
  // fragment-order codes its fp16 hi and lo halves in the same bytes][q'
  // GQP x D f32][stages].
  static constexpr uint32_t W_QF = 128;
  static constexpr uint32_t W_QN = W_QF + GQP * D * 4;
  static constexpr uint32_t W_STAGE0 = (W_QN + GQP * D * 4 + 127) / 128 * 128;
  static __host__ __device__ constexpr uint32_t warp_bytes(int ST) {
    return W_STAGE0 + ST * S_BYTES;
  }
};

// reduce over the lanes that share this lane's query head: all lanes with the
// same tig % GQP (xor over gid, and over the tig bits at and above GQP)
template <int GQP, typename F>
__device__ __forceinline__ float head_reduce(float v, F op) {
  v = op(v, __shfl_xor_sync(kFull, v, 4));
  v = op(v, __shfl_xor_sync(kFull, v, 8));
  v = op(v, __shfl_xor_sync(kFull, v, 16));
  if constexpr (GQP < 2) v = op(v, __shfl_xor_sync(kFull, v, 1));
  if constexpr (GQP < 4) v = op(v, __shfl_xor_sync(kFull, v, 2));
  return v;
}

struct MaxOp {
  __device__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct AddOp {
  __device__ float operator()(float a, float b) const { return a + b; }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
  return v;
}

__device__ __forceinline__ int find_seq(const int32_t *prefix, int B,
                                        int item) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Position in the flattened chunk space, advanced one chunk at a time, with
// the counts of its sequence cached (nc chunks per head, Tq quantized
// tokens).
struct Cursor {
  int b, h, k;
  int nc, Tq;
  __device__ __forceinline__ void load(const MmaTable &tab) {
    nc = tab.nc[b]; Tq = tab.Tq[b];
  }
  __device__ __forceinline__ void init(int c, const Geometry &geo,
                                       const MmaTable &tab) {
    b = find_seq(tab.bprefix, geo.B, c);
    load(tab);
    const int local = c - tab.bprefix[b];
    h = local / nc;
    k = local - h * nc;
  }
  __device__ __forceinline__ void next(const Geometry &geo, const MmaTable &tab) {
    if (++k == nc) {
      k = 0;
      if (++h == geo.H_kv) {
        h = 0;
        do { ++b; } while (b < geo.B && tab.nc[b] == 0);
        if (b < geo.B) load(tab);
      }
    }
  }
};

template <class C>
__global__ void __launch_bounds__(kNW * 32, C::MINB)
k_decode_mma(Geometry geo, Planes pl, MmaArgs args, MmaTable tab) {
  using L = Layout<C::BITS>;
  constexpr int D = C::D, KS = C::KS, NJ = C::NJ, GQP = C::GQP, WG = C::WG;
  constexpr int G = C::G, ROW = C::ROW, ROWQ = C::ROWQ;
  extern __shared__ __align__(128) unsigned char smem[];

  // Launched as a programmatic dependent of the stream's previous kernel:
  // griddepcontrol.wait returns once its writes are visible.  That kernel
  // started only after everything before it completed (it waits before it
  // releases this grid), so when it is not a k_flush of this cache
  // (args.early) it writes nothing this kernel reads from the planes, and
  // each warp's first copies are issued before the wait.  The merge kernel
  // is released only after the wait (it reads the residual ring early).
  if (!args.early) asm volatile("griddepcontrol.wait;" ::: "memory");
  static_assert(kNW == 1, "one warp per CTA");
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int wg = blockIdx.x;
  if (wg >= args.W) return;
  const int64_t N = args.N, W = args.W;
  const int lo_c = (int)(wg * N / W), hi_c = (int)((wg + 1) * N / W);
  const int n_mine = hi_c - lo_c;
  if (n_mine <= 0) return;
  const int ST = args.ST, GQ = args.GQ;

  unsigned char *ws = smem;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ws);
  float *qb = reinterpret_cast<float *>(ws + C::W_QF);      // [GQP][D], slot-scaled
  float *qn = reinterpret_cast<float *>(ws + C::W_QN);      // [GQP][D]
  unsigned char *stage0 = ws + C::W_STAGE0;

  if (lane == 0) {
    for (int s = 0; s < ST; ++s) mbar_init(&bars[s]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  // ---- producer: lane 0 issues a chunk's bulk copies (key codes, value
  // codes, the key scale / zero rows where a score window or the warp's
  // range starts, value scale / zero rows) after posting the stage's
  // transaction bytes.  The key scale / zero rows are copied only where a
  // window or the range starts: every other chunk reuses the operand built
  // from an earlier stage.  The plane bases of the producer's head are
  // warp-uniform.
  const unsigned char *pb_kc = nullptr, *pb_vc = nullptr, *pb_ks = nullptr,
                      *pb_kz = nullptr, *pb_vs = nullptr, *pb_vz = nullptr;
  auto set_prod_head = [&](const Cursor &cu) {
    const size_t hd = (size_t)cu.b * geo.H_kv + cu.h;
    const size_t r0 = hd * geo.Tcap, g0 = hd * (geo.Tcap / G);
    pb_kc = pl.Kc + r0 * ROW;
    pb_vc = pl.Vc + r0 * ROW;
    pb_ks = reinterpret_cast<const unsigned char *>(pl.Ks + g0 * D);
    pb_kz = reinterpret_cast<const unsigned char *>(pl.Kz + g0 * D);
    pb_vs = reinterpret_cast<const unsigned char *>(pl.Vs + r0 * NJ);
    pb_vz = reinterpret_cast<const unsigned char *>(pl.Vz + r0 * NJ);
  };
  auto issue = [&](const Cursor &cu, int s, int c) {
    const int t0 = cu.k * kC;
    const int rem = cu.Tq - t0;
    const int nvalid = rem < kC ? rem : kC;
    const bool with_ks = (t0 % C::WT) == 0 || c == lo_c;
    const int kg0 = ((t0 / G) / C::KG) * C::KG;
    const int ngv = cu.Tq / G - kg0;
    const int ng = ngv < C::KG ? ngv : C::KG;
    const bool go = c != args.fail_chunk;   // testing: copies that never come
    unsigned char *sb = stage0 + s * C::S_BYTES;
    if (lane == 0 && go) {
      mbar_expect_tx(&bars[s], 2 * (nvalid * (ROW + NJ * 2) + (with_ks ? ng * D * 2 : 0)));
      bulk_g2s(sb + C::S_KC, pb_kc + (size_t)t0 * ROW, nvalid * ROW, &bars[s]);
      bulk_g2s(sb + C::S_VC, pb_vc + (size_t)t0 * ROW, nvalid * ROW, &bars[s]);
      if (with_ks) {
        bulk_g2s(sb + C::S_KS, pb_ks + (size_t)kg0 * D * 2, ng * D * 2, &bars[s]);
        bulk_g2s(sb + C::S_KZ, pb_kz + (size_t)kg0 * D * 2, ng * D * 2, &bars[s]);
      }
      bulk_g2s(sb + C::S_VS, pb_vs + (size_t)t0 * NJ * 2, nvalid * NJ * 2, &bars[s]);
      bulk_g2s(sb + C::S_VZ, pb_vz + (size_t)t0 * NJ * 2, nvalid * NJ * 2, &bars[s]);
    }
    __syncwarp();
  };
  // the producer's step for the chunk at pc: its copies into stage s (all
  // lanes call it)
  auto produce = [&](const Cursor &cu, int s, int c) {
    if (cu.k == 0 || c == lo_c) set_prod_head(cu);
    issue(cu, s, c);
  };

  Cursor pc;  // producer cursor: the next chunk to issue
  pc.init(lo_c, geo, tab);
  uint32_t phase = 0;    // bit s = parity to wait for on stage s
  uint32_t pending = 0;  // bit s = copies in flight into stage s
  for (int i = 0; i < ST && i < n_mine; ++i) {
    produce(pc, i, lo_c + i);
    pending |= 1u << i;
    pc.next(geo, tab);
  }
  if (args.early) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  bool failed = false;

  // ---- per-lane constants ------------------------------------------------
  const uint32_t s_sel = L::score_sel(tig);
  const uint32_t v_sel = L::vsel(gid);
  const float rs0 = exp2i(24 - L::vpos0(gid)), rs1 = exp2i(24 - L::vpos1(gid));
  const int hl = gid & 1;               // B operand column: hi (0) or lo (1)
  const HiLo hls{hl ? 0x80000000u : 0u, hl ? 1.f : 0.f};
  const int pair_b = gid >> 1;          // B operand column pair
  const int h_b = pair_b % GQP;         // query head of the B column pair
  const int h_s = tig % GQP;            // this lane's query head (C layout)
  const int gw_s = tig / GQP;           // this lane's key group in a window

  // ---- running state of the current head segment ---------------------------
  float O[KS][4];
  // zero-point sums sum_t p_t z_t,j.  With one query head per kv head they
  // are taken in the value B layout (ZB), where every lane holds the p of
  // its tokens: Z[vb] covers column pair pair_b of value block vb over the
  // lane's tokens.  Otherwise in the score layout: Z[j] of head h_s, group
  // j over the lane's score rows.
  constexpr bool ZB = GQP == 1;
  constexpr int NZ = ZB ? C::NVB : NJ;
  float Z[NZ];
  float m_run = -INFINITY, l_run = 0.f;
  uint32_t Bs[KS][2];
  float beta_t = 0.f;    // zero-point term of pair tig, current window
  float unscale_t = 1.f; // 2^(24 - k) of this lane's score head
  int cur_w = -1;
  // KIVI-Sink: the head's sinks in the quantized region, one position per
  // lane (-1: none); sk_lo / sk_hi bound them (a chunk outside skips the
  // per-token test).  Their scores are masked here; the merge kernel adds
  // them from their fp16 rows.
  int my_sink = -1, sk_lo = 0x7fffffff, sk_hi = -1;
  auto load_sinks = [&](int b, int h, int Tq) {
    my_sink = -1;
    if (lane < geo.n_sink) {
      const int p = __ldg(pl.sink_pos + ((size_t)b * geo.H_kv + h) * geo.n_sink + lane);
      if (p >= 0 && p < Tq) my_sink = p;
    }
    sk_lo = __reduce_min_sync(kFull, my_sink >= 0 ? my_sink : 0x7fffffff);
    sk_hi = __reduce_max_sync(kFull, my_sink);
  };

  auto reset_state = [&]() {
#pragma unroll
    for (int mv = 0; mv < KS; ++mv)
#pragma unroll
      for (int r = 0; r < 4; ++r) O[mv][r] = 0.f;
#pragma unroll
    for (int j = 0; j < NZ; ++j) Z[j] = 0.f;
    m_run = -INFINITY;
    l_run = 0.f;
    cur_w = -1;
  };

  // q' of the head's GQP query heads: qn in channel order; qb with channel
  // c scaled by 2^-oexp(c) of its score slot and by the head's power of two
  // 2^k, which puts the bound max|q'| * max s_K of the score operand's
  // products (over every key group of the kv head) in [2^13, 2^14) — no
  // fp16 overflow, and the lo parts of the large products stay in fp16's
  // normal range — unless that would take max|q'| itself past 2^15 (small
  // key scales): q' enters the operand as fp16 hi + lo, so k is capped
  // there, and the products then stay further below fp16's limit.
  // unscale_t = 2^(24 - k) of this lane's score head.
  auto load_q = [&](int b, int h) {
    constexpr int NQ = GQP * D / 32;
    float mq[GQP], vb[NQ];
#pragma unroll
    for (int hh = 0; hh < GQP; ++hh) mq[hh] = 0.f;
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      const int i = lane + 32 * j;
      constexpr int PER = D / 32;
      const int hh = j / PER, c = i - hh * D;
      float v = 0.f;
      if (hh < GQ)
        v = __half2float(__ldcg(args.q + ((size_t)b * geo.H_q + h * GQ + hh) * D + c)) *
            args.scale_log2;
      vb[j] = v * exp2i(-L::oexp(c));
      qn[i] = v;
      mq[hh] = fmaxf(mq[hh], fabsf(vb[j]));
    }
    const float smax = __half2float(__ushort_as_half(
        (unsigned short)__ldcg(pl.ksmax + (size_t)b * geo.H_kv + h)));
    int kh[GQP];
#pragma unroll
    for (int hh = 0; hh < GQP; ++hh) {
      float m = mq[hh];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
      int k = 13 - (((__float_as_int(m * smax) >> 23) & 0xff) - 127);
      // q' itself stays below 2^15 (it enters the operand as fp16 hi + lo):
      // with small key scales the product bound alone would overflow it
      const int kq = 14 - (((__float_as_int(m) >> 23) & 0xff) - 127);
      if (kq < k) k = kq;
      kh[hh] = k < -60 ? -60 : (k > 60 ? 60 : k);
    }
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      constexpr int PER = D / 32;
      const float x = vb[j] * exp2i(kh[j / PER]);
      if constexpr (L::FRAG) {
        // fp16 hi + lo of the scaled q' (qb's region holds them): the score
        // operand is built from them in fp16 arithmetic.  With 4 query
        // heads per kv head, per 4-channel group 4 hi then 4 lo halves (one
        // 16-byte load per lane and K-step; measured faster there, while
        // one head keeps two arrays of halves, which needs fewer registers)
        const int i = lane + 32 * j;
        const __half xh = __float2half_rn(x);
        const __half xl = __float2half_rn(x - __half2float(xh));
        __half *q16 = reinterpret_cast<__half *>(qb);
        if constexpr (GQP == 4) {
          q16[2 * (i & ~3) + (i & 3)] = xh;
          q16[2 * (i & ~3) + (i & 3) + 4] = xl;
        } else {
          q16[i] = xh;
          q16[GQP * D + i] = xl;
        }
      } else {
        qb[lane + 32 * j] = x;
      }
    }
    int kl = kh[0];
#pragma unroll
    for (int hh = 1; hh < GQP; ++hh)
      if (hh == h_s) kl = kh[hh];
    unscale_t = exp2i(24 - kl);
    __syncwarp();
  };

  // B operand of the score MMA for the window starting at key group gw0 (the
  // stage's key scale/zero region starts at group kg0; qb carries the
  // head's operand scaling), and, for this lane's column pair, the
  // zero-point term beta.
  auto build_score_b = [&](const __half *Ks, const __half *Kz, int gw0, int kg0) {
    const int gr = gw0 + pair_b / GQP - kg0;   // group row in the region
    const __half *ksr = Ks + gr * D + 4 * tig;
    if constexpr (L::FRAG) {
      // products q' s in fp16 pairs: hi = RN(qh s), its exact rounding
      // error e = qh s - hi (at most 11 significant bits: representable),
      // lo = RN(ql s + e); hi + lo carries ~21 bits of q' s.  Slot order is
      // channel order here, so a pair of channels is one register.
      const __half *q16 = reinterpret_cast<const __half *>(qb);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint2 sr = *reinterpret_cast<const uint2 *>(ksr + 16 * ks);
        uint2 hr, lr;
        if constexpr (GQP == 4) {
          const uint4 q4 = *reinterpret_cast<const uint4 *>(
              q16 + 2 * (h_b * D + 4 * tig) + 32 * ks);   // hi 4, lo 4
          hr = make_uint2(q4.x, q4.y);
          lr = make_uint2(q4.z, q4.w);
        } else {
          hr = *reinterpret_cast<const uint2 *>(q16 + h_b * D + 4 * tig + 16 * ks);
          lr = *reinterpret_cast<const uint2 *>(q16 + GQP * D + h_b * D + 4 * tig + 16 * ks);
        }
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const uint32_t sw = w ? sr.y : sr.x, hw = w ? hr.y : hr.x, lw = w ? lr.y : lr.x;
          const __half2 sv2 = *reinterpret_cast<const __half2 *>(&sw);
          const __half2 h2 = *reinterpret_cast<const __half2 *>(&hw);
          const __half2 l2 = *reinterpret_cast<const __half2 *>(&lw);
          const __half2 hi = __hmul2(h2, sv2);
          const __half2 e = __hfma2(h2, sv2, __hneg2(hi));
          const __half2 lo = __hfma2(l2, sv2, e);
          const __half2 pick = hl ? lo : hi;
          Bs[ks][w] = *reinterpret_cast<const uint32_t *>(&pick);
        }
      }
    } else {
      const float *qbh = qb + h_b * D + 4 * tig;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint2 sraw = *reinterpret_cast<const uint2 *>(ksr + 16 * ks);
        const float4 qs = *reinterpret_cast<const float4 *>(qbh + 16 * ks);
        const float2 s01 = __half22float2(*reinterpret_cast<const __half2 *>(&sraw.x));
        const float2 s23 = __half22float2(*reinterpret_cast<const __half2 *>(&sraw.y));
        // channel order 4tig + 0..3
        const float2 a01 = hilo2(__fmul2_rn(f2(qs.x, qs.y), s01), hls);
        const float2 a23 = hilo2(__fmul2_rn(f2(qs.z, qs.w), s23), hls);
        const float a[4] = {a01.x, a01.y, a23.x, a23.y};
        // slot order: slot e holds channel 4tig + off(e)
        Bs[ks][0] = pack_half2(a[L::off(0)], a[L::off(1)]);
        Bs[ks][1] = pack_half2(a[L::off(2)], a[L::off(3)]);
      }
    }
    // zero-point term: the hi and lo lanes of a pair take half the K-steps
    const float *qnh = qn + h_b * D + 4 * tig;
    const __half *kzr = Kz + gr * D + 4 * tig;
    float2 zacc = f2(0.f, 0.f);
#pragma unroll
    for (int kk = 0; kk < KS / 2; ++kk) {
      const int ks = hl * (KS / 2) + kk;
      const float4 qz = *reinterpret_cast<const float4 *>(qnh + 16 * ks);
      const uint2 zr = *reinterpret_cast<const uint2 *>(kzr + 16 * ks);
      zacc = __ffma2_rn(f2(qz.x, qz.y),
                        __half22float2(*reinterpret_cast<const __half2 *>(&zr.x)), zacc);
      zacc = __ffma2_rn(f2(qz.z, qz.w),
                        __half22float2(*reinterpret_cast<const __half2 *>(&zr.y)), zacc);
    }
    float zpart = zacc.x + zacc.y;
    zpart += __shfl_xor_sync(kFull, zpart, 1);
    zpart += __shfl_xor_sync(kFull, zpart, 2);
    zpart += __shfl_xor_sync(kFull, zpart, 4);   // hi + lo lanes of the pair
    // lane (gid, tig) needs the values of pair tig, held by lanes gid = 2*tig
    beta_t = __shfl_sync(kFull, zpart, 8 * tig);
  };

  // write this warp's partial of head hd (slot wg + hd); k_merge_mma, run
  // after the decode kernel, merges each head's partials
  auto flush = [&](int hd) {
    float Lsum = head_reduce<GQP>(l_run, AddOp());
    float Zt[NJ];
    if constexpr (ZB) {
      // pair tig of block vb is (head h_s, group (4 vb + tig) / GQP): sum
      // over the lanes of column pair p (gid = 2p, 2p+1, every tig), then
      // take pair tig's sum from lane 8 tig
#pragma unroll
      for (int j = 0; j < NJ; ++j) Zt[j] = 0.f;
#pragma unroll
      for (int vb = 0; vb < C::NVB; ++vb) {
        float r = Z[vb];
        r += __shfl_xor_sync(kFull, r, 1);
        r += __shfl_xor_sync(kFull, r, 2);
        r += __shfl_xor_sync(kFull, r, 4);
        r = __shfl_sync(kFull, r, 8 * tig);
#pragma unroll
        for (int j = 0; j < NJ; ++j)
          if (((j * GQP) >> 2) == vb) Zt[j] = r;
      }
    } else {
#pragma unroll
      for (int j = 0; j < NJ; ++j) Zt[j] = head_reduce<GQP>(Z[j], AddOp());
    }
    if (h_s < GQ) {
      float *dst = args.part + ((size_t)(wg + hd) * GQP + h_s) * part_stride<D>();
#pragma unroll
      for (int mv = 0; mv < KS; ++mv) {
        const int j = (16 * mv) / G;
        const int vb = (j * GQP) >> 2;
        if ((4 * vb + tig) / GQP != j) continue;
        const int c0 = 16 * mv + 2 * gid;
        // rows gid / gid+8 of tile mv (channels c0, c0+1) arrive scaled by
        // 2^(p - 24) for the code's bit position p
        float sa = rs0, sb = rs1;
        if constexpr (L::FRAG) {
          sa = exp2i(24 - L::fexp(2 * (mv % L::KPW)));
          sb = exp2i(24 - L::fexp(2 * (mv % L::KPW) + 1));
        }
        const float o0 = (O[mv][0] + O[mv][1]) * sa + Zt[j];
        const float o1 = (O[mv][2] + O[mv][3]) * sb + Zt[j];
        __stcg(reinterpret_cast<float2 *>(dst + c0), make_float2(o0, o1));
      }
      if (gid == 0 && tig < GQP)
        __stcg(reinterpret_cast<float2 *>(dst + D), make_float2(m_run, Lsum));
    }
  };

  // ---- one staged chunk, in two halves of two m16 tiles (32 tokens):
  // scores(0), softmax(0), then scores(1) and values(0) in one straight-line
  // block (independent work the scheduler interleaves), softmax(1),
  // values(1).  FULL: all four tiles hold tokens (every chunk but a head's
  // last quantized one). ----
  auto chunk = [&](auto full_tag, const unsigned char *st, int t0, int nmt,
                   uint64_t smask) {
    constexpr bool FULL = decltype(full_tag)::value;
    constexpr int MPW = C::MPW;
    const uint4 *kc = reinterpret_cast<const uint4 *>(st + C::S_KC);
    const uint4 *vc = reinterpret_cast<const uint4 *>(st + C::S_VC);
    const __half *Ks = reinterpret_cast<const __half *>(st + C::S_KS);
    const __half *Kz = reinterpret_cast<const __half *>(st + C::S_KZ);
    const __half *Vs = reinterpret_cast<const __half *>(st + C::S_VS);
    const __half *Vz = reinterpret_cast<const __half *>(st + C::S_VZ);
    const int G0 = t0 / G;                        // first key group
    const int kg0 = (G0 / C::KG) * C::KG;
    float sv[4][2];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) sv[mt][0] = sv[mt][1] = -INFINITY;
    float p[4][2];

    // score MMAs of tiles T0 .. T0+NT-1 (one window) with the current B
    auto score_tiles = [&](auto t0_tag, auto nt_tag, float (&acc)[2][4]) {
      constexpr int T0 = decltype(t0_tag)::value, NT = decltype(nt_tag)::value;
      if constexpr (L::FRAG) {
        // fragment order: lane group tig's NH words of a token row are
        // contiguous; word hw holds K-steps KPW hw ... KPW hw + KPW - 1
        constexpr int NH = D * C::BITS / 128, KPW = L::KPW;
        using RowW = std::conditional_t<NH == 4, uint4, std::conditional_t<NH == 2, uint2, uint32_t>>;
        RowW r0[NT], r1[NT];
#pragma unroll
        for (int m = 0; m < NT; ++m) {
          const unsigned char *row = st + C::S_KC + (16 * (T0 + m) + gid) * ROW + 4 * NH * tig;
          r0[m] = *reinterpret_cast<const RowW *>(row);
          r1[m] = *reinterpret_cast<const RowW *>(row + 8 * ROW);
        }
#pragma unroll
        for (int hw = 0; hw < NH; ++hw) {
          uint32_t w0[NT], w1[NT], s0[NT], s1[NT];
#pragma unroll
          for (int m = 0; m < NT; ++m) {
            if constexpr (NH == 1) {
              w0[m] = r0[m];
              w1[m] = r1[m];
            } else {
              w0[m] = reinterpret_cast<const uint32_t *>(&r0[m])[hw];
              w1[m] = reinterpret_cast<const uint32_t *>(&r1[m])[hw];
            }
            s0[m] = w0[m] >> L::SHIFT;
            s1[m] = w1[m] >> L::SHIFT;
          }
#pragma unroll
          for (int kk = 0; kk < KPW; ++kk) {
            const int ks = KPW * hw + kk;
#pragma unroll
            for (int m = 0; m < NT; ++m) {
              if (FULL || T0 + m < nmt) {
                mma16816(acc[m], L::field(w0[m], s0[m], 2 * kk),
                         L::field(w1[m], s1[m], 2 * kk),
                         L::field(w0[m], s0[m], 2 * kk + 1),
                         L::field(w1[m], s1[m], 2 * kk + 1), Bs[ks][0], Bs[ks][1]);
              }
            }
          }
        }
      } else {
#pragma unroll
        for (int q = 0; q < KS / L::WPQ; ++q) {
          uint4 r0[NT], r1[NT];
#pragma unroll
          for (int m = 0; m < NT; ++m) {
            const uint4 *row = kc + (16 * (T0 + m) + gid) * ROWQ;
            r0[m] = row[q];
            r1[m] = row[8 * ROWQ + q];
          }
#pragma unroll
          for (int kq = 0; kq < L::WPQ; ++kq) {
            const int ks = q * L::WPQ + kq;
#pragma unroll
            for (int m = 0; m < NT; ++m) {
              if (FULL || T0 + m < nmt) {
                uint32_t a0, a1, a2, a3;
                L::score_a(r0[m], ks, s_sel, a0, a2);
                L::score_a(r1[m], ks, s_sel, a1, a3);
                mma16816(acc[m], a0, a1, a2, a3, Bs[ks][0], Bs[ks][1]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int m = 0; m < NT; ++m) {
        const int mt = T0 + m;
        if ((FULL || mt < nmt) && ((G0 + (16 * mt) / G) % WG) == gw_s) {
          sv[mt][0] = fmaf(acc[m][0] + acc[m][1], unscale_t, beta_t);
          sv[mt][1] = fmaf(acc[m][2] + acc[m][3], unscale_t, beta_t);
        }
      }
    };

    // scores of half H (tiles 2H, 2H+1), window by window.  A window that
    // spans the chunk (NWIN == 1) may continue from the previous chunk; a
    // smaller one is always new.
    auto scores_half = [&](auto h_tag) {
      constexpr int H = decltype(h_tag)::value;
      constexpr int WA = (2 * H) / MPW, WB = (2 * H + 1) / MPW;
#pragma unroll
      for (int win = WA; win <= WB; ++win) {
        const int ta = win * MPW > 2 * H ? win * MPW : 2 * H;   // first tile
        if (!FULL && ta >= nmt) continue;
        if (C::NWIN > 1 || H == 0) {
          const int gw0 = ((G0 + (16 * win * MPW) / G) / WG) * WG;
          if (C::NWIN > 1 || gw0 != cur_w) {
            build_score_b(Ks, Kz, gw0, kg0);
            cur_w = gw0;
          }
        }
        float acc[2][4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[m][r] = 0.f;
        if constexpr (MPW == 1) {
          if (win == WA)
            score_tiles(std::integral_constant<int, 2 * H>{}, std::integral_constant<int, 1>{}, acc);
          else
            score_tiles(std::integral_constant<int, 2 * H + 1>{}, std::integral_constant<int, 1>{}, acc);
        } else {
          score_tiles(std::integral_constant<int, 2 * H>{}, std::integral_constant<int, 2>{}, acc);
        }
      }
    };

    // online softmax update with the scores of half H; the head maximum is
    // reduced only when some lane holds a score above the running maximum
    auto softmax_half = [&](auto h_tag) {
      constexpr int H = decltype(h_tag)::value;
      if (smask) {
        // sink tokens of this chunk: bit (token - t0) of smask
#pragma unroll
        for (int mt = 2 * H; mt < 2 * H + 2; ++mt)
#pragma unroll
          for (int r = 0; r < 2; ++r)
            if ((smask >> (16 * mt + gid + 8 * r)) & 1ull) sv[mt][r] = -INFINITY;
      }
      const float lmax = fmaxf(fmaxf(sv[2 * H][0], sv[2 * H][1]),
                               fmaxf(sv[2 * H + 1][0], sv[2 * H + 1][1]));
      float alpha = 1.f;
      if (__any_sync(kFull, lmax > m_run)) {
        const float m_new = fmaxf(m_run, head_reduce<GQP>(lmax, MaxOp()));
        alpha = m_run == -INFINITY ? 0.f : exp2_neg(m_run - m_new);
        m_run = m_new;
        const float2 a2 = f2(alpha, alpha);
#pragma unroll
        for (int mv = 0; mv < KS; ++mv) {
          const float2 o01 = __fmul2_rn(f2(O[mv][0], O[mv][1]), a2);
          const float2 o23 = __fmul2_rn(f2(O[mv][2], O[mv][3]), a2);
          O[mv][0] = o01.x; O[mv][1] = o01.y; O[mv][2] = o23.x; O[mv][3] = o23.y;
        }
#pragma unroll
        for (int j = 0; j < NZ; ++j) Z[j] *= alpha;
      }
      // with sinks masked a head's first half may hold no score at all
      // (m_run still -inf): subtract 0 there, so that every weight is 0
      const float msub = (smask && m_run == -INFINITY) ? 0.f : m_run;
#pragma unroll
      for (int mt = 2 * H; mt < 2 * H + 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) p[mt][r] = exp2_neg(sv[mt][r] - msub);   // -inf -> 0
      const float psum = (p[2 * H][0] + p[2 * H][1]) + (p[2 * H + 1][0] + p[2 * H + 1][1]);
      l_run = fmaf(l_run, alpha, psum);
    };

    // ---- values of K-step kt = tokens 16kt ... 16kt+15 of the chunk.  K
    // slots (2tig, 2tig+1, 2tig+8, 2tig+9) <-> tokens (tig, tig+4, tig+8,
    // tig+12): the four rows a lane group reads hit distinct banks. ----
    auto values_kt = [&](auto kt_tag) {
      constexpr int kt = decltype(kt_tag)::value;
      if (!FULL && kt >= nmt) return;
      // p of head h_b for tokens tig, tig+4, tig+8, tig+12
      const int src = ((G0 + (16 * kt) / G) % WG) * GQP + h_b;
      const float p0 = __shfl_sync(kFull, p[kt][0], 4 * tig + src);
      const float p1 = __shfl_sync(kFull, p[kt][0], 4 * tig + 16 + src);
      const float p2 = __shfl_sync(kFull, p[kt][1], 4 * tig + src);
      const float p3 = __shfl_sync(kFull, p[kt][1], 4 * tig + 16 + src);
      const int ta = 16 * kt + tig;
      if constexpr (ZB) {
        // zero-point term in the B layout: the hi lane of a column pair
        // takes tokens ta, ta+4, the lo lane ta+8, ta+12
        const float pz0 = hl ? p2 : p0, pz1 = hl ? p3 : p1;
        const int tz = ta + 8 * hl;
#pragma unroll
        for (int vb = 0; vb < C::NVB; ++vb) {
          const int jb = (4 * vb + pair_b) / GQP;
          if (jb < NJ) {
            const float z0 = __half2float(Vz[tz * NJ + jb]);
            const float z1 = __half2float(Vz[(tz + 4) * NJ + jb]);
            Z[vb] = fmaf(pz0, z0, fmaf(pz1, z1, Z[vb]));
          }
        }
      }
      // zero-point term in the score layout (tokens gid, gid+8)
      if constexpr (!ZB) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float vz[NJ];
          load_halves<NJ>(Vz + (16 * kt + gid + 8 * r) * NJ, vz);
          if constexpr (NJ == 1) {
            Z[0] = fmaf(p[kt][r], vz[0], Z[0]);
          } else {
#pragma unroll
            for (int j = 0; j < NJ; j += 2) {
              const float2 z = __ffma2_rn(f2(p[kt][r], p[kt][r]), f2(vz[j], vz[j + 1]),
                                          f2(Z[j], Z[j + 1]));
              Z[j] = z.x; Z[j + 1] = z.y;
            }
          }
        }
      }
      // s_V of the four tokens: whole rows when every block needs a
      // different group, single values otherwise
      float vs[4][C::NVB];
      if constexpr (C::NVB == NJ && NJ >= 2) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float row[NJ];
          load_halves<NJ>(Vs + (ta + 4 * u) * NJ, row);
#pragma unroll
          for (int vb = 0; vb < C::NVB; ++vb) vs[u][vb] = row[(4 * vb + pair_b) / GQP];
        }
      } else {
#pragma unroll
        for (int vb = 0; vb < C::NVB; ++vb) {
          const int jb = (4 * vb + pair_b) / GQP;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            vs[u][vb] = jb < NJ ? __half2float(Vs[(ta + 4 * u) * NJ + jb]) : 0.f;
        }
      }
      uint32_t bv[C::NVB][2];
#pragma unroll
      for (int vb = 0; vb < C::NVB; ++vb) {
        const float2 w01 = hilo2(__fmul2_rn(f2(p0, p1), f2(vs[0][vb], vs[1][vb])), hls);
        const float2 w23 = hilo2(__fmul2_rn(f2(p2, p3), f2(vs[2][vb], vs[3][vb])), hls);
        bv[vb][0] = pack_half2(w01.x, w01.y);
        bv[vb][1] = pack_half2(w23.x, w23.y);
      }
      if constexpr (L::FRAG) {
        // fragment order: pair (ta, ta+4) is pair tig of block kt, pair
        // (ta+8, ta+12) pair 4+tig; lane gid's NV words of a pair are
        // contiguous, word hw covering tiles KPW hw ... KPW hw + KPW - 1
        constexpr int NV = D * C::BITS / 128, KPW = L::KPW;
        using PairW = std::conditional_t<NV == 4, uint4, std::conditional_t<NV == 2, uint2, uint32_t>>;
        const unsigned char *blk = st + C::S_VC + kt * 16 * ROW;
        const PairW pa = *reinterpret_cast<const PairW *>(blk + (8 * tig + gid) * 4 * NV);
        const PairW pb = *reinterpret_cast<const PairW *>(blk + (8 * (4 + tig) + gid) * 4 * NV);
#pragma unroll
        for (int hw = 0; hw < NV; ++hw) {
          uint32_t wa, wb;
          if constexpr (NV == 1) {
            wa = pa;
            wb = pb;
          } else {
            wa = reinterpret_cast<const uint32_t *>(&pa)[hw];
            wb = reinterpret_cast<const uint32_t *>(&pb)[hw];
          }
          const uint32_t sa = wa >> L::SHIFT, sb = wb >> L::SHIFT;
#pragma unroll
          for (int mm = 0; mm < KPW; ++mm) {
            const int mv = KPW * hw + mm;
            const int vb = (((16 * mv) / G) * GQP) >> 2;
            mma16816(O[mv], L::field(wa, sa, 2 * mm), L::field(wa, sa, 2 * mm + 1),
                     L::field(wb, sb, 2 * mm), L::field(wb, sb, 2 * mm + 1),
                     bv[vb][0], bv[vb][1]);
          }
        }
      } else {
        // m16 channel tiles, VTPQ per uint4 of the token rows
#pragma unroll
        for (int q = 0; q < KS / L::VTPQ; ++q) {
          const uint4 xa = vc[ta * ROWQ + q];
          const uint4 xb = vc[(ta + 4) * ROWQ + q];
          const uint4 xc = vc[(ta + 8) * ROWQ + q];
          const uint4 xd = vc[(ta + 12) * ROWQ + q];
#pragma unroll
          for (int u = 0; u < L::VTPQ; ++u) {
            const int mv = q * L::VTPQ + u;
            const int vb = (((16 * mv) / G) * GQP) >> 2;
            uint32_t a0, a1, a2, a3;
            L::value_a(__byte_perm(L::vword(xa, u, gid), L::vword(xb, u, gid), v_sel),
                       gid, a0, a1);
            L::value_a(__byte_perm(L::vword(xc, u, gid), L::vword(xd, u, gid), v_sel),
                       gid, a2, a3);
            mma16816(O[mv], a0, a1, a2, a3, bv[vb][0], bv[vb][1]);
          }
        }
      }
    };

    using I0 = std::integral_constant<int, 0>;
    using I1 = std::integral_constant<int, 1>;
    using I2 = std::integral_constant<int, 2>;
    using I3 = std::integral_constant<int, 3>;
    scores_half(I0{});
    softmax_half(I0{});
    scores_half(I1{});
    values_kt(I0{});
    values_kt(I1{});
    softmax_half(I1{});
    values_kt(I2{});
    values_kt(I3{});
  };

  // ---- main loop over my chunks ---------------------------------------------
  Cursor cu;
  cu.init(lo_c, geo, tab);
  int cur_hd = -1;
  int s = 0;   // stage of chunk i (= i mod ST)
  for (int i = 0; i < n_mine; ++i) {
    const int hd = cu.b * geo.H_kv + cu.h;
    if (hd != cur_hd) {
      reset_state();
      load_q(cu.b, cu.h);
      if constexpr (C::SINK) load_sinks(cu.b, cu.h, cu.Tq);
      cur_hd = hd;
    }
    {
      const bool ok = __all_sync(kFull, mbar_wait(&bars[s], (phase >> s) & 1u));
      if (!ok) { failed = true; break; }
      phase ^= 1u << s;
      pending &= ~(1u << s);
      const unsigned char *st = stage0 + s * C::S_BYTES;
      const int t0 = cu.k * kC;
      const int rem = cu.Tq - t0;
      uint64_t smask = 0;
      if (C::SINK && sk_hi >= t0 && sk_lo < t0 + kC) {
        const int d = my_sink - t0;
        const bool in = my_sink >= 0 && d >= 0 && d < kC;
        const unsigned lo = __reduce_or_sync(kFull, in && d < 32 ? 1u << d : 0u);
        const unsigned hi = __reduce_or_sync(kFull, in && d >= 32 ? 1u << (d - 32) : 0u);
        smask = (uint64_t)lo | ((uint64_t)hi << 32);
      }
      if (rem >= kC) {
        chunk(std::true_type{}, st, t0, 4, smask);
      } else {
        chunk(std::false_type{}, st, t0, rem >> 4, smask);
      }
    }
    const bool head_ends = cu.k == cu.nc - 1 || i == n_mine - 1;
    if (head_ends) flush(hd);
    __syncwarp();
    if (i + ST < n_mine) {
      // every lane read the stage: order those reads before the copies
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      produce(pc, s, lo_c + i + ST);
      pending |= 1u << s;
      pc.next(geo, tab);
    }
    cu.next(geo, tab);
    if (++s == ST) s = 0;
  }

  if (failed) {
    if (lane == 0) atomicOr(args.err, 1u);
    // let every copy still in flight land (bounded) before the CTA's shared
    // memory can be reused
    for (int j = 0; j < ST; ++j)
      if (pending & (1u << j)) mbar_wait(&bars[j], (phase >> j) & 1u);
  }
}

// ---- merge of the per-warp partials and the fp16 residual window ---------
//
// One CTA per (sequence, kv head, query head, channel slice): NSL =
// min(4 / GQP, D / 32) slices of D / NSL channels, so that one query head
// per kv head keeps four CTAs of 32 channels and four query heads one CTA
// each over all channels (every window score is then computed once per
// slice, never once per head and slice).  nw <= kMergeWarps warps, sized by
// the launcher.  Warp j first takes the residual window's tokens j,
// j + nw, ... (kMergeRT at a time): lanes hold 32-channel strides of the
// key row and of the head's q' (one warp-wide sum gives a score) and the
// slice's channels of the value row.  Then, once the decode kernel's
// writes are visible, the partials: those of kv head hd sit in slots w + hd
// for the warps w whose chunk range touches the head, and warp j merges
// partials j, j + nw, ... (kMergeU at a time, all in flight).  Every warp
// keeps a running (max, sum, o); warp 0 then combines the warps' states
// with a log-sum-exp.  The unroll depths keep the CTAs small (4 warps for
// the usual window and partial counts), so that every CTA of a large batch
// runs in one wave and, where the decode kernel leaves room on an SM, the
// CTAs reside beside it and read the residual window while it runs.
constexpr int kMergeWarps = 16;
constexpr int kMergeU = 16;
constexpr int kMergeRT = 8;

template <int D, int GQP> __host__ __device__ constexpr int merge_slices() {
  return (4 / GQP) < (D / 32) ? (4 / GQP) : (D / 32);
}

template <int D, int GQP>
__global__ void __launch_bounds__(kMergeWarps * 32)
k_merge_mma(Geometry geo, Planes pl, MmaArgs args, MmaTable tab) {
  constexpr int CPL = D / 32;                       // key channels per lane
  constexpr int NSL = merge_slices<D, GQP>();
  constexpr int SW = D / NSL, OC = SW / 32;         // slice width, o per lane
  __shared__ float sm_m[kMergeWarps], sm_l[kMergeWarps];
  __shared__ float sm_o[kMergeWarps][SW];
  // let the stream's next kernel launch now: whatever it writes that this
  // kernel reads (the residual ring for an append, the partials for a
  // decode) it writes only after its own griddepcontrol.wait, which waits
  // for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;");
  const int b = blockIdx.x / geo.H_kv, h = blockIdx.x - b * geo.H_kv;
  const int hq = blockIdx.y;                        // query head of the kv head
  const int nq = tab.nq[b], nres = tab.nres[b];
  if (nq == 0 && nres == 0) return;   // no tokens: the launcher zeroed it
  const int GQ = args.GQ;
  const int hd = b * geo.H_kv + h;
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  const int c0 = blockIdx.z * SW + lane;            // channel of o[0]; o[u] at c0 + 32 u

  float m_run = -INFINITY, l_run = 0.f, o_run[OC];
#pragma unroll
  for (int u = 0; u < OC; ++u) o_run[u] = 0.f;
  // fold n entries (m_e, l_e, o_e) into the running state; entries with
  // m = -inf (empty partial slots, tokens past the end) weigh nothing
  auto fold = [&](const float *me, const float *le, const float (*oe)[OC], int n) {
    float mr = m_run;
    for (int e = 0; e < n; ++e) mr = fmaxf(mr, me[e]);
    if (mr == -INFINITY) return;
    const float a = m_run == -INFINITY ? 0.f : exp2_neg(m_run - mr);
    l_run *= a;
#pragma unroll
    for (int u = 0; u < OC; ++u) o_run[u] *= a;
    for (int e = 0; e < n; ++e) {
      const float f = me[e] == -INFINITY ? 0.f : exp2_neg(me[e] - mr);
      l_run = fmaf(f, le[e], l_run);
#pragma unroll
      for (int u = 0; u < OC; ++u) o_run[u] = fmaf(f, oe[e][u], o_run[u]);
    }
    m_run = mr;
  };

  // (1) the fp16 residual window: tokens T_q ... T_q + nres - 1 in ring
  // slots (T_q + t) mod Rcap.  When the decode kernel ran (N > 0), the ring
  // and q were written before it released this grid (it waits for the
  // append first), so the window is read, from L2, while it drains;
  // otherwise the append itself precedes this kernel and is waited for.
  if (args.N <= 0) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (nres > 0) {
    float qv[CPL];
    {
      const __half *qrow = args.q + ((size_t)b * geo.H_q + h * GQ + hq) * D;
#pragma unroll
      for (int u = 0; u < CPL; ++u)
        qv[u] = __half2float(__ldcg(qrow + lane + 32 * u)) * args.scale_log2;
    }
    const size_t ring0 = (size_t)hd * geo.Rcap;
    const int Tq = tab.Tq[b];
    for (int t0 = wp; t0 < nres; t0 += nw * kMergeRT) {
      float kv[kMergeRT][CPL], vv[kMergeRT][OC], me[kMergeRT], le[kMergeRT];
      bool ok[kMergeRT];
#pragma unroll
      for (int r = 0; r < kMergeRT; ++r) {
        const int t = t0 + r * nw;
        ok[r] = t < nres;
        const size_t row = (ring0 + (Tq + (ok[r] ? t : t0)) % geo.Rcap) * D;
#pragma unroll
        for (int u = 0; u < CPL; ++u) kv[r][u] = __half2float(__ldcg(pl.Kr + row + lane + 32 * u));
#pragma unroll
        for (int u = 0; u < OC; ++u) vv[r][u] = __half2float(__ldcg(pl.Vr + row + c0 + 32 * u));
      }
#pragma unroll
      for (int r = 0; r < kMergeRT; ++r) {
        float sc = 0.f;
#pragma unroll
        for (int u = 0; u < CPL; ++u) sc = fmaf(qv[u], kv[r][u], sc);
        sc = warp_sum(sc);
        me[r] = ok[r] ? sc : -INFINITY;
        le[r] = 1.f;
      }
      fold(me, le, vv, kMergeRT);
    }
  }

  // (1b) KIVI-Sink: sinks of the quantized region, from their fp16 rows
  // (written at prefill; the decode kernel masked their quantized slots)
  if (geo.n_sink > 0) {
    const int Tq = tab.Tq[b];
    const __half *qrow = args.q + ((size_t)b * geo.H_q + h * GQ + hq) * D;
    for (int k = wp; k < geo.n_sink; k += nw) {
      const int t = __ldg(pl.sink_pos + (size_t)hd * geo.n_sink + k);
      if (t < 0 || t >= Tq) continue;
      const size_t row = ((size_t)hd * geo.n_sink + k) * D;
      float sc = 0.f;
#pragma unroll
      for (int u = 0; u < CPL; ++u)
        sc = fmaf(__half2float(__ldcg(qrow + lane + 32 * u)) * args.scale_log2,
                  __half2float(__ldg(pl.sink_k + row + lane + 32 * u)), sc);
      sc = warp_sum(sc);
      float vv[1][OC];
#pragma unroll
      for (int u = 0; u < OC; ++u) vv[0][u] = __half2float(__ldg(pl.sink_v + row + c0 + 32 * u));
      const float one = 1.f;
      fold(&sc, &one, vv, 1);
    }
  }

  // (2) the decode kernel's partials, visible once griddepcontrol.wait
  // returns
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (nq > 0) {
    const int64_t N = args.N, W = args.W;
    const int64_t cs = tab.bprefix[b] + (int64_t)h * tab.nc[b];
    const int64_t ce = cs + tab.nc[b];
    const int w0 = (int)(((cs + 1) * W - 1) / N);
    const int n = (int)((ce * W - 1) / N) - w0 + 1;
    for (int k0 = wp; k0 < n; k0 += nw * kMergeU) {
      float me[kMergeU], le[kMergeU], oe[kMergeU][OC];
#pragma unroll
      for (int u = 0; u < kMergeU; ++u) {
        const int k = k0 + u * nw;
        const bool ok = k < n;
        const float *e = args.part +
                         ((size_t)(w0 + (ok ? k : k0) + hd) * GQP + hq) * part_stride<D>();
        const float2 ml = ok ? __ldcg(reinterpret_cast<const float2 *>(e + D))
                             : make_float2(-INFINITY, 0.f);
        me[u] = ml.x;
        le[u] = ml.y;
#pragma unroll
        for (int v = 0; v < OC; ++v) oe[u][v] = ok ? __ldcg(e + c0 + 32 * v) : 0.f;
      }
      fold(me, le, oe, kMergeU);
    }
  }

  // (3) the warps' states combined
  if (lane == 0) { sm_m[wp] = m_run; sm_l[wp] = l_run; }
#pragma unroll
  for (int u = 0; u < OC; ++u) sm_o[wp][lane + 32 * u] = o_run[u];
  __syncthreads();
  if (wp == 0) {
    float M = -INFINITY;
    for (int j = 0; j < nw; ++j) M = fmaxf(M, sm_m[j]);
    float L = 0.f, o[OC];
#pragma unroll
    for (int u = 0; u < OC; ++u) o[u] = 0.f;
    for (int j = 0; j < nw; ++j) {
      const float f = sm_m[j] == -INFINITY ? 0.f : exp2_neg(sm_m[j] - M);
      L = fmaf(f, sm_l[j], L);
#pragma unroll
      for (int u = 0; u < OC; ++u) o[u] = fmaf(f, sm_o[j][lane + 32 * u], o[u]);
    }
    float *orow = args.out + ((size_t)b * geo.H_q + h * GQ + hq) * D;
#pragma unroll
    for (int u = 0; u < OC; ++u) orow[c0 + 32 * u] = o[u] / L;
  }
}

using MergeFn = void (*)(Geometry, Planes, MmaArgs, MmaTable);

template <int D, int GQP>
MergeFn merge_fn() {
  return &k_merge_mma<D, GQP>;
}

using KernelFn = void (*)(Geometry, Planes, MmaArgs, MmaTable);

struct KernelInfo {
  KernelFn fn;
  uint32_t stage_bytes, stage0;
};

template <class C>
KernelInfo info() {
  return KernelInfo{&k_decode_mma<C>, C::S_BYTES, C::W_STAGE0};
}

// the instantiations of one bit width (decode_mma_b{2,4,8}.cu; with sink
// masking, decode_mma_sink_b{2,4,8}.cu)
bool kernel_b2(int D, int GQP, int G, KernelInfo *out);
bool kernel_b4(int D, int GQP, int G, KernelInfo *out);
bool kernel_b8(int D, int GQP, int G, KernelInfo *out);
bool kernel_sink_b2(int D, int GQP, int G, KernelInfo *out);
bool kernel_sink_b4(int D, int GQP, int G, KernelInfo *out);
bool kernel_sink_b8(int D, int GQP, int G, KernelInfo *out);

}  // namespace mma
}  // namespace vqk
