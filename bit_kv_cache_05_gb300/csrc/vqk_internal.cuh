// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "vq_kivi.h"

namespace vqk {

constexpr int kMaxB = 256;        // sequences per cache
constexpr int kMaxGroupHeads = 8; // H_q / H_kv
constexpr int kMaxD = 256;

// Device memory of one cache, carved from a single cudaMallocAsync block.
struct Planes {
  uint8_t *Kc, *Vc;          // [B][H_kv][Tcap][row]        packed codes
  __half *Ks, *Kz;           // [B][H_kv][Tcap/g][D]        key scale / zero
  __half *Vs, *Vz;           // [B][H_kv][Tcap][D/g]        value scale / zero
  __half *Kr, *Vr;           // [B][H_kv][Rcap][D]          residual ring
  float *part;               // [B][H_q][max_items][D+2]    split partials
  uint32_t *ksmax;           // [B][H_kv] fp16 bits of the largest key scale
                             // flushed for the head (a bound for the decode)
  // KIVI-Sink store (Geometry::n_sink > 0): per (b, h) the sink tokens'
  // positions, ascending, -1 in unused slots, and their fp16 rows
  int32_t *sink_pos = nullptr;   // [B][H_kv][n_sink]
  __half *sink_k = nullptr;      // [B][H_kv][n_sink][D]
  __half *sink_v = nullptr;      // [B][H_kv][n_sink][D]
  // Kitty (Geometry::kitty): the 4-bit channels of every key group, the
  // fp16 values of the quantized tokens, and per (b, h, channel) the running
  // sums of the quantized keys in 2^-24 units (sum x: int64; sum x^2: a
  // 128-bit integer as two uint64, low word first)
  uint32_t *kmask = nullptr;     // [B][H_kv][Tcap/g][D/32]
  __half *Vf = nullptr;          // [B][H_kv][Tcap][D]
  long long *ksum = nullptr;     // [B][H_kv][D]
  unsigned long long *ksq = nullptr;  // [B][H_kv][D][2]
  // AgeTieredKV (Geometry::age_b1 > 0): each group's current tier
  int8_t *tier = nullptr;        // [B][H_kv][Tcap/g]
};

constexpr int kMaxSink = 16;     // sinks per (sequence, kv head)

// orders of the code planes (see "code-plane orders" below)
constexpr int kLayoutPacked = 0;
constexpr int kLayoutFrag = 1;

struct Geometry {
  int B, H_q, H_kv, D, bits, g, R;
  int Tcap;   // quantized-token capacity per sequence (multiple of g)
  int Rcap;   // residual ring slots per sequence (R + g)
  int row;    // packed bytes per token row (D*bits/8)
  int max_items;  // decode work items per sequence (quantized splits + 1)
  int layout = kLayoutPacked;   // order of the code planes (below)
  int n_sink = 0;               // KIVI-Sink tokens per (sequence, kv head)
  int kitty = 0;                // Kitty cache (mixed 4/2-bit keys, fp16 values)
  int kitty_hi = 0;             // Kitty: 4-bit channels per key group
  // AgeTieredKV (age_b1 > 0): a group whose newest token has fewer than
  // age_b1 newer tokens is stored at age_bits[0], fewer than age_b2 at
  // age_bits[1], else at age_bits[2].  A group owns g * D bytes of a code
  // plane (its rows at the widest width); at width w its g rows are packed
  // densely in the leading g * D * w / 8 bytes (age_row_off)
  int age_b1 = 0, age_b2 = 0;
  int age_bits[3] = {0, 0, 0};
};

// 64-bit words of one chunk of a Kitty flush's ranking totals: an int64 sum
// and a 128-bit sum of squares per (sequence, kv head, channel)
inline size_t kitty_chunk_words(const Geometry &geo) {
  return (size_t)geo.B * geo.H_kv * 3 * geo.D;
}

// floats of the decode's partial buffer (CUDA-core and staged decodes):
// B * H_q * max_items * (D + 2).  A Kitty flush borrows the buffer for its
// ranking totals, so a Kitty cache's holds at least one chunk of them.
inline size_t part_floats(const Geometry &geo) {
  size_t n = (size_t)geo.B * geo.H_q * geo.max_items * (geo.D + 2);
  if (geo.kitty && 2 * kitty_chunk_words(geo) > n) n = 2 * kitty_chunk_words(geo);
  return n;
}

// AgeTieredKV tier of group G of a sequence of S tokens
__host__ __device__ inline int age_tier(const Geometry &geo, int S, int G) {
  const int age = S - (G + 1) * geo.g;
  return age < geo.age_b1 ? 0 : (age < geo.age_b2 ? 1 : 2);
}

// width of AgeTieredKV tier t (selects, so that a kernel does not index its
// parameter block at run time)
__host__ __device__ inline int age_width(const Geometry &geo, int t) {
  return t == 0 ? geo.age_bits[0] : (t == 1 ? geo.age_bits[1] : geo.age_bits[2]);
}

// Byte offset in an AgeTieredKV code plane of row i (0 <= i < g) of group G
// of (sequence, kv head) bh, the group stored at width w: the group's block
// starts at its first token's row of D bytes, its rows follow at D * w / 8
// bytes (LSB-first codes, as a packed row).  The export expands them to
// D-byte rows.
__host__ __device__ inline size_t age_row_off(const Geometry &geo, size_t bh,
                                              int G, int i, int w) {
  return (bh * geo.Tcap + (size_t)G * geo.g) * geo.D + (size_t)i * (geo.D * w / 8);
}

// One AgeTieredKV flush: per sequence b, new groups [gn0, gn1) quantized
// from fp16 (token position p from the residual ring below src_split, else
// input row p - src_split) to their tier at length S_new, and stored groups
// in [gd0, gd1) moved from their tier at S_old to their tier at S_new.
struct AgeTable {
  int32_t prefix[kMaxB + 1];   // items (new groups, then demotions) per b
  int32_t gn0[kMaxB], gn1[kMaxB];
  int32_t gd0[kMaxB], gd1[kMaxB];
  int32_t src_split[kMaxB];
  int32_t S_old[kMaxB], S_new[kMaxB];
};
cudaError_t launch_age_flush(const Geometry &geo, const Planes &pl,
                             const __half *Kin, const __half *Vin,
                             int64_t in_stride, const AgeTable &tab,
                             cudaStream_t st);


// ---- code-plane orders --------------------------------------------------
//
// kLayoutPacked: the method's packing, code of channel c of a token row at
// byte c*b/8, bit (c*b) mod 8 (LSB first); every export uses this order.
// kLayoutFrag: 2- and 4-bit codes of a cache decoded on the tensor cores, in
// the order the decode kernel's MMA fragments consume them (same bytes per
// row and per 16-token block, permuted so that one and-mask per register,
// after at most one shift of the word, yields two codes in place).  A 32-bit
// word has two 16-bit halves of 16/b fields each; field r of a half sits at
// bits 16*half + b*r.  With KPW = 8/b (K-steps, or value tiles, per word) and
// NW = D*b/128 (words per lane group):
//  keys, per token row of D*b/32 words: channel c = 16 ks + 4 tig + e sits
//    in word NW tig + ks/KPW, half e mod 2, field 2 (ks mod KPW) + e/2;
//  values, per 16-token block of D*b/2 words: the block's tokens pair up as
//    (tl, tl + 4), tl in {0..3, 8..11}, pair index pi = tl (tl < 4) or
//    tl - 4; channel c = 16 mv + 2 j + rho of both tokens of pair pi sits in
//    word (8 pi + j) NW + mv/KPW, field 2 (mv mod KPW) + rho, the first
//    token in the low half, the second in the high half.
struct FragPos {
  int word;   // 32-bit word within the token row (keys) or block (values)
  int bit;    // position of the field in that word
};

__host__ __device__ inline FragPos frag_key(int D, int b, int c) {
  const int kpw = 8 / b, nw = D * b / 128;
  const int ks = c >> 4, tig = (c >> 2) & 3, e = c & 3;
  const int r = 2 * (ks % kpw) + (e >> 1);
  return FragPos{nw * tig + ks / kpw, 16 * (e & 1) + b * r};
}

// tl: token within its 16-token block
__host__ __device__ inline FragPos frag_value(int D, int b, int tl, int c) {
  const int kpw = 8 / b, nw = D * b / 128;
  const int u = tl & 7, s = u >> 2, pi = 4 * (tl >> 3) + (u & 3);
  const int mv = c >> 4, j = (c & 15) >> 1, rho = c & 1;
  const int r = 2 * (mv % kpw) + rho;
  return FragPos{(8 * pi + j) * nw + mv / kpw, 16 * s + b * r};
}

// Codes of channels c0 ... c0+7 (c0 a multiple of 8) of one quantized token:
// keys from the token's row krow, values from the token's 16-token block
// vblk (tl = token within the block), in the cache's own order: packed (the
// 8 codes are b consecutive bytes of the row) or MMA-fragment (2 words for
// keys, 4 for values, by frag_key / frag_value specialised to 8 channels of
// one 16-channel step).
__device__ inline void codes8(const Geometry &geo, const uint8_t *krow,
                              const uint8_t *vblk, int tl, int c0,
                              uint32_t (&kc)[8], uint32_t (&vc)[8]) {
  const int b = geo.bits;
  const uint32_t m = (1u << b) - 1u;
  if (geo.layout == kLayoutFrag) {
    const int kpw = 8 / b, nw = geo.D * b / 128;
    const int ks = c0 >> 4, h = (c0 >> 3) & 1, r0 = 2 * (ks % kpw);
    const uint32_t *kw = reinterpret_cast<const uint32_t *>(krow);
    for (int q = 0; q < 2; ++q) {              // tig = 2h + q: channels 4q ... 4q+3
      const uint32_t w = kw[nw * (2 * h + q) + ks / kpw];
      for (int e = 0; e < 4; ++e)
        kc[4 * q + e] = (w >> (16 * (e & 1) + b * (r0 + (e >> 1)))) & m;
    }
    const int u = tl & 7, sh = 16 * (u >> 2), pi = 4 * (tl >> 3) + (u & 3);
    const uint32_t *vw = reinterpret_cast<const uint32_t *>(vblk);
    for (int jj = 0; jj < 4; ++jj) {           // j = (c0 & 15) / 2 + jj
      const uint32_t w = vw[(8 * pi + ((c0 & 15) >> 1) + jj) * nw + ks / kpw];
      for (int rho = 0; rho < 2; ++rho)
        vc[2 * jj + rho] = (w >> (sh + b * (r0 + rho))) & m;
    }
  } else {
    // 8 codes = b bytes at byte c0 * b / 8
    uint64_t kx = 0, vx = 0;
    const uint8_t *kp = krow + c0 * b / 8, *vp = vblk + (size_t)tl * geo.row + c0 * b / 8;
    for (int i = 0; i < b; ++i) {
      kx |= (uint64_t)kp[i] << (8 * i);
      vx |= (uint64_t)vp[i] << (8 * i);
    }
    for (int e = 0; e < 8; ++e) {
      kc[e] = (uint32_t)(kx >> (b * e)) & m;
      vc[e] = (uint32_t)(vx >> (b * e)) & m;
    }
  }
}

// ---- quantize / flush ------------------------------------------------------

// One launch quantizes whole groups of g tokens of every (b, h).  Group k of
// sequence b (k in [0, n_groups[b])) covers token positions
// first_pos[b] + k*g ... + g-1.  Token position p of sequence b is read from
// the residual ring (slot p % Rcap) when p < src_split[b], otherwise from row
// p - src_split[b] of the input block [b][h] (stride in_stride rows).
struct FlushTable {
  int32_t prefix[kMaxB + 1];  // group-item prefix sums over b
  int32_t first_pos[kMaxB];
  int32_t src_split[kMaxB];
};

// Copy of input rows into the residual ring: for sequence b, input rows
// [row0[b], row0[b] + count[b]) go to token positions pos0[b] + i, stored at
// ring slot (pos0[b] + i) % Rcap.
struct TailTable {
  int32_t prefix[kMaxB + 1];  // token prefix sums over b
  int32_t row0[kMaxB];
  int32_t pos0[kMaxB];
};

cudaError_t launch_flush(const Geometry &geo, const Planes &pl,
                         const __half *Kin, const __half *Vin,
                         int64_t in_stride, const FlushTable &tab,
                         int total_groups, cudaStream_t st);
// KIVI-Sink: per (b, h) the min(n_sink, S_b) prefill tokens with the
// largest key norms (fp32 sum of squares in channel order; equal norms: the
// earlier token), their positions ascending in pl.sink_pos and their rows
// copied into pl.sink_k / pl.sink_v.  K, V: the prefill inputs.
struct SinkTable {
  int32_t S[kMaxB];
};
cudaError_t launch_pick_sinks(const Geometry &geo, const Planes &pl,
                              const __half *K, const __half *V,
                              int64_t s_stride, const SinkTable &tab,
                              cudaStream_t st);
// input_ready: Kin / Vin were complete before the append's first kernel
// (not written by the kernel before the ring append)
cudaError_t launch_tail(const Geometry &geo, const Planes &pl,
                        const __half *Kin, const __half *Vin,
                        int64_t in_stride, const TailTable &tab,
                        int total_tokens, bool input_ready, cudaStream_t st);
// code plane 0 (keys) or 3 (values) of a kLayoutFrag cache, converted to
// the packed order, into dst
cudaError_t launch_export_frag(const Geometry &geo, const uint8_t *src,
                               bool values, void *dst, cudaStream_t st);
cudaError_t launch_dequantize(const Geometry &geo, const Planes &pl,
                              const int32_t *Tq, const int32_t *nres,
                              __half *Kh, __half *Vh, int64_t s_stride,
                              cudaStream_t st);
cudaError_t launch_export_residual(const Geometry &geo, const Planes &pl,
                                   int which, void *dst, const int32_t *Tq,
                                   const int32_t *nres, cudaStream_t st);

// ---- decode ----------------------------------------------------------------

// Work list of one decode: for sequence b, items prefix[b] ... prefix[b+1]-1;
// local item k < nq[b] covers quantized tokens [k*tps, min((k+1)*tps, Tq[b])),
// local item k == nq[b] (present when nres[b] > 0) covers the residual.
// per sequence: quantized tokens and residual-window tokens
struct LenTable {
  int32_t Tq[kMaxB];
  int32_t nres[kMaxB];
};

struct DecodeTable {
  int32_t prefix[kMaxB + 1];
  int32_t Tq[kMaxB];
  int32_t nres[kMaxB];
  int32_t nq[kMaxB];
};

struct DecodeArgs {
  const __half *q;  // [B][H_q][D]
  float *out;       // [B][H_q][D]
  float scale_log2; // softmax scale * log2(e)
  int tps;          // quantized tokens per split item
  int total_items;
  unsigned *err = nullptr;  // set to nonzero when a pipeline wait gave up
};

cudaError_t launch_decode(const Geometry &geo, const Planes &pl,
                          const DecodeArgs &args, const DecodeTable &tab,
                          cudaStream_t st);
// the log-sum-exp merge of the split partials of launch_decode
cudaError_t launch_combine(const Geometry &geo, const Planes &pl,
                           const DecodeArgs &args, const DecodeTable &tab,
                           cudaStream_t st);

// ---- Kitty (kitty.cu): channel-wise mixed-precision keys, fp16 values ------
//
// Per key group of g tokens the kitty_hi channels with the largest running
// variance (N sum x^2 - (sum x)^2 over tokens 0 ... the group's last, in
// 128-bit integers of 2^-24 units; the smaller channel first on ties) get
// 4-bit codes, the other 2-bit.  A token row of Kc holds krow = (D +
// kitty_hi) / 4 bytes: the 4-bit channels' codes in ascending channel order,
// LSB first, then the 2-bit channels'.  Kmask marks the 4-bit channels of
// each group; values of quantized tokens are kept in fp16 in Vf.
cudaError_t launch_flush_kitty(const Geometry &geo, const Planes &pl,
                               const __half *Kin, const __half *Vin,
                               int64_t in_stride, const FlushTable &tab,
                               int total_groups, cudaStream_t st);
// CTAs of the Kitty decode resident per SM (its split is planned for one
// wave, as the AgeTieredKV decode's)
int kitty_decode_ctas_per_sm(const Geometry &geo);
cudaError_t launch_decode_kitty(const Geometry &geo, const Planes &pl,
                                const DecodeArgs &args, const DecodeTable &tab,
                                cudaStream_t st);
// CTAs of the AgeTieredKV decode resident per SM (its split is planned
// for one wave)
int age_decode_ctas_per_sm(const Geometry &geo);
// plane 0 (keys) or 3 (values) of an AgeTieredKV cache in D-byte rows (the
// packed row order): token t < T_q of each sequence holds its codes in the
// leading D * w / 8 bytes, zeros after them; rows t >= T_q are zero
cudaError_t launch_age_export(const Geometry &geo, const Planes &pl, bool values,
                              void *dst, const int32_t *Tq, cudaStream_t st);
// decode over an AgeTieredKV cache (tables as the CUDA-core decode); S =
// Tq + nres of a sequence gives every group's tier (age.cu)
cudaError_t launch_decode_age(const Geometry &geo, const Planes &pl,
                              const DecodeArgs &args, const DecodeTable &tab,
                              cudaStream_t st);

// ---- decode on the tensor cores (D = 64/128, H_q/H_kv <= 4) ---------------

// Flattened chunk space of the quantized tokens: sequence b owns chunks
// [bprefix[b], bprefix[b+1]), H_kv heads of nc[b] = nq[b] 64-token chunks
// each.  The fp16 residual window (nres[b] tokens from Tq[b]) is read by the
// merge kernel.
struct MmaTable {
  int32_t bprefix[kMaxB + 1];
  int32_t nc[kMaxB];
  int32_t nq[kMaxB];
  int32_t Tq[kMaxB];
  int32_t nres[kMaxB];
};

struct MmaArgs {
  const __half *q;   // [B][H_q][D]
  float *out;        // [B][H_q][D]
  float *part;       // partials: slot (warp + head) x GQp x (D + 2)
  unsigned *err;     // set to nonzero when a pipeline wait gave up
  float scale_log2;  // softmax scale * log2(e)
  int N;             // total chunks
  int fail_chunk;    // testing: chunk whose copies are not issued (-1: none)
  int early;         // 1: the previous kernel in the stream writes no code or
                     // metadata plane of this cache (it is not a k_flush of
                     // it), so the first copies may precede griddepcontrol.wait
  int W;             // warps used (<= N), filled in by the launcher
  int GQ, GQp, KG, ST;
};

struct MmaPlan {
  int GQ, GQp, KG, ST, chunk;
  unsigned smem;     // dynamic shared memory per CTA
  int warps_max;     // resident warps of the persistent grid
  int sm_count;      // SMs of the device
};

// false when the shape has no tensor-core kernel (then the CUDA-core kernel
// of launch_decode serves it)
bool mma_plan(const Geometry &geo, int sm_count, MmaPlan *plan);
size_t mma_part_floats(const Geometry &geo, const MmaPlan &plan);
cudaError_t launch_decode_mma(const Geometry &geo, const Planes &pl,
                              const MmaPlan &plan, MmaArgs args,
                              const MmaTable &tab, cudaStream_t st);

// ---- several query tokens per sequence (tcgen05, attend_multi.cu) ---------

struct MultiTable {
  int32_t S[kMaxB];    // tokens per sequence
  int32_t Tq[kMaxB];   // quantized tokens per sequence
};

struct MultiArgs {
  const __half *q;     // [B][H_q][S_q][D]
  float *out;          // [B][H_q][S_q][D]
  unsigned *err;       // set to nonzero when a wait gave up
  float scale_log2;    // softmax scale * log2(e)
  int S_q;             // query tokens per sequence (its newest S_q tokens)
  int GQ;              // query heads per kv head (1, 2, 4 or 8)
  // key-range splits per query tile (1: none).  With several, split 0
  // leaves its unnormalised rows in out, split k > 0 in part_o + (k - 1)
  // rows x D, and every split its rows' (max, sum) in part_ml + k rows; a
  // combine kernel merges them into out
  int splits = 1;
  float *part_o = nullptr;
  float2 *part_ml = nullptr;
};

// key-range splits for a multi-query attend: about 16 waves of CTAs (two
// per SM), at most 8 splits, each at least 8 key tiles of 64 tokens;
// split_tokens > 0 asks for about that many keys per split instead (tests,
// tuning)
int multi_splits(const Geometry &geo, const MultiArgs &args, const MultiTable &tab,
                 int sm_count, int split_tokens);

// D = 64 or 128; cudaErrorNotSupported when the driver offers no tensor-map
// encoder
cudaError_t launch_attend_multi(const Geometry &geo, const Planes &pl,
                                const MultiArgs &args, const MultiTable &tab,
                                cudaStream_t st);

// counts every kernel launch made by the library
void count_launch(int n = 1);

// launch with programmatic stream serialization: the kernel may be
// scheduled once the stream's previous kernel has released its dependents
// (griddepcontrol.launch_dependents), and waits for that kernel's writes
// with griddepcontrol.wait
template <typename... P, typename... A>
cudaError_t launch_pdl(void (*fn)(P...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, A... args) {
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, args...);
}

// sets the message vq_kivi_last_error() returns on the calling thread
void set_last_error(const char *msg);

}  // namespace vqk
