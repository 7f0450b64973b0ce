/*
 * vq_kivi.h -- C ABI of a KIVI-style 2/4/8-bit KV cache with a fused decode
 * step, for NVIDIA GB300 (sm_103a).
 *
 * The method (VeloxQuant-MLX pages):
 *  - Changelog v0.8.0 "New", KIVI: asymmetric group quantization with keys
 *    grouped per channel and values per token, an fp16 residual window
 *    (`residual_length`) and a group size (`kivi_group_size`).
 *  - Changelog v0.42.0 "Added", scalar_fused_decode_attend: attention runs
 *    directly over the quantized cache; k_hat / v_hat are rebuilt in
 *    registers inside a FlashAttention-style online softmax with fp32
 *    accumulation, so no dequantized K/V is ever written to memory.
 *  - Changelog v0.28.0: the residual is flushed in whole chunks and prefill
 *    and decode give the same quantized state.
 *  - veloxquant_mlx.cache API, KVCacheConfig fields residual_length
 *    (default 128) and kivi_group_size (default 32).
 *
 * Quantization (per group of g values x, fp32 arithmetic, IEEE rounding):
 *   scale = (max(x) - min(x)) / (2^b - 1)
 *   code  = scale == 0 ? 0 : clamp(rint((x - min(x)) / scale), 0, 2^b - 1)
 *   stored scale = fp16 round-to-nearest-even of scale; stored zero = min(x)
 * Keys: a group is g consecutive tokens of one channel.  Values: a group is
 * g consecutive channels of one token.  Dequantized value: code*scale + zero.
 *
 * Residual rule: a sequence of S tokens keeps its newest n_res tokens in
 * fp16 and the older T_q = S - n_res tokens quantized, where
 *   T_q = (S < R) ? 0 : g * floor((S - R) / g),   so R <= n_res < R + g
 * (or n_res = S when S < R).  Appends flush whole groups of g tokens.
 *
 * Decode (S_q = 1, no mask): for query head h (kv head h / (H_q/H_kv)),
 *   out[b][h] = sum_t softmax_t(scale * q[b][h] . k_hat_t) * v_hat_t
 * over every token t of sequence b, quantized and residual; fp32 result.
 * Empty sequences give an all-zero output row.
 *
 * Conventions for every entry point:
 *  - Device pointers are addresses in the memory of the CUDA device that is
 *    current on the calling thread; a cache must be used on the device that
 *    created it.  Host pointers are ordinary process memory.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *    are asynchronous and stream-ordered; nothing synchronizes the device
 *    except vq_kivi_free (see there).  A cache must not be used from two
 *    streams at once.
 *  - Every call returns a status: VQ_OK (0) or a negative VQ_ERR_* code.  A
 *    failing call leaves the cache as it was (except VQ_ERR_CUDA from an
 *    asynchronous fault, after which the cache contents are undefined).
 *    vq_kivi_last_error() gives a message for the last failure on the
 *    calling thread.  No call throws, aborts or traps.
 */
#ifndef VQ_KIVI_H
#define VQ_KIVI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define VQ_OK 0
#define VQ_ERR_ARG (-1)         /* null pointer, negative size, bad length */
#define VQ_ERR_UNSUPPORTED (-2) /* a shape or bit width the kernels lack */
#define VQ_ERR_CAPACITY (-3)    /* a sequence would exceed max_seq */
#define VQ_ERR_OOM (-4)         /* device or host allocation failed */
#define VQ_ERR_CUDA (-5)        /* a CUDA runtime call or launch failed */

/* Problem statement (changelog v0.42.0 workload: B, H, D, b, g, S_q=1, S_kv;
 * KVCacheConfig residual_length, kivi_group_size).
 *   B        batch (sequences), 1 <= B <= 256
 *   H_q      query heads; H_q % H_kv == 0, H_q / H_kv <= 8
 *   H_kv     key/value heads
 *   D        head dimension: 64, 128 or 256
 *   bits     code width: 2, 4 or 8
 *   group    g: 16, 32, 64 or 128, dividing D
 *   residual R: fp16 window, 0 <= R <= 4096
 *   max_seq  capacity in tokens per sequence, >= 0 */
typedef struct vq_kivi_params {
  int32_t B, H_q, H_kv, D, bits, group, residual, max_seq;
} vq_kivi_params;

/* Opaque cache handle.  It owns (device memory, from cudaMallocAsync on the
 * creating stream) the packed code planes, the fp16 scale/zero planes, the
 * fp16 residual ring and the split-KV workspace, and (host memory) the
 * per-sequence lengths, so no call needs a device-to-host read. */
typedef struct vq_kivi_cache vq_kivi_cache;

/* Prefill: build a cache from K, V and quantize each sequence's old tokens.
 * (Changelog v0.8.0 KIVI; the residual rule above.)
 *   p         parameters (host)
 *   K, V      device, fp16, [B][H_kv][s_stride][D] row-major; sequence b
 *             uses rows [0, seq_lens[b]) of its (b, h) block
 *   s_stride  rows per (b, h) block, >= max(seq_lens)
 *   seq_lens  host int32[B], 0 <= seq_lens[b] <= max_seq
 *   stream    cudaStream_t
 *   out       receives the new handle (unchanged on failure)
 * K and V are read by kernels on `stream`; keep them alive until then. */
int vq_kivi_quantize(const vq_kivi_params *p, const void *K, const void *V,
                     int64_t s_stride, const int32_t *seq_lens, void *stream,
                     vq_kivi_cache **out);

/* Options of a cache beyond the problem statement (all zero: plain KIVI).
 *   n_sink  KIVI-Sink (changelog v0.9.0 "New"): per (sequence, kv head) the
 *           n_sink prefill tokens with the largest key L2 norms (fp32 sum of
 *           squares, channel 0 first; on equal norms the earlier token) are
 *           kept in fp16 beside the cache and left out of their groups'
 *           min/max: a key group is quantized from its other tokens (the
 *           sink's codes are 0; a group of sinks only stores scale and zero
 *           +0), and a sink's own value groups are empty (scale, zero and
 *           codes 0).  Attention reads a sink of the quantized region from
 *           its fp16 rows.  Chosen once, at vq_kivi_quantize_ex, among all
 *           the prefill tokens; appended tokens never become sinks.
 *           0 <= n_sink <= 16; 0 is plain KIVI, bit for bit. */
typedef struct vq_kivi_options {
  int32_t n_sink;
  /* Kitty (changelog v0.11.0 "New"), kitty != 0: channel-wise
   * mixed-precision keys and fp16 values.  Every key group of g tokens
   * quantizes its kitty_hi channels of largest running variance in 4 bits
   * and the others in 2 bits (KIVI's per-channel group quantizer at that
   * width); the running variance of a group is taken over the tokens up to
   * the group's last one, exactly (N sum x^2 - (sum x)^2 in 128-bit
   * integers of 2^-24 units), the smaller channel first on ties.  Values
   * of quantized tokens are kept in fp16.  A key row holds (D + kitty_hi)/4
   * bytes: the 4-bit channels' codes in ascending channel order, LSB
   * first, then the 2-bit channels'.  Requires bits = 2, n_sink = 0,
   * D = 64 or 128, kitty_hi a multiple of 16 in [0, D], max_seq <= 2^20.  The pages'
   * default is kitty_hi = D / 4.  Decode runs on the CUDA cores;
   * vq_kivi_attend_multi and vq_kivi_dequantize do not serve Kitty caches
   * (VQ_ERR_UNSUPPORTED). */
  int32_t kitty;
  int32_t kitty_hi;
  /* AgeTieredKV (method overview, AgeTieredKV entry), age_recent > 0: three
   * widths of the group quantizer by token age.  A quantized group whose
   * newest token has fewer than age_recent newer tokens holds
   * age_bits_recent-bit codes, fewer than age_mid age_bits_mid-bit codes,
   * else age_bits_old-bit codes.  A group enters at the top tier and moves
   * down one tier at a time as it ages (on an append), re-quantized from
   * its values rebuilt in fp32 (code * scale, then + zero, each rounded to
   * nearest), so a prefill and any chunking of appends give the same
   * cache.  Rows of planes 0 and 3 are D bytes (the widest tier): a group's
   * codes fill their leading D * bits / 8 bytes, the rest zero.  Requires
   * bits = 8 (the row capacity), n_sink = 0, no Kitty, D = 64 or 128,
   * 0 < age_recent < age_mid, both multiples of g, widths in {2, 4, 8},
   * non-increasing.  The pages' defaults: 128, 1024, 8 / 4 / 2 bits.
   * Decode runs on the CUDA cores; vq_kivi_attend_multi and
   * vq_kivi_dequantize do not serve these caches (VQ_ERR_UNSUPPORTED). */
  int32_t age_recent, age_mid;
  int32_t age_bits_recent, age_bits_mid, age_bits_old;
} vq_kivi_options;

/* vq_kivi_quantize with options (NULL options = all zero). */
int vq_kivi_quantize_ex(const vq_kivi_params *p, const vq_kivi_options *opt,
                        const void *K, const void *V, int64_t s_stride,
                        const int32_t *seq_lens, void *stream,
                        vq_kivi_cache **out);

/* Append n_new[b] tokens to sequence b: push them onto the fp16 residual and
 * flush the oldest whole groups so that the residual rule holds again
 * (changelog v0.8.0 update_and_fetch; v0.28.0 chunk-flush).  The result is
 * bit-identical to a prefill of the whole sequence.
 *   K_new, V_new  device, fp16, [B][H_kv][n_stride][D]; rows [0, n_new[b])
 *   n_new         host int32[B], >= 0, S + n_new[b] <= max_seq
 * Returns VQ_ERR_CAPACITY (cache unchanged) if a sequence would overflow. */
int vq_kivi_append(vq_kivi_cache *c, const void *K_new, const void *V_new,
                   int64_t n_stride, const int32_t *n_new, void *stream);

/* Fused decode step over the quantized cache (changelog v0.42.0,
 * scalar_fused_decode_attend): split-KV online softmax rebuilding k_hat and
 * v_hat in registers, then a log-sum-exp merge of the splits.
 *   q              device, fp16, [B][H_q][D]  (one query token per sequence)
 *   out            device, fp32, [B][H_q][D]
 *   softmax_scale  <= 0 selects 1/sqrt(D)
 * Uses the cache's split workspace: one decode per cache in flight. */
int vq_kivi_decode_attend(vq_kivi_cache *c, const void *q, float *out,
                          float softmax_scale, void *stream);

/* One serving step from host memory: append one token per sequence, then
 * the fused decode step (the two calls above, changelog v0.8.0 and
 * v0.42.0), with the inputs in pinned host memory and the output written
 * into pinned host memory.  The kernels read the token's K and V and the
 * query through the pinned buffers' device mappings (no copy engine, no
 * second stream): a step that only adds the token to the residual window
 * reads them where they are; a step that also quantizes a group first
 * stores them into a device slot held by the cache, while the previous
 * step's last kernel finishes.  The decode stores its output rows straight
 * into h_out through its device mapping (no separate device-to-host copy).
 * Asynchronous like cudaMemcpyAsync: h_out holds the result once `stream`
 * has reached the end of the step, and the inputs may be overwritten only
 * then.
 *   h_k_new, h_v_new  pinned host, fp16, [B][H_kv][D], 16-byte aligned
 *   h_q               pinned host, fp16, [B][H_q][D], 16-byte aligned
 *   h_out             pinned host, fp32, [B][H_q][D], 16-byte aligned
 *   softmax_scale     <= 0 selects 1/sqrt(D)
 * VQ_ERR_ARG when a pointer is NULL, not pinned host memory or not
 * aligned; VQ_ERR_CAPACITY as vq_kivi_append (cache unchanged).  The first
 * call allocates the slot (B x (2 H_kv + H_q) x D x 2 bytes), released by
 * vq_kivi_free. */
int vq_kivi_step_host(vq_kivi_cache *c, const void *h_k_new,
                      const void *h_v_new, const void *h_q, float *h_out,
                      float softmax_scale, void *stream);

/* Several query tokens per sequence: multi-token (speculative) decode, or
 * attention of a chunk of tokens that was just appended (chunked prefill).
 * Attention over the same quantized cache (changelog v0.42.0 "Added":
 * k_hat / v_hat rebuilt from the codes, never written to global memory),
 * with a causal mask: the S_q queries of sequence b are its newest S_q
 * tokens, already in the cache, so query i is token S_b - S_q + i and
 * attends every token t <= S_b - S_q + i (quantized, residual window and
 * its own).  The pages' matrix-tiled prefill companion of another cache
 * (changelog v0.40.0 "Added") is the prior art for this shape of the work.
 * Runs on the tensor cores (tcgen05 with tensor-memory accumulators; the
 * query tile is brought in by a TMA tensor copy); k_hat, v_hat and the
 * softmax weights enter as fp16 hi + lo pairs, the softmax is fp32.
 *   q              device, fp16, [B][H_q][S_q][D], 16-byte aligned
 *   S_q            >= 1, at most the length of every sequence
 *   out            device, fp32, [B][H_q][S_q][D], 16-byte aligned
 *   softmax_scale  <= 0 selects 1/sqrt(D)
 * When the query tiles make few waves on the GPU (e.g. a 512-token chunk
 * of 8 sequences: 1024 CTAs on 304 slots) each tile's keys are cut into up
 * to 8 ranges (5 there), whose partial rows a second kernel merges with a
 * log-sum-exp;
 * their partials live in a scratch the cache allocates on first need
 * ((ranges - 1) x B x H_q x S_q x D x 4 bytes, plus 8 bytes per row and
 * range) and keeps.
 * Supported: D = 64 or 128 and H_q/H_kv in {1, 2, 4, 8}
 * (VQ_ERR_UNSUPPORTED otherwise); VQ_ERR_ARG when a sequence holds fewer
 * than S_q tokens; VQ_ERR_OOM when the scratch cannot be allocated.  Uses
 * none of the decode's workspace, so it may follow or precede
 * vq_kivi_decode_attend in any order on the cache's stream (two multi-query
 * calls on one cache share the scratch: one in flight at a time). */
int vq_kivi_attend_multi(vq_kivi_cache *c, const void *q, int32_t S_q,
                         float *out, float softmax_scale, void *stream);

/* Release the cache.  NULL is accepted.  Frees are stream-ordered on the
 * stream of the last call that used the cache, then that stream is
 * synchronized, so the handle's memory is gone when this returns. */
int vq_kivi_free(vq_kivi_cache *c);

/* ---- helpers ----------------------------------------------------------- */

/* Message of the last failure on the calling thread ("" if none).  The
 * string stays valid until the thread's next failing call. */
const char *vq_kivi_last_error(void);

/* Host copies of the per-sequence lengths: S (tokens), T_q (quantized),
 * n_res (fp16 residual).  Each pointer may be NULL; else int32[B]. */
int vq_kivi_lengths(const vq_kivi_cache *c, int32_t *S, int32_t *T_q,
                    int32_t *n_res);

/* The cache's parameters (host copy). */
int vq_kivi_get_params(const vq_kivi_cache *c, vq_kivi_params *p);

/* Canonical planes, for parity checks and inspection.  `which`:
 *   0 Kc  uint8 [B][H_kv][Tcap][D*bits/8]  key codes, LSB-first packing:
 *         code of channel e at byte e*bits/8, bit (e*bits) mod 8
 *   1 Ks  fp16  [B][H_kv][Tcap/g][D]       key scales (per channel, group)
 *   2 Kz  fp16  [B][H_kv][Tcap/g][D]       key zeros
 *   3 Vc  uint8 [B][H_kv][Tcap][D*bits/8]  value codes, same packing
 *   4 Vs  fp16  [B][H_kv][Tcap][D/g]       value scales (per token, group)
 *   5 Vz  fp16  [B][H_kv][Tcap][D/g]       value zeros
 *   6 Kr  fp16  [B][H_kv][R+g][D]          residual keys, slot i = token T_q+i
 *   7 Vr  fp16  [B][H_kv][R+g][D]          residual values
 *   8 sink positions  int32 [B][H_kv][n_sink]  ascending, -1 when unused
 *   9 sink keys       fp16  [B][H_kv][n_sink][D]
 *  10 sink values     fp16  [B][H_kv][n_sink][D]  (8-10: size 0 without sinks)
 *  11 Kitty 4-bit channel masks  uint32 [B][H_kv][Tcap/g][D/32]
 *  12 Kitty fp16 values          fp16   [B][H_kv][Tcap][D]
 *  13 AgeTieredKV group tiers    int8   [B][H_kv][Tcap/g]  (0 recent, 1 mid, 2 old)
 * A Kitty cache's plane 0 has rows of (D + kitty_hi)/4 bytes (see
 * vq_kivi_options) and planes 3-5 are empty; without Kitty 11-12 are empty,
 * without AgeTieredKV 13.
 * An empty plane has size 0 and its export does nothing.
 * where Tcap = ceil(max_seq/g)*g (at least g).  vq_kivi_plane_bytes gives
 * the size (0 for a bad `which`); vq_kivi_export writes the whole plane to
 * device memory `dst` of at least that size, on `stream`.  Only the valid
 * rows (tokens < T_q, slots < n_res) are defined.  A cache may hold its
 * code planes internally in another order of the same bytes (2- and 4-bit
 * caches decoded on the tensor cores keep them in the order the MMA fragments
 * consume them); the export always produces the packing described above. */
size_t vq_kivi_plane_bytes(const vq_kivi_cache *c, int which);
int vq_kivi_export(const vq_kivi_cache *c, int which, void *dst,
                   size_t dst_bytes, void *stream);

/* Dequantized copy of the cache: the unfused path that the pages measure the
 * fused decode against (changelog v0.42.0, scalar_fused_decode_attend: a
 * dequantize to fp16 K_hat / V_hat in memory, then a separate attention).
 * For every sequence b, kv head h and token t < S[b]:
 *   K_hat[b][h][t][c] = fp16_rn(fma(code, Ks, Kz)) for quantized tokens (the
 *   fp32 fma of the fp16 scale and zero, then rounded to fp16), and the fp16
 *   residual rows for the rest; V_hat likewise.  Rows t >= S[b] are not
 *   written.
 *   K_hat, V_hat  device, fp16, [B][H_kv][s_stride][D], 16-byte aligned,
 *                 caller-owned
 *   s_stride      >= the longest sequence
 * Returns VQ_ERR_ARG for NULL or misaligned outputs or a short stride. */
int vq_kivi_dequantize(const vq_kivi_cache *c, void *K_hat, void *V_hat,
                       int64_t s_stride, void *stream);

/* Bytes held, per the cache's byte accounting (changelog v0.8.0 "full
 * byte-accounting"): packed codes, fp16 scale/zero metadata and the fp16
 * residual, over the tokens currently stored (not the capacity), and the
 * fp16 size of the same tokens for comparison. */
typedef struct vq_kivi_bytes {
  uint64_t code_bytes, meta_bytes, residual_bytes, fp16_bytes;
  uint64_t sink_bytes;  /* fp16 K and V of the sinks in the quantized region
                           (a sink still in the residual window is counted
                           there, once) */
  uint64_t value_fp16_bytes;  /* Kitty: fp16 values of the quantized tokens */
} vq_kivi_bytes;
int vq_kivi_cache_bytes(const vq_kivi_cache *c, vq_kivi_bytes *out);

/* Decode work partition: about this many quantized tokens per split-KV work
 * item (a multiple of 64 and of g, at least the workspace minimum of 256),
 * or 0 for the automatic choice (the default); for the multi-query attend,
 * about this many keys per key range (at most 8 ranges).  Results are
 * invariant to it up to fp32 rounding; exposed for tests and tuning. */
int vq_kivi_set_split_tokens(vq_kivi_cache *c, int32_t tokens_per_split);

/* Number of kernels this library has launched in this process. */
uint64_t vq_kivi_launch_count(void);

/* Synchronizes the cache's last stream and reports whether a decode kernel
 * gave up on a pipeline wait since the last check (its waits are bounded, so
 * a stuck copy ends the kernel instead of hanging the GPU): VQ_OK, or
 * VQ_ERR_CUDA with a message (the flag is then cleared). */
int vq_kivi_device_status(vq_kivi_cache *c);

/* Which decode kernel serves this cache's shape: 1 = tensor-core kernel
 * (D = 64 or 128, H_q/H_kv <= 4), 0 = CUDA-core kernel; < 0 on error. */
int vq_kivi_decode_kernel(const vq_kivi_cache *c);

/* Testing hook for failure detection.  The next tensor-core decode on this
 * cache does not issue the shared-memory copies of global chunk `chunk`
 * (chunks are numbered over sequences, kv heads and 64-token chunks), so
 * the warp that owns it waits in vain: its bounded wait gives up after about
 * half a second, the kernel records the failure and returns, and
 * vq_kivi_device_status reports VQ_ERR_CUDA.  Nothing faults; the outputs
 * of that decode are not valid.  One-shot; -1 clears it. */
int vq_kivi_debug_fail_chunk(vq_kivi_cache *c, int32_t chunk);

/* ---- decode without any allocation ------------------------------------- */

/* The pages have no counterpart to this entry point; it exists for callers
 * that may not allocate device memory once they run (engines that reserve
 * all device memory at start-up and serve only from their own pool, plugins
 * whose host forbids allocations, latency-critical loops where cudaMalloc
 * would synchronize the device).  It computes the same fused decode step as
 * vq_kivi_decode_attend, from cache planes that the caller keeps in its own
 * device memory, and allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library call.  It runs the CUDA-core split-KV kernel over
 * packed-order planes for every shape (vq_kivi_decode_attend uses the
 * tensor-core kernel for D = 64 or 128 with at most 4 query heads per kv
 * head), so it is slower than the regular entry point on those shapes.
 *
 * Scratch: the split-KV partial results go to one fixed array of
 * VQ_KIVI_STATIC_SCRATCH_BYTES in this library's device memory, which every
 * GPU that loads the library holds until the process exits.  Every call
 * shares it and it keeps the last call's contents (nothing in it needs to
 * start at zero), so calls that overlap on the GPU -- on two streams, or
 * from two threads -- race and give wrong results: serialize them.  The first
 * call on each device looks up the array's device address on that device
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  With lazy module loading (CUDA_MODULE_LOADING
 * = LAZY, the default) that first call is also when the driver loads this
 * library's device code and the array onto the device: the one allocation
 * this entry point causes, made by the driver, once per device; later calls
 * allocate nothing.  The address stays valid for the life of the device's
 * primary context: after cudaDeviceReset (or anything else that destroys
 * that context) do not call this entry point again in the same process.
 *
 * Planes (device memory, 16-byte aligned; Tcap = ceil(max_seq/g)*g, at least
 * g; R = residual; per sequence T_q and n_res follow the residual rule):
 *   Kc, Vc  uint8 [B][H_kv][Tcap][D*bits/8]   as vq_kivi_export planes 0, 3
 *   Ks, Kz  fp16  [B][H_kv][Tcap/g][D]        as planes 1, 2
 *   Vs, Vz  fp16  [B][H_kv][Tcap][D/g]        as planes 4, 5
 *   Kr, Vr  fp16  [B][H_kv][R+g][D]  residual ring: the token at position p
 *           (T_q <= p < S) is in slot p mod (R+g)
 *   seq_lens host int32[B] (S per sequence); q, out, softmax_scale and stream
 *   as in vq_kivi_decode_attend.
 * Errors: VQ_ERR_CAPACITY when B*H_q*(D+2)*4 bytes times two work items
 * exceeds the scratch (or a length exceeds max_seq), VQ_ERR_ARG /
 * VQ_ERR_UNSUPPORTED as elsewhere; the message is in vq_kivi_last_error(). */
#define VQ_KIVI_STATIC_SCRATCH_BYTES (8u << 20)

typedef struct vq_kivi_planes {
  const void *Kc, *Ks, *Kz, *Vc, *Vs, *Vz, *Kr, *Vr;
} vq_kivi_planes;

int vq_kivi_decode_attend_static(const vq_kivi_params *p,
                                 const vq_kivi_planes *planes,
                                 const int32_t *seq_lens, const void *q,
                                 float *out, float softmax_scale,
                                 void *stream);

#ifdef __cplusplus
}
#endif

#endif /* VQ_KIVI_H */
