/*
 * mla72.h - C ABI of the B300 (sm_103a) MLA absorbed-decode library.
 *
 * The operation is one decode step of Multi-head Latent Attention in its
 * decode-time MQA form (kexue.fm "From MHA, MQA, GQA to MLA", section
 * "Part 3", eq. mla-mqa): every head s of a sequence attends, with its
 * absorbed query q_cat^(s) = [q_nope^(s) W_UK^(s), RoPE(q_rope^(s), pos)]
 * (d_c + d_r = 576 values), over the cached rows k_i = [c_i, k_R,i]
 * (the 512-d latent and the shared 64-d rotated RoPE key), with score scale
 * 1/sqrt(d_nope + d_r) = 1/sqrt(192); the probabilities are applied to c_i,
 * giving a 512-d latent output that W_UV maps to the 128-d value space
 * (kexue.fm eq. mla-mqa, first line: o_t = [o^(s) W_v^(s)]).  Per-head keys
 * and values are never formed.
 *
 * The step is four calls, all asynchronous on the caller's CUDA stream:
 *   mla_absorb_q   -> q_cat            (W_UK folded into the query; RoPE of q_R)
 *   mla_decode_fwd -> partials         (online softmax over the latent cache,
 *                                       balanced parts of all sequences' blocks)
 *   mla_combine    -> o_lat, lse       (log-sum-exp merge of the splits)
 *   mla_out_proj   -> out              (W_UV applied after attention)
 * plus the per-step cache write (mla_cache_append) and two preparation/test
 * helpers (mla_cache_fill, mla_paged_gather).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or synchronises.  Arrays are dense, row-major, in
 *     the shapes stated (last index fastest).
 *   - Tensor pointers and row strides must be 16-byte aligned (MLA_ERR_ALIGN
 *     otherwise).  When q_cat and o_part are 32-byte aligned (as every
 *     cudaMalloc or PyTorch allocation is), the tensor-core decode moves them
 *     with 32-byte accesses; otherwise with 16-byte ones, same results.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - mla_absorb_q, mla_decode_fwd(_multi), mla_combine, mla_combine_out_proj
 *     and mla_out_proj launch with programmatic stream serialization: their
 *     CTAs may be scheduled while the previous kernel of the stream finishes,
 *     and they read no memory before that kernel has completed, so stream
 *     order holds as for any launch.
 *   - Host-side argument checks run before anything is launched; on failure
 *     the call returns a negative mla_status and launches nothing.
 *   - A CUDA launch error is returned as MLA_ERR_LAUNCH.
 *   - Faults found on the device (a block-table entry outside the pool, a
 *     bounded pipeline wait that ran out) are written to *dev_status where a
 *     call takes one (0 = no fault; the word is only ever set, never cleared,
 *     by the library); the offending access is skipped, never performed.
 *   - No exception crosses the ABI.
 */
#ifndef MLA72_H
#define MLA72_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. */
typedef enum {
  MLA_F32 = 0,      /* IEEE binary32 */
  MLA_BF16 = 1,     /* bfloat16 */
  MLA_FP8E4M3 = 2   /* OCP FP8 E4M3 (latent cache only), one float32 scale per block */
} mla_dtype;

/* Return codes. */
typedef enum {
  MLA_OK = 0,
  MLA_ERR_ARG = -1,     /* null pointer, non-positive size, bad enum value */
  MLA_ERR_ALIGN = -2,   /* a pointer or row stride is not 16-byte aligned */
  MLA_ERR_DTYPE = -3,   /* unsupported dtype combination */
  MLA_ERR_SHAPE = -4,   /* dimensions outside what the kernels support */
  MLA_ERR_LAUNCH = -5,  /* CUDA reported an error at launch */
  MLA_ERR_DEVICE = -6   /* no usable CUDA device / wrong architecture */
} mla_status;

/* Values a kernel may write to *dev_status. */
#define MLA_DEV_OK 0
#define MLA_DEV_BAD_BLOCK 1      /* block_table entry outside [0, num_blocks) */
#define MLA_DEV_BAD_LENGTH 2     /* seq_len > max_blocks_per_seq * block_size */
#define MLA_DEV_WAIT_TIMEOUT 3   /* a bounded pipeline wait gave up */

/* Flags of mla_decode_fwd (exactly one of them). */
#define MLA_DECODE_AUTO 0u          /* tensor-core kernel where supported, else SIMT */
#define MLA_DECODE_FORCE_SIMT 1u    /* always the CUDA-core (SIMT) kernel */
/* Diagnostic, for testing the device-side error path: the tensor-core
 * kernel's MMA issuer first waits on a barrier that nothing signals, with a
 * limit of about 1e4 SM clocks.  The wait runs out, the kernel writes
 * MLA_DEV_WAIT_TIMEOUT to *dev_status, every other role of the kernel sees
 * the abort and winds down (in-flight copies are waited for, tensor memory
 * is freed) and the kernel returns; the outputs are left unwritten.  Calls
 * that would run the SIMT kernel return MLA_ERR_ARG with this flag. */
#define MLA_DECODE_TEST_WAIT_TIMEOUT 2u

/*
 * Paged latent cache (iotdigitaltwinplm.com "Interaction with quantisation
 * and paging": a page holds block_size * (d_c + d_r) elements per layer; the
 * latent may be stored in FP8).  Token slot t of physical block p lives at
 *   latent + (p * block_size + t) * latent_stride   (d_c elements)
 *   rope   + (p * block_size + t) * rope_stride     (d_r elements, already rotated)
 * (strides in elements of the respective dtype).  The packed bf16/f32 layout
 * [num_blocks, block_size, d_c + d_r] is latent = pool, rope = pool + d_c,
 * both strides d_c + d_r.  A contiguous per-sequence cache is the paged cache
 * with an identity block table.  For MLA_FP8E4M3 latents, scale[p] is the
 * float32 dequantisation scale of block p (value = e4m3(code) * scale[p]);
 * scale is ignored otherwise and may be NULL.
 */
typedef struct {
  void* latent;
  void* rope;
  float* scale;
  int64_t latent_stride;
  int64_t rope_stride;
  int32_t latent_dtype;   /* mla_dtype */
  int32_t rope_dtype;     /* mla_dtype: F32 or BF16 */
  int32_t num_blocks;
  int32_t block_size;
  int32_t d_c;
  int32_t d_r;
} mla_kv_cache;

/* Text for a status code (static storage). */
const char* mla_status_string(int status);

/* ABI version of this library (major * 100 + minor). */
int mla_version(void);

/*
 * Bytes one cached token occupies per layer (iotdigitaltwinplm.com, "The
 * Cache Arithmetic": MLA stores d_c + d_r elements per token per layer).  The
 * FP8 per-block float32 scale is amortised over block_size tokens.
 * Returns a negative value for an invalid combination.
 */
double mla_cache_bytes_per_token(int latent_dtype, int rope_dtype, int d_c, int d_r,
                                 int block_size);

/*
 * mla_absorb_q: first step of the absorbed decode.
 * kexue.fm section "Part 1" (q k^T = x (W_q W_k^T) c^T) and its note 2 (apply
 * W_k^T to the already projected query, not a merged matrix); section "Part 3",
 * eq. mla-mqa (q = [q_c W_kc^T, q_r R_t]); iotdigitaltwinplm.com, absorbed
 * decode listing (q_lat = q . W_UK per head; RoPE of the rotary query part).
 *
 *   q_cat[b, s, c]       = sum_d q_nope[b, s, d] * w_uk[s, d, c]      c < d_c
 *   q_cat[b, s, d_c + j] = RoPE(q_rope[b, s, :], q_pos[b])[j]           j < d_r
 * RoPE rotates interleaved pairs (2i, 2i+1) by q_pos[b] * theta^(-2i/d_r)
 * (angles formed in float64).  Accumulation is float32.
 *
 *   q_nope [B, h, d_nope], q_rope [B, h, d_r], w_uk [h, d_nope, d_c]: dtype
 *   q_pos  [B] int32 (position of the decoded token)
 *   q_cat  [B, h, d_c + d_r]: dtype (output)
 * dtype is MLA_F32 or MLA_BF16 for all five float tensors.
 * Supported: d_c % 64 == 0, d_c <= 1024, d_r even and <= 256, d_nope <= 512.
 */
int mla_absorb_q(const void* q_nope, const void* q_rope, const int32_t* q_pos,
                 const void* w_uk, void* q_cat, int B, int h, int d_nope, int d_c, int d_r,
                 int dtype, double rope_theta, void* stream);

/* Largest num_parts accepted by mla_decode_fwd / mla_combine. */
#define MLA_MAX_PARTS 1024

/*
 * Work partition shared by mla_decode_fwd and mla_combine (not on the pages:
 * it only decides which key ranges are attended separately; the merge in
 * mla_combine is exact).  The logical blocks of all sequences, in order
 * (sequence 0's ceil(L_0 / block_size) blocks, then sequence 1's, ...), form
 * one stream of T blocks, L_b = seq_lens[b] clamped to
 * [0, max_blocks_per_seq * block_size].  With P = min(num_parts, T), part p
 * covers stream blocks [floor(p T / P), floor((p + 1) T / P)): parts are
 * contiguous, non-empty and balanced to within one block, whatever the
 * length mix.  A part writes one partial result for each sequence b it
 * touches, into partial slot p + b (unique, since parts and sequences are
 * both ordered along the stream).  Slots no part touches are not written.
 *
 * mla_decode_num_partials: number of partial slots, B + num_parts - 1, or a
 * negative mla_status for invalid arguments.
 */
int mla_decode_num_partials(int B, int num_parts);

/*
 * mla_decode_fwd: attention of each sequence's single query token over its
 * cached latent rows (kexue.fm eq. mla-mqa, Attention(q_t, k_<=t, c_<=t);
 * iotdigitaltwinplm.com absorbed decode listing: s = q_lat c^T + q_r k_R^T,
 * softmax(s / sqrt(192)), ctx = p c).  Every cached row 0 .. seq_lens[b]-1 is
 * visible to the query (it sits at the last position).
 *
 * For each part p, each sequence b it touches (rows R = the part's blocks of
 * b, clipped to L_b) and each head s:
 *   o_part[p + b, s, :] = sum_{i in R} p_i c_i / sum_{i in R} p_i
 *   lse_part[p + b, s]  = log(sum_{i in R} exp(score_i))   (natural log)
 * with score_i = softmax_scale * (q_cat[b, s, :] . [c_i, k_R,i]) and
 * p_i = exp(score_i).
 *
 *   q_cat      [B, h, d_c + d_r]: q_dtype (MLA_F32 or MLA_BF16)
 *   kv         cache descriptor (host pointer to the struct; its data pointers
 *              are device pointers)
 *   block_table[B, max_blocks_per_seq] int32: physical block of each logical block
 *   seq_lens   [B] int32, each in [1, max_blocks_per_seq * block_size]; a longer
 *              length is clamped and reported (MLA_DEV_BAD_LENGTH)
 *   num_parts  1 .. MLA_MAX_PARTS; the tensor-core kernel runs one CTA pair per
 *              part (about half the SM count fills the GPU once)
 *   o_part     [mla_decode_num_partials(B, num_parts), h, d_c] float32 (output)
 *   lse_part   [mla_decode_num_partials(B, num_parts), h] float32 (output)
 *   dev_status int32 device word, may be NULL (see conventions)
 *   flags      MLA_DECODE_AUTO, MLA_DECODE_FORCE_SIMT or MLA_DECODE_TEST_WAIT_TIMEOUT
 * Supported dtypes: (q, latent, rope) = (F32, F32, F32) on the SIMT kernel;
 * (BF16, BF16, BF16) and (BF16, FP8E4M3, BF16) on both kernels.  The tensor-core
 * kernel runs for d_c = 512, d_r = 64, block_size = 64, h <= 128; for an FP8
 * latent it dequantises each code to bf16(e4m3 value x block scale) before
 * the MMAs (relative rounding <= 2^-9 per element).  It runs one CTA pair per
 * part and per 128 heads.
 * softmax_scale <= 0 selects 1/sqrt(d_nope + d_r) with d_nope = 128.
 */
int mla_decode_fwd(const void* q_cat, int q_dtype, const mla_kv_cache* kv,
                   const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                   int B, int h, int num_parts, float softmax_scale, float* o_part,
                   float* lse_part, int32_t* dev_status, unsigned flags, void* stream);

/* Largest q_len accepted by mla_decode_fwd_multi. */
#define MLA_MAX_Q_LEN 8

/*
 * mla_decode_fwd_multi: attention of q_len new tokens per sequence (multi-
 * token prediction, or speculative decoding verifying several drafted tokens
 * in one step; iotdigitaltwinplm.com "Interaction with quantisation and
 * paging" and "Arithmetic intensity changes under absorption": more query
 * rows share each latent row read).  The L_b cached rows of sequence b
 * include its q_len new tokens (appended first), so token j sits at position
 * L_b - q_len + j and attends to rows 0 .. L_b - q_len + j (kexue.fm MHA
 * equation: keys i <= t).  The query rows of a sequence are (j, s) at row
 * j * h + s; everything else is as in mla_decode_fwd with h replaced by the
 * q_len * h rows:
 *   q_cat    [B, q_len, h, d_c + d_r] (mla_absorb_q with B * q_len query
 *            rows and one position per token gives it)
 *   o_part   [mla_decode_num_partials(B, num_parts), q_len * h, d_c] float32
 *   lse_part [mla_decode_num_partials(B, num_parts), q_len * h] float32
 * mla_combine with h = q_len * h merges the partials into o_lat
 * [B, q_len, h, d_c].  A token that sees no row (L_b < q_len - j) gets
 * o = 0 and lse = -inf.  Supported: 1 <= q_len <= MLA_MAX_Q_LEN,
 * q_len * h <= 4096.  The tensor-core kernel runs a CTA pair per part and
 * per 128 query rows: give it about (SM count / 2) / ceil(q_len h / 128)
 * parts.
 */
int mla_decode_fwd_multi(const void* q_cat, int q_dtype, const mla_kv_cache* kv,
                         const int32_t* block_table, int max_blocks_per_seq,
                         const int32_t* seq_lens, int B, int q_len, int h, int num_parts,
                         float softmax_scale, float* o_part, float* lse_part,
                         int32_t* dev_status, unsigned flags, void* stream);

/*
 * mla_combine: merge the partials of mla_decode_fwd (log-sum-exp weighting;
 * the pages do not split the key range, this is the exact merge of softmax
 * attention over disjoint key ranges).  For sequence b, with J its partial
 * slots (the parts that touch it, recomputed from seq_lens, block_size,
 * max_blocks_per_seq and num_parts, which must be those of the decode call):
 *   M = max_{j in J} lse_part[j, s];  w_j = exp(lse_part[j, s] - M)
 *   o_lat[b, s, :] = sum_j w_j o_part[j, s, :] / sum_j w_j
 *   lse[b, s]      = M + log(sum_j w_j)
 * A sequence with no rows gets o_lat = 0 and lse = -inf.
 *   o_part, lse_part as written by mla_decode_fwd (float32)
 *   o_lat  [B, h, d_c]: o_dtype (MLA_F32 or MLA_BF16) (output)
 *   lse    [B, h] f32 (output, may be NULL)
 * Supported: d_c % 4 == 0, d_c <= 2048.
 */
int mla_combine(const float* o_part, const float* lse_part, const int32_t* seq_lens,
                int block_size, int max_blocks_per_seq, int B, int h, int d_c, int num_parts,
                void* o_lat, int o_dtype, float* lse, void* stream);

/*
 * mla_decode_attend_noalloc: mla_decode_fwd followed by mla_combine, for
 * callers that cannot allocate device memory (code running under another
 * framework's allocator or memory pool, or a runtime that forbids cudaMalloc
 * on its hot path).  The pages have no counterpart: this is a packaging of
 * the same two calls, not part of the method.
 *
 * The split partials live in a file-scope device array of the library
 * instead of caller buffers; the caller passes only inputs and outputs
 * (arguments as for mla_decode_fwd, then o_lat [B, h, d_c] in o_dtype and
 * lse [B, h] float32 or NULL, as for mla_combine).  Limits: with
 * S = B + num_parts - 1 partial slots, S * h * d_c <= 16 Mi and S * h <= 1 Mi
 * (the array holds 68 MiB on every device that loads the library, until the
 * process exits); larger calls return MLA_ERR_SHAPE and launch nothing.
 * The first call on a device looks up the array's device address with that
 * device current; make it before any stream capture.  The address is kept per
 * device and CUDA context, so a call after a device reset looks it up again
 * (that call, too, belongs outside a stream capture).  All calls share the
 * array: calls that overlap on the GPU race on it.  Nothing in it needs to
 * start at zero (each call writes every slot it reads).  Allocates nothing.
 */
int mla_decode_attend_noalloc(const void* q_cat, int q_dtype, const mla_kv_cache* kv,
                              const int32_t* block_table, int max_blocks_per_seq,
                              const int32_t* seq_lens, int B, int h, int num_parts,
                              float softmax_scale, void* o_lat, int o_dtype, float* lse,
                              int32_t* dev_status, void* stream);

/*
 * mla_out_proj: W_UV applied after attention (kexue.fm section "Part 1": W_v
 * is absorbed into the projection that follows o_t; eq. mla-mqa first line
 * o_t = [o^(1) W_v^(1), ..., o^(h) W_v^(h)]; iotdigitaltwinplm.com absorbed
 * decode listing, out = ctx . W_UV per head):
 *   out[b, s, v] = sum_c o_lat[b, s, c] * w_uv[s, v, c]
 *   o_lat [B, h, d_c]: in_dtype;  w_uv [h, d_v, d_c]: in_dtype
 *   out   [B, h, d_v]: out_dtype (output)
 * in_dtype, out_dtype in {MLA_F32, MLA_BF16}.  Accumulation is float32.
 * Supported: d_c % 64 == 0, d_c <= 1024, d_v <= 1024.
 */
int mla_out_proj(const void* o_lat, const void* w_uv, void* out, int B, int h, int d_c,
                 int d_v, int in_dtype, int out_dtype, void* stream);

/*
 * mla_combine_out_proj: mla_combine followed by mla_out_proj in one call,
 * without the merged rows passing through memory (iotdigitaltwinplm.com, the
 * absorbed decode listing; kexue.fm "From MHA, MQA, GQA to MLA", eq. mla-mqa,
 * first line: the latent output of head s goes through W_v^(s)):
 *   o_lat[b, s, :] = the merge of mla_combine (same arithmetic and slot
 *                    order: equal to mla_combine's output bit for bit)
 *   out[b, s, v]   = sum_c bf16(o_lat[b, s, c]) w_uv[s, v, c]   (float32 accumulation)
 *   o_part, lse_part, seq_lens, block_size, max_blocks_per_seq, num_parts: as
 *                    for mla_combine (those of the decode call)
 *   w_uv [h, d_v, d_c] bf16; out [B, h, d_v] in out_dtype (MLA_F32 or MLA_BF16)
 *   o_lat [B, h, d_c] in o_dtype, or NULL (not written); lse [B, h] or NULL
 *   dev_status: MLA_DEV_WAIT_TIMEOUT is or-ed in if a bounded wait gave up
 *                    (may be NULL)
 * Supported: d_c = 512, d_v = 128, h <= 65535.
 */
int mla_combine_out_proj(const float* o_part, const float* lse_part, const int32_t* seq_lens,
                         int block_size, int max_blocks_per_seq, int B, int h, int d_c,
                         int num_parts, const void* w_uv, int d_v, void* out, int out_dtype,
                         void* o_lat, int o_dtype, float* lse, int32_t* dev_status,
                         void* stream);

/*
 * The hidden-state boundary of the step: the query side starts from the
 * hidden state x_t through the compressed query (kexue.fm "Part 3": the
 * query is also low-rank, c'_t = x_t W_c', and each head's query is read off
 * c'_t; iotdigitaltwinplm.com "Query compression is separate": the query's
 * own down-projection is not cached), and the output side ends in the
 * output projection W_O (kexue.fm "Part 1": W_v can be merged into the
 * projection that follows o_t).  Those are plain linear layers:
 *
 * mla_linear: y[m, n] = sum_k x[m, k] w[n, k]   (w stored [N, K], as a
 * linear layer's weight), bf16 x and w, float32 accumulation, y in y_dtype
 * (MLA_F32 or MLA_BF16).  Supported: K % 64 == 0, N % 128 == 0.  Long
 * contractions are split over CTAs; the float32 split partials go to the
 * caller's workspace of mla_linear_workspace_bytes(M, K, N) bytes (0: none
 * needed; then workspace may be NULL) and are summed in a fixed order, so
 * results do not depend on timing.  A too small workspace is MLA_ERR_ARG.
 */
size_t mla_linear_workspace_bytes(int M, int K, int N);
int mla_linear(const void* x, const void* w, void* y, int M, int K, int N, int y_dtype,
               void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_fold_uv_into_o: merge W_UV into the output projection (kexue.fm "Part
 * 1": the value up-projection moves into the projection after attention):
 *   w_fold[n, s, c] = sum_v w_o[n, s * d_v + v] * w_uv[s, v, c]
 *   w_uv [h, d_v, d_c], w_o [d_model, h * d_v], w_fold [d_model, h * d_c]: bf16
 * so that y = o_lat . w_fold^T (mla_linear over the h * d_c latent outputs)
 * equals (o_lat W_UV) W_O^T.  Supported: d_c = 512, d_v = 128.  The merged
 * matrix holds d_c / d_v = 4 times the elements of W_O, so at decode, where
 * weight reads bound these layers, the unmerged pair reads fewer bytes.
 */
int mla_fold_uv_into_o(const void* w_uv, const void* w_o, void* w_fold, int h, int d_c, int d_v,
                       int d_model, void* stream);

/*
 * Prefill in the MHA form (kexue.fm "Part 3", eq. mla-mha, the form used for
 * training and prefill; iotdigitaltwinplm.com "Prefill versus decode": the
 * prompt's per-head keys and values are formed once and attention is
 * compute-bound).  For every head s the key of token i is
 * [c_i W_UK^(s), RoPE(k_R,i, i)] (192 values) and its value c_i W_UV^(s)
 * (128 values); token t of a sequence attends to its tokens i <= t with
 * the query [q_nope,t, RoPE(q_R,t, t)] and the scale 1/sqrt(192).  The
 * sequences are packed: sequence b's tokens are rows cu_seqlens[b] ..
 * cu_seqlens[b+1] - 1 (device int32 array of B + 1 entries), positions
 * 0 .. L_b - 1, T = cu_seqlens[B] = total_rows rows in all.
 *
 * mla_prefill_query: q[t, s, 0:128] = q_nope[t, s, :] and
 *   q[t, s, 128 + j] = RoPE(q_rope[t, s, :], position of t)[j] (angles in
 *   float64, as mla_absorb_q).  q_nope [T, h, 128], q_rope [T, h, 64],
 *   q [T, h, 192]: bf16.
 * mla_prefill_fwd: out[t, s, :] = sum_{i <= t} p_ti v_i^(s), p the causal
 *   softmax of the scores, lse[t, s] its natural-log denominator (lse may be
 *   NULL).  q [T, h, 192] (from mla_prefill_query), k_nope [T, h, 128]
 *   (= c W_UK^T: mla_linear of c with W_UK viewed [h * 128, 512]),
 *   k_rope [T, 64] (the rotated RoPE key, shared by the heads: the cache's
 *   rope rows), v [T, h, 128] (= c W_UV^T), all bf16; out [T, h, 128] in
 *   out_dtype (MLA_F32 or MLA_BF16).  softmax_scale <= 0 selects 1/sqrt(192).
 *   max_len bounds every L_b (it sizes the launch).
 */
int mla_prefill_query(const void* q_nope, const void* q_rope, const int32_t* cu_seqlens, int B,
                      int max_len, int h, double rope_theta, void* q, void* stream);
int mla_prefill_fwd(const void* q, const void* k_nope, const void* k_rope, const void* v,
                    const int32_t* cu_seqlens, int B, int max_len, int64_t total_rows, int h,
                    float softmax_scale, void* out, int out_dtype, float* lse,
                    int32_t* dev_status, void* stream);

/*
 * mla_cache_fill: write whole sequences into the paged cache (the cache
 * content of iotdigitaltwinplm.com's listing, appended rows c_t and
 * RoPE(k_R, t); intvml.com: the RoPE key is cached in rotated form).
 * Row t of sequence b (source row cu_seqlens[b] + t, 0 <= t < L_b with
 * L_b = cu_seqlens[b+1] - cu_seqlens[b]) goes to physical block
 * block_table[b, t / block_size], slot t % block_size:
 *   latent row = c_kv row            (F32/BF16 cache: copied; FP8 cache: see below)
 *   rope row   = RoPE(k_rope row, t) (angles t * theta^(-2i/d_r) in float64,
 *                                     rotation in float32, stored in rope dtype)
 * FP8 latent: per physical block, amax over the block's written rows and all
 * d_c columns; scale = amax / 448 (float32 division; 1 if amax == 0);
 * code = e4m3(c / scale) with the correctly rounded float32 quotient, rounding
 * to nearest even and saturating to +-448; scale[p] is written.  Slots past
 * L_b in a sequence's last block are not written.
 *   c_kv [T, d_c]: src_dtype (MLA_F32, or MLA_BF16 for BF16/FP8 caches)
 *   k_rope [T, d_r]: the cache's rope dtype
 *   cu_seqlens [B + 1] int32 device array, T = cu_seqlens[B]
 *   max_len: an upper bound of every L_b (sizes the launch)
 * Block-table entries outside the pool are skipped and reported in *dev_status.
 */
int mla_cache_fill(const void* c_kv, const void* k_rope, int src_dtype,
                   const int32_t* cu_seqlens, int B, int max_len, const int32_t* block_table,
                   int max_blocks_per_seq, const mla_kv_cache* kv, double rope_theta,
                   int32_t* dev_status, void* stream);

/*
 * mla_cache_append: the per-step cache write of decoding - one new token per
 * sequence (iotdigitaltwinplm.com, the absorbed-decode listing in "A latent
 * KV projection in PyTorch": the new c and rotated k_R are appended before
 * attention; "Interaction with quantisation and paging": paged blocks, FP8
 * latent; intvml.com "DL0107 MLA": the RoPE key is cached in rotated form).
 * For sequence b, with t = pos[b] (the token's position = the sequence's
 * length before the append; the caller raises seq_lens afterwards), the row
 * goes to physical block block_table[b, t / block_size], slot t % block_size:
 *   latent row = c_new[b]                 (F32/BF16 cache: copied)
 *   rope row   = RoPE(k_rope_new[b], t)   (as in mla_cache_fill)
 * FP8 latent (the cache keeps only codes and one float32 scale per block):
 *   - slot 0 (an empty block): scale = amax(row) / 448 (1 if 0), code =
 *     e4m3(c / scale), as mla_cache_fill quantises a one-row block;
 *   - otherwise, with a = amax(row) and s = scale[p]: if a <= 448 s (float32
 *     product) the scale stays and code = e4m3(c / s); else the scale grows to
 *     s' = a / 448, every earlier code of the block becomes
 *     e4m3((e4m3(code) * s) / s') (float32 steps) and code = e4m3(c / s').
 *   Rounding is to nearest even, saturating to +-448, as in mla_cache_fill.
 *   c_new [B, d_c]: src_dtype (MLA_F32, or MLA_BF16 for BF16/FP8 caches)
 *   k_rope_new [B, d_r]: the cache's rope dtype, unrotated
 *   pos [B] int32 device array; block_table [B, max_blocks_per_seq] int32
 * A position outside [0, max_blocks_per_seq * block_size) or a block-table
 * entry outside the pool is skipped and reported in *dev_status.  Sequences
 * must not share physical blocks (CTA b owns its block for the call).
 */
int mla_cache_append(const void* c_new, const void* k_rope_new, int src_dtype,
                     const int32_t* pos, int B, const int32_t* block_table,
                     int max_blocks_per_seq, const mla_kv_cache* kv, double rope_theta,
                     int32_t* dev_status, void* stream);

/*
 * mla_paged_gather: copy each sequence's logical rows out of the pool, bit for
 * bit (latent in its stored dtype - e4m3 codes for FP8 - and the rotated rope).
 *   latent_out [T, d_c], rope_out [T, d_r] (T = cu_seqlens[B]); either may be NULL.
 */
int mla_paged_gather(const mla_kv_cache* kv, const int32_t* block_table,
                     int max_blocks_per_seq, const int32_t* cu_seqlens, int B, int max_len,
                     void* latent_out, void* rope_out, int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA72_H */
