// Shared device helpers and internal launcher declarations of the MLA library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/mla72.h"

namespace mla {

// ---------------------------------------------------------------------------
// element access
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// e4m3 code -> float (exact)
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  __nv_fp8_e4m3 v;
  v.__x = c;
  return static_cast<float>(v);
}

// float -> e4m3 code, round to nearest even, saturate to +-448
__device__ __forceinline__ uint8_t f32_to_e4m3_rn_sat(float f) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(f, __NV_SATFINITE, __NV_E4M3));
}

// Load element i of an array of the given dtype as float.
__device__ __forceinline__ float load_as_f32(const void* p, int dtype, int64_t i) {
  if (dtype == MLA_F32) return static_cast<const float*>(p)[i];
  if (dtype == MLA_BF16) return bf16_to_f32(static_cast<const uint16_t*>(p)[i]);
  return e4m3_to_f32(static_cast<const uint8_t*>(p)[i]);
}

__device__ __forceinline__ void store_from_f32(void* p, int dtype, int64_t i, float v) {
  if (dtype == MLA_F32) {
    static_cast<float*>(p)[i] = v;
  } else {
    static_cast<uint16_t*>(p)[i] = f32_to_bf16_rn(v);
  }
}

__device__ __forceinline__ void set_status(int32_t* st, int code) {
  if (st) atomicCAS(st, 0, code);
}

__host__ __device__ __forceinline__ int dtype_bytes(int dt) {
  return dt == MLA_F32 ? 4 : (dt == MLA_BF16 ? 2 : 1);
}

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// RoPE angles (iotdigitaltwinplm.com "MLA vs GQA vs MQA", the rope helper of
// the listing: pair i of a d_r-vector at position pos is rotated by
// pos * theta^(-2i/d_r))
// ---------------------------------------------------------------------------

// cos and sin of pos * inv_freq: the angle is formed and reduced modulo 2 pi in
// float64 (positions reach 1e5 rad, where a float32 angle would be off by
// ~1e-2), and the reduced angle (|r| <= pi) goes through float32 sincosf.
__device__ __forceinline__ void rope_cos_sin(double pos, double inv_freq, float* c, float* s) {
  const double two_pi = 6.283185307179586;
  const double inv_two_pi = 0.15915494309189535;
  const double ang = pos * inv_freq;
  const double k = rint(ang * inv_two_pi);   // off by one at worst: |r| stays < pi + 1e-9
  const float r = (float)fma(-k, two_pi, ang);
  sincosf(r, s, c);
}

// The same in float32 for an integer position 0 <= pos < 2^24, with the angle
// measured in turns: pos * inv_freq / (2 pi) = pos * (f_hi + f_lo), f_hi and
// f_lo the float32 head and tail of inv_freq / (2 pi) (formed in float64 on
// the host).  Whole turns are removed exactly (Cody and Waite's additive
// reduction, with the product kept exact inside the FMA): n is within one of
// pos * f_hi, so |pos * f_hi - n| < 1 is rounded once (<= 2^-25 turns); the
// tail adds pos * f_lo (< 1/8) with one more such rounding.  The angle error
// is below 2 pi * 2^-23 turns ~ 7.5e-7 rad, then sincospif(2 t).
__device__ __forceinline__ void rope_cos_sin_turns(int pos, float f_hi, float f_lo, float* c,
                                                   float* s) {
  const float p = (float)pos;
  const float n = rintf(p * f_hi);
  float t = fmaf(p, f_hi, -n);
  t = fmaf(p, f_lo, t);
  sincospif(2.0f * t, s, c);
}

// ---------------------------------------------------------------------------
// work partition of the decode (shared by the decode kernels and the combine)
// ---------------------------------------------------------------------------
//
// The logical blocks of all sequences, in order (sequence 0's blocks, then
// sequence 1's, ...), form one stream of T blocks.  With P = min(num_parts, T)
// effective parts, part p covers stream blocks [floor(p T / P), floor((p+1) T / P));
// every part is non-empty.  A part writes one partial result (o, lse) per
// sequence it touches, into slot p + b; slots are unique because parts and
// sequences are both ordered along the stream.

// Blocks of sequence b (its length clamped to [0, max_blocks * bs]).
__device__ __forceinline__ int seq_blocks(const int32_t* lens, int b, int bs, int max_blocks) {
  int L = lens[b];
  L = L < 0 ? 0 : (L > max_blocks * bs ? max_blocks * bs : L);
  return (L + bs - 1) / bs;
}

__host__ __device__ __forceinline__ long long part_begin(long long T, int P, int p) {
  return (long long)p * T / P;
}

// The part holding stream block g (largest p with part_begin(p) <= g).
__host__ __device__ __forceinline__ int part_of(long long T, int P, long long g) {
  return (int)(((g + 1) * (long long)P - 1) / T);
}

// Warp-cooperative scan over the sequence lengths (all 32 lanes call it with the
// same arguments).  Returns T; *s_qb = stream index of block 0 of sequence qb
// (if 0 <= qb < B); *b_qg / *s_bqg = the sequence holding stream block qg and
// its first stream block (if 0 <= qg < T; *b_qg = -1 otherwise).
__device__ __forceinline__ long long warp_stream_scan(const int32_t* lens, int B, int bs,
                                                     int max_blocks, int qb, long long qg,
                                                     long long* s_qb, int* b_qg,
                                                     long long* s_bqg) {
  const int lane = threadIdx.x & 31;
  long long run = 0, sq = 0, sg = 0;
  int bg = -1;
  for (int base = 0; base < B; base += 32) {
    const int b = base + lane;
    const int n = b < B ? seq_blocks(lens, b, bs, max_blocks) : 0;
    int inc = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += v;
    }
    const long long excl = run + inc - n;
    if (qb >= base && qb < base + 32) sq = __shfl_sync(0xffffffffu, excl, qb - base);
    const unsigned own = __ballot_sync(0xffffffffu, n > 0 && qg >= excl && qg < excl + n);
    if (own != 0u && bg < 0) {
      const int src = __ffs(own) - 1;
      bg = base + src;
      sg = __shfl_sync(0xffffffffu, excl, src);
    }
    run += __shfl_sync(0xffffffffu, inc, 31);
  }
  if (s_qb) *s_qb = sq;
  if (b_qg) *b_qg = bg;
  if (s_bqg) *s_bqg = sg;
  return run;
}

// ---------------------------------------------------------------------------
// internal launchers (one per kernel family); each returns cudaError_t
// ---------------------------------------------------------------------------

cudaError_t launch_absorb_q_simt(const void* q_nope, const void* q_rope, const int32_t* q_pos,
                                 const void* w_uk, void* q_cat, int B, int h, int d_nope,
                                 int d_c, int d_r, int dtype, double theta, cudaStream_t s);

// q_len query tokens per sequence, heads heads each: q_len * heads query rows
cudaError_t launch_decode_simt(const void* q_cat, int q_dtype, const mla_kv_cache& kv,
                               const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                               int B, int q_len, int heads, int num_parts, float scale,
                               float* o_part, float* lse_part, int32_t* status, cudaStream_t s);

bool decode_tc_supported(int q_dtype, const mla_kv_cache& kv, int rows);

// True on an sm_100-family device with the tensor-map encoder available.
bool tc_device();

cudaError_t launch_absorb_q_tc(const void* q_nope, const void* q_rope, const int32_t* q_pos,
                               const void* w_uk, void* q_cat, int B, int h, double theta,
                               cudaStream_t s);

cudaError_t launch_out_proj_tc(const void* o_lat, const void* w_uv, void* out, int B, int h,
                               int out_dtype, cudaStream_t s);

// y[M, N] = x[M, K] W[N, K]^T (bf16 in, y_dtype out); part: float32 split
// partials of linear_splits(M, K, N) * M * N floats when that is above 1
int linear_splits(int M, int K, int N);
cudaError_t launch_linear_tc(const void* x, const void* w, void* y, int M, int K, int N,
                             int y_dtype, float* part, cudaStream_t s);
// W_fold[n, s, c] = sum_v W_O[n, s * 128 + v] W_UV[s, v, c] (bf16)
cudaError_t launch_fold_uv_o_tc(const void* w_uv, const void* w_o, void* w_fold, int h,
                                int d_model, cudaStream_t s);

// causal prefill attention in the MHA form (d_qk = 192, d_v = 128), bf16
cudaError_t launch_prefill_tc(const void* q, const void* k_nope, const void* k_rope,
                              const void* v, const int32_t* cu_seqlens, int B, int max_len,
                              int h, int64_t total_rows, float scale, void* out, int out_dtype,
                              float* lse, int32_t* status, cudaStream_t s);
cudaError_t launch_prefill_query(const void* q_nope, const void* q_rope, const int32_t* cu_seqlens,
                                 int B, int max_len, int h, double theta, void* q, cudaStream_t s);

cudaError_t launch_decode_tc(const void* q_cat, const mla_kv_cache& kv,
                             const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                             int B, int q_len, int heads, int num_parts, float scale,
                             float* o_part, float* lse_part, int32_t* status, bool test_timeout,
                             cudaStream_t s);

cudaError_t launch_combine(const float* o_part, const float* lse_part, const int32_t* seq_lens,
                           int block_size, int max_blocks, int B, int h, int d_c, int num_parts,
                           void* o_lat, int o_dtype, float* lse, cudaStream_t s);

cudaError_t launch_out_proj_simt(const void* o_lat, const void* w_uv, void* out, int B, int h,
                                 int d_c, int d_v, int in_dtype, int out_dtype, cudaStream_t s);

cudaError_t launch_cache_fill(const void* c_kv, const void* k_rope, int src_dtype,
                              const int32_t* cu_seqlens, int B, int max_len,
                              const int32_t* block_table, int max_blocks,
                              const mla_kv_cache& kv, double theta, int32_t* status,
                              cudaStream_t s);

cudaError_t launch_cache_append(const void* c_new, const void* k_rope, int src_dtype,
                                const int32_t* pos, int B, const int32_t* block_table,
                                int max_blocks, const mla_kv_cache& kv, double theta,
                                int32_t* status, cudaStream_t s);

cudaError_t launch_paged_gather(const mla_kv_cache& kv, const int32_t* block_table,
                                int max_blocks, const int32_t* cu_seqlens, int B, int max_len,
                                void* latent_out, void* rope_out, int32_t* status,
                                cudaStream_t s);

// ---------------------------------------------------------------------------
// launches of the decode step's kernels: programmatic stream serialization, so
// that a kernel's CTAs are scheduled while the previous kernel of the stream
// finishes (each of these kernels calls grid_dep_wait before it reads memory
// an earlier kernel may write, and grid_dep_launch at its start)
// ---------------------------------------------------------------------------
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace mla
