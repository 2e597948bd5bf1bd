// Paged latent cache: fill (rows -> blocks, RoPE of the key, optional FP8
// quantisation per block), the per-step append of one token per sequence,
// and the bit-exact logical gather.
//
// The cache holds, per token, the latent c_i and the shared RoPE key already
// rotated to the token's position (intvml.com "DL0107 Multi-head Latent
// Attention MLA": the 64-d positional key is cached in rotated form;
// iotdigitaltwinplm.com "MLA vs GQA vs MQA", section "Interaction with
// quantisation and paging": pages of block_size * 576 elements, FP8 latent).
#include <math.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;

// inverse frequencies theta^(-2i/d_r), formed on the host in float64 (the
// FP64 pipe of this GPU is slow; one launch needs them once)
struct InvFreq {
  double v[128];
};


// grid: (ceil(max_len / block_size), B); block: 256 threads.  One CTA writes
// one logical block of one sequence.
__global__ void __launch_bounds__(kThreads)
cache_fill_kernel(const void* __restrict__ c_kv, const void* __restrict__ k_rope, int src_dtype,
                  const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ block_table,
                  int max_blocks, mla_kv_cache kv, const __grid_constant__ InvFreq inv_freq,
                  int32_t* status) {
  const int jb = blockIdx.x, b = blockIdx.y;
  const int bs = kv.block_size;
  const int row0 = cu_seqlens[b];
  const int L = cu_seqlens[b + 1] - row0;
  const int t0 = jb * bs;
  if (t0 >= L) return;
  if (jb >= max_blocks) {
    if (threadIdx.x == 0) set_status(status, MLA_DEV_BAD_LENGTH);
    return;
  }
  const int n = min(bs, L - t0);
  const int pb = block_table[(int64_t)b * max_blocks + jb];
  if (pb < 0 || pb >= kv.num_blocks) {
    if (threadIdx.x == 0) set_status(status, MLA_DEV_BAD_BLOCK);
    return;
  }
  const int d_c = kv.d_c, d_r = kv.d_r;
  const int64_t src0 = (int64_t)row0 + t0;     // first source row of this block
  const int64_t dst0 = (int64_t)pb * bs;       // first slot row of this block

  if (kv.latent_dtype == MLA_FP8E4M3) {
    __shared__ float red[kThreads / 32];
    __shared__ float s_scale;
    float amax = 0.f;
    for (int i = threadIdx.x; i < n * d_c; i += kThreads)
      amax = fmaxf(amax, fabsf(load_as_f32(c_kv, src_dtype, src0 * d_c + i)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
      float a = red[0];
      for (int w = 1; w < kThreads / 32; ++w) a = fmaxf(a, red[w]);
      float sc = a > 0.f ? __fdiv_rn(a, 448.0f) : 1.0f;
      s_scale = sc;
      kv.scale[pb] = sc;
    }
    __syncthreads();
    const float sc = s_scale;
    uint8_t* lat = static_cast<uint8_t*>(kv.latent);
    for (int i = threadIdx.x; i < n * d_c; i += kThreads) {
      int r = i / d_c, c = i % d_c;
      float x = load_as_f32(c_kv, src_dtype, src0 * d_c + i);
      lat[(dst0 + r) * kv.latent_stride + c] = f32_to_e4m3_rn_sat(__fdiv_rn(x, sc));
    }
  } else {
    for (int i = threadIdx.x; i < n * d_c; i += kThreads) {
      int r = i / d_c, c = i % d_c;
      float x = load_as_f32(c_kv, src_dtype, src0 * d_c + i);
      store_from_f32(kv.latent, kv.latent_dtype, (dst0 + r) * kv.latent_stride + c, x);
    }
  }

  // RoPE of the key at its position t: pair p rotated by t * theta^(-2p/d_r)
  const int half = d_r / 2;
  for (int i = threadIdx.x; i < n * half; i += kThreads) {
    int r = i / half, p = i % half;
    int t = t0 + r;
    float cs, sn;
    rope_cos_sin((double)t, inv_freq.v[p], &cs, &sn);
    float x0 = load_as_f32(k_rope, kv.rope_dtype, (src0 + r) * d_r + 2 * p);
    float x1 = load_as_f32(k_rope, kv.rope_dtype, (src0 + r) * d_r + 2 * p + 1);
    int64_t o = (dst0 + r) * kv.rope_stride + 2 * p;
    store_from_f32(kv.rope, kv.rope_dtype, o, x0 * cs - x1 * sn);
    store_from_f32(kv.rope, kv.rope_dtype, o + 1, x0 * sn + x1 * cs);
  }
}

// Block-wide maximum of v over the CTA (every thread gets it).
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  __syncthreads();  // red may still be read from a previous call
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = v;
  __syncthreads();
  float a = red[0];
  for (int w = 1; w < kThreads / 32; ++w) a = fmaxf(a, red[w]);
  return a;
}

// grid: B; block: 256 threads.  CTA b appends one token to sequence b: the
// latent row c_new[b] at logical slot t = pos[b] (physical block
// block_table[b, t / block_size], slot t % block_size) and the RoPE key row
// rotated to position t.  For an FP8 latent the block's scale grows when the
// new row does not fit it; the block's earlier codes are then re-quantised
// from their dequantised values.
__global__ void __launch_bounds__(kThreads)
cache_append_kernel(const void* __restrict__ c_new, const void* __restrict__ k_rope,
                    int src_dtype, const int32_t* __restrict__ pos,
                    const int32_t* __restrict__ block_table, int max_blocks, mla_kv_cache kv,
                    const __grid_constant__ InvFreq inv_freq, int32_t* status) {
  __shared__ float red[kThreads / 32];
  const int b = blockIdx.x;
  const int bs = kv.block_size;
  const int t = pos[b];
  if (t < 0 || t >= max_blocks * bs) {
    if (threadIdx.x == 0) set_status(status, MLA_DEV_BAD_LENGTH);
    return;
  }
  const int pb = block_table[(int64_t)b * max_blocks + t / bs];
  if (pb < 0 || pb >= kv.num_blocks) {
    if (threadIdx.x == 0) set_status(status, MLA_DEV_BAD_BLOCK);
    return;
  }
  const int d_c = kv.d_c, d_r = kv.d_r;
  const int slot = t % bs;
  const int64_t row0 = (int64_t)pb * bs;          // slot 0 of the block
  const int64_t src = (int64_t)b * d_c;

  if (kv.latent_dtype == MLA_FP8E4M3) {
    uint8_t* lat = static_cast<uint8_t*>(kv.latent);
    float amax = 0.f;
    for (int i = threadIdx.x; i < d_c; i += kThreads)
      amax = fmaxf(amax, fabsf(load_as_f32(c_new, src_dtype, src + i)));
    amax = block_max(amax, red);
    float sc;
    if (slot == 0) {
      // an empty block: its scale comes from this row alone
      sc = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    } else {
      const float s_old = kv.scale[pb];
      sc = s_old;
      if (amax > __fmul_rn(448.0f, s_old)) {
        // the row does not fit: grow the scale and re-quantise the block's
        // earlier rows from their dequantised values
        sc = __fdiv_rn(amax, 448.0f);
        for (int i = threadIdx.x; i < slot * d_c; i += kThreads) {
          const int r = i / d_c, c = i % d_c;
          uint8_t* q = lat + (row0 + r) * kv.latent_stride + c;
          const float deq = __fmul_rn(e4m3_to_f32(*q), s_old);
          *q = f32_to_e4m3_rn_sat(__fdiv_rn(deq, sc));
        }
      }
    }
    for (int i = threadIdx.x; i < d_c; i += kThreads)
      lat[(row0 + slot) * kv.latent_stride + i] =
          f32_to_e4m3_rn_sat(__fdiv_rn(load_as_f32(c_new, src_dtype, src + i), sc));
    __syncthreads();  // every thread has read the old scale
    if (threadIdx.x == 0) kv.scale[pb] = sc;
  } else {
    for (int i = threadIdx.x; i < d_c; i += kThreads)
      store_from_f32(kv.latent, kv.latent_dtype, (row0 + slot) * kv.latent_stride + i,
                     load_as_f32(c_new, src_dtype, src + i));
  }

  // RoPE of the key at position t (the same arithmetic as the fill kernel)
  const int half = d_r / 2;
  for (int p = threadIdx.x; p < half; p += kThreads) {
    float cs, sn;
    rope_cos_sin((double)t, inv_freq.v[p], &cs, &sn);
    const float x0 = load_as_f32(k_rope, kv.rope_dtype, (int64_t)b * d_r + 2 * p);
    const float x1 = load_as_f32(k_rope, kv.rope_dtype, (int64_t)b * d_r + 2 * p + 1);
    const int64_t o = (row0 + slot) * kv.rope_stride + 2 * p;
    store_from_f32(kv.rope, kv.rope_dtype, o, x0 * cs - x1 * sn);
    store_from_f32(kv.rope, kv.rope_dtype, o + 1, x0 * sn + x1 * cs);
  }
}

// grid: (ceil(max_len / block_size), B); block: 256.  Byte copy of logical rows.
__global__ void __launch_bounds__(kThreads)
paged_gather_kernel(mla_kv_cache kv, const int32_t* __restrict__ block_table, int max_blocks,
                    const int32_t* __restrict__ cu_seqlens, void* latent_out, void* rope_out,
                    int32_t* status) {
  const int jb = blockIdx.x, b = blockIdx.y;
  const int bs = kv.block_size;
  const int row0 = cu_seqlens[b];
  const int L = cu_seqlens[b + 1] - row0;
  const int t0 = jb * bs;
  if (t0 >= L) return;
  if (jb >= max_blocks) {
    if (threadIdx.x == 0) set_status(status, MLA_DEV_BAD_LENGTH);
    return;
  }
  const int n = min(bs, L - t0);
  const int pb = block_table[(int64_t)b * max_blocks + jb];
  if (pb < 0 || pb >= kv.num_blocks) {
    if (threadIdx.x == 0) set_status(status, MLA_DEV_BAD_BLOCK);
    return;
  }
  const int lb = dtype_bytes(kv.latent_dtype), rb = dtype_bytes(kv.rope_dtype);
  const int64_t dst0 = (int64_t)row0 + t0, src0 = (int64_t)pb * bs;
  if (latent_out) {
    const int row_bytes = kv.d_c * lb;
    const uint8_t* src = static_cast<const uint8_t*>(kv.latent);
    uint8_t* dst = static_cast<uint8_t*>(latent_out);
    for (int i = threadIdx.x; i < n * row_bytes; i += kThreads) {
      int r = i / row_bytes, k = i % row_bytes;
      dst[(dst0 + r) * row_bytes + k] = src[(src0 + r) * kv.latent_stride * lb + k];
    }
  }
  if (rope_out) {
    const int row_bytes = kv.d_r * rb;
    const uint8_t* src = static_cast<const uint8_t*>(kv.rope);
    uint8_t* dst = static_cast<uint8_t*>(rope_out);
    for (int i = threadIdx.x; i < n * row_bytes; i += kThreads) {
      int r = i / row_bytes, k = i % row_bytes;
      dst[(dst0 + r) * row_bytes + k] = src[(src0 + r) * kv.rope_stride * rb + k];
    }
  }
}

InvFreq inv_freq(int d_r, double theta) {
  InvFreq f{};
  for (int i = 0; i < d_r / 2; ++i) f.v[i] = pow(theta, -2.0 * (double)i / (double)d_r);
  return f;
}

}  // namespace

cudaError_t launch_cache_fill(const void* c_kv, const void* k_rope, int src_dtype,
                              const int32_t* cu_seqlens, int B, int max_len,
                              const int32_t* block_table, int max_blocks,
                              const mla_kv_cache& kv, double theta, int32_t* status,
                              cudaStream_t s) {
  dim3 grid(ceil_div(max_len, kv.block_size), B);
  if (grid.x == 0) return cudaSuccess;
  cache_fill_kernel<<<grid, kThreads, 0, s>>>(c_kv, k_rope, src_dtype, cu_seqlens, block_table,
                                              max_blocks, kv, inv_freq(kv.d_r, theta), status);
  return cudaGetLastError();
}

cudaError_t launch_cache_append(const void* c_new, const void* k_rope, int src_dtype,
                                const int32_t* pos, int B, const int32_t* block_table,
                                int max_blocks, const mla_kv_cache& kv, double theta,
                                int32_t* status, cudaStream_t s) {
  cache_append_kernel<<<B, kThreads, 0, s>>>(c_new, k_rope, src_dtype, pos, block_table,
                                             max_blocks, kv, inv_freq(kv.d_r, theta), status);
  return cudaGetLastError();
}

cudaError_t launch_paged_gather(const mla_kv_cache& kv, const int32_t* block_table,
                                int max_blocks, const int32_t* cu_seqlens, int B, int max_len,
                                void* latent_out, void* rope_out, int32_t* status,
                                cudaStream_t s) {
  dim3 grid(ceil_div(max_len, kv.block_size), B);
  if (grid.x == 0) return cudaSuccess;
  paged_gather_kernel<<<grid, kThreads, 0, s>>>(kv, block_table, max_blocks, cu_seqlens,
                                                latent_out, rope_out, status);
  return cudaGetLastError();
}

}  // namespace mla
