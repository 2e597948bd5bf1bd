// mla_absorb_q: fold W_UK into the query and rotate the RoPE query part.
//
// kexue.fm "From MHA, MQA, GQA to MLA", section "Part 1" (note 2: the query
// is formed as (x W_q) W_k^T, sequentially) and eq. mla-mqa (first block of
// q: c' W_qc W_kc^T, second block: RoPE of the rotary part).
#include "common.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kBatchTile = 16;   // query rows per CTA
constexpr int kMaxColsPerThread = 4;  // d_c <= 1024

// grid: (h, ceil(B / kBatchTile)); block: 256 threads.
// Thread t accumulates latent columns t, t + 256, ... for kBatchTile queries of one head.
__global__ void __launch_bounds__(kThreads)
absorb_q_simt_kernel(const void* __restrict__ q_nope, const void* __restrict__ q_rope,
                     const int32_t* __restrict__ q_pos, const void* __restrict__ w_uk,
                     void* __restrict__ q_cat, int B, int h, int d_nope, int d_c, int d_r,
                     int dtype, double theta) {
  extern __shared__ float sq[];  // [kBatchTile][d_nope]
  const int s = blockIdx.x;
  const int b0 = blockIdx.y * kBatchTile;
  const int nb = min(kBatchTile, B - b0);
  const int dqk = d_c + d_r;

  for (int i = threadIdx.x; i < kBatchTile * d_nope; i += kThreads) {
    int bb = i / d_nope, d = i % d_nope;
    sq[i] = bb < nb ? load_as_f32(q_nope, dtype, ((int64_t)(b0 + bb) * h + s) * d_nope + d) : 0.f;
  }
  __syncthreads();

  float acc[kBatchTile][kMaxColsPerThread];
#pragma unroll
  for (int bb = 0; bb < kBatchTile; ++bb)
#pragma unroll
    for (int k = 0; k < kMaxColsPerThread; ++k) acc[bb][k] = 0.f;

  const int64_t wbase = (int64_t)s * d_nope * d_c;
  for (int d = 0; d < d_nope; ++d) {
    float w[kMaxColsPerThread];
#pragma unroll
    for (int k = 0; k < kMaxColsPerThread; ++k) {
      int c = threadIdx.x + k * kThreads;
      w[k] = c < d_c ? load_as_f32(w_uk, dtype, wbase + (int64_t)d * d_c + c) : 0.f;
    }
#pragma unroll
    for (int bb = 0; bb < kBatchTile; ++bb) {
      float q = sq[bb * d_nope + d];
#pragma unroll
      for (int k = 0; k < kMaxColsPerThread; ++k) acc[bb][k] = fmaf(q, w[k], acc[bb][k]);
    }
  }
#pragma unroll
  for (int bb = 0; bb < kBatchTile; ++bb) {
    if (bb >= nb) break;
    int64_t obase = ((int64_t)(b0 + bb) * h + s) * dqk;
#pragma unroll
    for (int k = 0; k < kMaxColsPerThread; ++k) {
      int c = threadIdx.x + k * kThreads;
      if (c < d_c) store_from_f32(q_cat, dtype, obase + c, acc[bb][k]);
    }
  }

  // RoPE of the rotary query part: pair i of row (b, s) rotated by q_pos[b] * theta^(-2i/d_r).
  const int half = d_r / 2;
  __shared__ double inv_freq[128];
  for (int i = threadIdx.x; i < half; i += kThreads) inv_freq[i] = pow(theta, -2.0 * (double)i / (double)d_r);
  __syncthreads();
  for (int i = threadIdx.x; i < nb * half; i += kThreads) {
    int bb = i / half, p = i % half;
    int b = b0 + bb;
    float cs, sn;
    rope_cos_sin((double)q_pos[b], inv_freq[p], &cs, &sn);
    int64_t ib = ((int64_t)b * h + s) * d_r;
    float x0 = load_as_f32(q_rope, dtype, ib + 2 * p);
    float x1 = load_as_f32(q_rope, dtype, ib + 2 * p + 1);
    int64_t obase = ((int64_t)b * h + s) * dqk + d_c;
    store_from_f32(q_cat, dtype, obase + 2 * p, x0 * cs - x1 * sn);
    store_from_f32(q_cat, dtype, obase + 2 * p + 1, x0 * sn + x1 * cs);
  }
}

}  // namespace

cudaError_t launch_absorb_q_simt(const void* q_nope, const void* q_rope, const int32_t* q_pos,
                                 const void* w_uk, void* q_cat, int B, int h, int d_nope,
                                 int d_c, int d_r, int dtype, double theta, cudaStream_t s) {
  dim3 grid(h, ceil_div(B, kBatchTile));
  size_t smem = sizeof(float) * kBatchTile * d_nope;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(absorb_q_simt_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  absorb_q_simt_kernel<<<grid, kThreads, smem, s>>>(q_nope, q_rope, q_pos, w_uk, q_cat, B, h,
                                                    d_nope, d_c, d_r, dtype, theta);
  return cudaGetLastError();
}

}  // namespace mla
