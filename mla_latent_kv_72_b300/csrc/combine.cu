// mla_combine: log-sum-exp merge of the split-KV partials.
//
// Exact merge of softmax attention computed over disjoint key ranges: each
// range's normalised output is weighted by exp(lse_j - max_j lse_j).  The
// partials of sequence b are the slots p + b of the parts p that touch it
// (the balanced part partition of the block stream, recomputed here from the
// sequence lengths exactly as the decode kernels compute it).
#include <math.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace {

constexpr int kHeadsPerCta = 8;              // one warp per head
constexpr int kThreads = 32 * kHeadsPerCta;
constexpr int kMaxSplits = 1024;

// grid: (ceil(h / kHeadsPerCta), B); warp w merges head blockIdx.x * 8 + w of
// sequence blockIdx.y.  Lane l owns latent columns 4l + 128 i of each
// 512-column run (16-byte loads, each warp access a contiguous 512-byte run).
__global__ void __launch_bounds__(kThreads)
combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
               const int32_t* __restrict__ seq_lens, int bs, int max_blocks, int B, int h,
               int d_c, int num_parts, void* __restrict__ o_lat, int o_dtype,
               float* __restrict__ lse_out) {
  __shared__ int s_first, s_count;
  // scheduled while the decode finishes; its partials are read after it completes
  tc::grid_dep_launch();
  tc::grid_dep_wait();
  const int b = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (warp == 0) {
    long long sb = 0;
    const long long T = warp_stream_scan(seq_lens, B, bs, max_blocks, b, -1, &sb, nullptr, nullptr);
    const int nb = seq_blocks(seq_lens, b, bs, max_blocks);
    if (lane == 0) {
      if (nb == 0) {
        s_first = 0;
        s_count = 0;
      } else {
        const int P = (int)(T < num_parts ? T : num_parts);
        const int p0 = part_of(T, P, sb), p1 = part_of(T, P, sb + nb - 1);
        s_first = p0 + b;
        s_count = p1 - p0 + 1;
      }
    }
  }
  __syncthreads();
  const int s = blockIdx.x * kHeadsPerCta + warp;
  if (s >= h) return;
  const int first = s_first, count = s_count;
  const float* lse_col = lse_part + (int64_t)first * h + s;   // split j at lse_col[j * h]

  // maximum and weight sum over the splits (lanes stride over splits)
  float m = -INFINITY;
  for (int j = lane; j < count; j += 32) m = fmaxf(m, lse_col[(int64_t)j * h]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float wsum = 0.f;
  for (int j = lane; j < count; j += 32) {
    const float l = lse_col[(int64_t)j * h];
    wsum += (m == -INFINITY || l == -INFINITY) ? 0.f : expf(l - m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;

  const int64_t obase = ((int64_t)b * h + s) * d_c;
  // lane j of each round of 32 splits holds split j's weight; every split's
  // loads go out without waiting on its weight (a zero weight, an empty
  // split, is applied by select, so whatever its slot holds is ignored)
  for (int c0 = 0; c0 < d_c; c0 += 512) {
    float4 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < count; j0 += 32) {
      float wl = 0.f;
      if (j0 + lane < count) {
        const float l = lse_col[(int64_t)(j0 + lane) * h];
        wl = (m == -INFINITY || l == -INFINITY) ? 0.f : expf(l - m);
      }
      const int n = count - j0 < 32 ? count - j0 : 32;
#pragma unroll 2
      for (int jj = 0; jj < n; ++jj) {
        const float w = __shfl_sync(0xffffffffu, wl, jj);
        const float* src = o_part + (((int64_t)first + j0 + jj) * h + s) * d_c + c0 + 4 * lane;
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          v[i] = (c0 + 4 * lane + 128 * i < d_c) ? *reinterpret_cast<const float4*>(src + 128 * i)
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        if (w != 0.f) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[i].x = fmaf(w, v[i].x, acc[i].x);
            acc[i].y = fmaf(w, v[i].y, acc[i].y);
            acc[i].z = fmaf(w, v[i].z, acc[i].z);
            acc[i].w = fmaf(w, v[i].w, acc[i].w);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = c0 + 4 * lane + 128 * i;
      if (c >= d_c) continue;
      if (o_dtype == MLA_F32) {
        *reinterpret_cast<float4*>(static_cast<float*>(o_lat) + obase + c) =
            make_float4(acc[i].x * inv, acc[i].y * inv, acc[i].z * inv, acc[i].w * inv);
      } else {
        uint16_t* o = static_cast<uint16_t*>(o_lat) + obase + c;
        uint2 pk;
        pk.x = (uint32_t)f32_to_bf16_rn(acc[i].x * inv) | ((uint32_t)f32_to_bf16_rn(acc[i].y * inv) << 16);
        pk.y = (uint32_t)f32_to_bf16_rn(acc[i].z * inv) | ((uint32_t)f32_to_bf16_rn(acc[i].w * inv) << 16);
        *reinterpret_cast<uint2*>(o) = pk;
      }
    }
  }
  if (lse_out && lane == 0)
    lse_out[(int64_t)b * h + s] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const float* o_part, const float* lse_part, const int32_t* seq_lens,
                           int block_size, int max_blocks, int B, int h, int d_c, int num_parts,
                           void* o_lat, int o_dtype, float* lse, cudaStream_t s) {
  if (num_parts > kMaxSplits) return cudaErrorInvalidValue;
  dim3 grid(ceil_div(h, kHeadsPerCta), B);
  return launch_pdl(combine_kernel, grid, dim3(kThreads), 0, s, o_part, lse_part, seq_lens,
                    block_size, max_blocks, B, h, d_c, num_parts, o_lat, o_dtype, lse);
}

}  // namespace mla
