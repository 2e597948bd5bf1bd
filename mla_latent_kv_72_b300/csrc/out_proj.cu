// mla_out_proj: W_UV applied to the latent attention output (kexue.fm
// "From MHA, MQA, GQA to MLA", eq. mla-mqa, first line: o_t = [o^(s) W_v^(s)]).
#include "common.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBatchTile = 16;

// grid: (h, ceil(B / kBatchTile)); block: 256 threads.  Warp w computes rows
// v = w, w + 8, ... of head s for kBatchTile queries; lanes stride over d_c.
__global__ void __launch_bounds__(kThreads)
out_proj_simt_kernel(const void* __restrict__ o_lat, const void* __restrict__ w_uv,
                     void* __restrict__ out, int B, int h, int d_c, int d_v, int in_dtype,
                     int out_dtype) {
  extern __shared__ float so[];  // [kBatchTile][d_c]
  const int s = blockIdx.x;
  const int b0 = blockIdx.y * kBatchTile;
  const int nb = min(kBatchTile, B - b0);
  for (int i = threadIdx.x; i < kBatchTile * d_c; i += kThreads) {
    int bb = i / d_c, c = i % d_c;
    so[i] = bb < nb ? load_as_f32(o_lat, in_dtype, ((int64_t)(b0 + bb) * h + s) * d_c + c) : 0.f;
  }
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int v = warp; v < d_v; v += kWarps) {
    float acc[kBatchTile];
#pragma unroll
    for (int bb = 0; bb < kBatchTile; ++bb) acc[bb] = 0.f;
    const int64_t wrow = ((int64_t)s * d_v + v) * d_c;
    for (int c = lane; c < d_c; c += 32) {
      float w = load_as_f32(w_uv, in_dtype, wrow + c);
#pragma unroll
      for (int bb = 0; bb < kBatchTile; ++bb) acc[bb] = fmaf(w, so[bb * d_c + c], acc[bb]);
    }
#pragma unroll
    for (int bb = 0; bb < kBatchTile; ++bb) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[bb] += __shfl_xor_sync(0xffffffffu, acc[bb], off);
    }
    if (lane == 0) {
      for (int bb = 0; bb < nb; ++bb)
        store_from_f32(out, out_dtype, ((int64_t)(b0 + bb) * h + s) * d_v + v, acc[bb]);
    }
  }
}

}  // namespace

cudaError_t launch_out_proj_simt(const void* o_lat, const void* w_uv, void* out, int B, int h,
                                 int d_c, int d_v, int in_dtype, int out_dtype, cudaStream_t s) {
  size_t smem = sizeof(float) * kBatchTile * d_c;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(out_proj_simt_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(h, ceil_div(B, kBatchTile));
  out_proj_simt_kernel<<<grid, kThreads, smem, s>>>(o_lat, w_uv, out, B, h, d_c, d_v, in_dtype,
                                                    out_dtype);
  return cudaGetLastError();
}

}  // namespace mla
