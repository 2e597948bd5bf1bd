// mla_combine_out_proj: the log-sum-exp merge of the split-KV partials and
// the W_UV output projection in one kernel (tcgen05 + TMEM + TMA).
//
// For sequence b and head s (iotdigitaltwinplm.com, the absorbed decode
// listing; kexue.fm "From MHA, MQA, GQA to MLA", eq. mla-mqa, first line:
// o_t = [o^(s) W_v^(s)]):
//   o_lat[b, s, :] = sum_j w_j o_part[j, s, :] / sum_j w_j,  w_j = exp(lse_j - max lse)
//   out[b, s, v]   = sum_c bf16(o_lat[b, s, c]) W_UV[s, v, c]
// The merge is the same per-element arithmetic, in the same slot order, as
// mla_combine (row maximum and weight sum by the same warp-level reduction,
// then one fused multiply-add per slot), so o_lat and lse equal mla_combine's
// bit for bit; the merged rows go straight into the B operand of the
// projection in shared memory instead of through memory.
//
// One CTA per (head s, 64 batch rows), 576 threads:
//   warp 0       TMA: the eight 64-column chunks of W_UV[s] (128 x 512, the A
//                operand, K-major), all in flight at once;
//   warp 1       TMEM (64 columns) and, on one thread, the 32 MMAs
//                D[v][b] = sum_c A[v][c] X[b][c] (M = 128, N = 64, K = 16);
//   warps 2..17  the merge: first each warp takes four rows' slot ranges and
//                weights (one row per pass, as mla_combine's warp does), then
//                thread t merges row t / 8, latent columns [64 q, 64 q + 64)
//                with q = t % 8 (X chunk q), and writes bf16 pairs into the
//                128-byte-swizzled chunk; warps 2..5 then write out from TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "device_registry.h"
#include "tc_ptx.cuh"

namespace mla {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

namespace {

using namespace tc;

constexpr int kRows = 64;                   // batch rows per CTA (the MMA's N)
constexpr int kDc = 512, kDv = 128;
constexpr int kChunks = kDc / 64;           // 64-column chunks of the contraction
constexpr int kABytes = 128 * 64 * 2;       // 16 KB: 128 v x 64 c
constexpr int kXBytes = kRows * 64 * 2;     // 8 KB: 64 rows x 64 c
constexpr int kMergeWarps = 16;
constexpr int kThreads = 64 + 32 * kMergeWarps;
constexpr int kOffA = 0;
constexpr int kOffX = kOffA + kChunks * kABytes;
constexpr int kOffRow = kOffX + kChunks * kXBytes;     // per row: first slot, count, max, 1/sum
constexpr int kOffBar = kOffRow + kRows * 16;
constexpr int kOffMisc = kOffBar + 4 * 8;
constexpr int kSmemBytes = kOffMisc + 16;
constexpr int kSmemAlloc = kSmemBytes + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory budget");
static_assert(kOffX % 1024 == 0, "swizzled chunks start on 1 KB");
constexpr uint32_t kTmemCols = 64;

enum { BAR_A_FULL = 0, BAR_X_FULL = 1, BAR_DONE = 2 };

struct CpParams {
  const float* o_part;     // [slots, h, 512]
  const float* lse_part;   // [slots, h]
  const int32_t* seq_lens;
  int bs, max_blocks, B, h, num_parts;
  void* out;               // [B, h, 128], out_dtype
  int out_dtype;
  void* o_lat;             // [B, h, 512] in o_dtype, or null
  int o_dtype;
  float* lse;              // [B, h] or null
  int32_t* status;
  long long wait_limit;
};

__global__ void __launch_bounds__(kThreads, 1)
combine_proj_kernel(const __grid_constant__ CUtensorMap tm_a, const CpParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int s = blockIdx.x, b0 = blockIdx.y * kRows;
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8 * i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  int* row_first = reinterpret_cast<int*>(smem + kOffRow);
  int* row_count = row_first + kRows;
  float* row_max = reinterpret_cast<float*>(row_count + kRows);
  float* row_inv = row_max + kRows;
  grid_dep_launch();

  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_A_FULL), 1);
    mbar_init(bar(BAR_X_FULL), kMergeWarps);
    mbar_init(bar(BAR_DONE), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const long long lim = p.wait_limit;
  // W_UV[s] into L2 while the previous grid of the stream finishes; every
  // read of memory comes after the wait
  if (warp == 0 && lane == 0)
    for (int kc = 0; kc < kChunks; ++kc) tma_prefetch_2d(&tm_a, kc * 64, s * kDv);
  grid_dep_wait();
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA: W_UV[s]
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(BAR_A_FULL), kChunks * kABytes);
      for (int kc = 0; kc < kChunks; ++kc)
        tma_load_2d(sbase + kOffA + kc * kABytes, &tm_a, kc * 64, s * kDv, bar(BAR_A_FULL));
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA (one thread)
    if (lane == 0) {
      ok = mbar_wait(bar(BAR_A_FULL), 0, lim) && mbar_wait(bar(BAR_X_FULL), 0, lim);
      if (ok) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, kRows, false, false);
        for (int kc = 0; kc < kChunks; ++kc) {
          const uint32_t a_st = sbase + kOffA + kc * kABytes;
          const uint32_t x_st = sbase + kOffX + kc * kXBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc(a_st + kk * 32, 16, 1024, kSwizzle128B);
            const uint64_t xd = smem_desc(x_st + kk * 32, 16, 1024, kSwizzle128B);
            mma_ss(tmem, ad, xd, idesc, (kc > 0 || kk > 0) ? 1u : 0u);
          }
        }
      }
      // commit even after a failure, so that the epilogue's wait ends
      mma_commit(bar(BAR_DONE));
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ merge
    const int cw = warp - 2;                  // 0..15
    // (1) slot range, maximum and 1 / weight sum of rows 4 cw .. 4 cw + 3,
    //     one row per pass of the warp (lanes stride over the slots)
    for (int i = 0; i < kRows / kMergeWarps; ++i) {
      const int r = cw * (kRows / kMergeWarps) + i;
      const int b = b0 + r;
      int first = 0, count = 0;
      if (b < p.B) {
        long long sb = 0;
        const long long T =
            warp_stream_scan(p.seq_lens, p.B, p.bs, p.max_blocks, b, -1, &sb, nullptr, nullptr);
        const int nbk = seq_blocks(p.seq_lens, b, p.bs, p.max_blocks);
        if (nbk > 0) {
          const int P = (int)(T < p.num_parts ? T : p.num_parts);
          const int p0 = part_of(T, P, sb), p1 = part_of(T, P, sb + nbk - 1);
          first = p0 + b;
          count = p1 - p0 + 1;
        }
      }
      const float* lse_col = p.lse_part + (int64_t)first * p.h + s;
      float m = -INFINITY;
      for (int j = lane; j < count; j += 32) m = fmaxf(m, lse_col[(int64_t)j * p.h]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      float wsum = 0.f;
      for (int j = lane; j < count; j += 32) {
        const float l = lse_col[(int64_t)j * p.h];
        wsum += (m == -INFINITY || l == -INFINITY) ? 0.f : expf(l - m);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
      if (lane == 0) {
        row_first[r] = first;
        row_count[r] = count;
        row_max[r] = m;
        row_inv[r] = wsum > 0.f ? 1.f / wsum : 0.f;
        if (p.lse != nullptr && b < p.B)
          p.lse[(int64_t)b * p.h + s] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(32 * kMergeWarps) : "memory");
    // (2) thread t merges row t / 8, columns [64 q, 64 q + 64) (X chunk q), in
    //     two halves of 32 columns; slots in order, one fused multiply-add each
    const int t = threadIdx.x - 64;
    const int r = t >> 3, q = t & 7;
    const int b = b0 + r;
    const int first = row_first[r], count = row_count[r];
    const float m = row_max[r], inv = row_inv[r];
    uint8_t* xrow = smem + kOffX + q * kXBytes + r * 128;
    for (int half = 0; half < 2; ++half) {
      const int c0 = 64 * q + 32 * half;
      float acc[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = 0.f;
      for (int j = 0; j < count; ++j) {
        const float l = p.lse_part[(int64_t)(first + j) * p.h + s];
        const float w = (m == -INFINITY || l == -INFINITY) ? 0.f : expf(l - m);
        const float4* src = reinterpret_cast<const float4*>(
            p.o_part + ((int64_t)(first + j) * p.h + s) * kDc + c0);
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = src[i];
        if (w != 0.f) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            acc[4 * i] = fmaf(w, v[i].x, acc[4 * i]);
            acc[4 * i + 1] = fmaf(w, v[i].y, acc[4 * i + 1]);
            acc[4 * i + 2] = fmaf(w, v[i].z, acc[4 * i + 2]);
            acc[4 * i + 3] = fmaf(w, v[i].w, acc[4 * i + 3]);
          }
        }
      }
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] *= inv;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        pk[i] = (uint32_t)f32_to_bf16_rn(acc[2 * i]) | ((uint32_t)f32_to_bf16_rn(acc[2 * i + 1]) << 16);
      if (b >= p.B) {
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = 0u;   // rows past the batch: finite zeros
      }
      // 16-byte chunks 4 half .. 4 half + 3 of the 128-byte row, swizzled by row % 8
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(xrow + (((4 * half + c) ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      if (p.o_lat != nullptr && b < p.B) {
        const int64_t o = ((int64_t)b * p.h + s) * kDc + c0;
        if (p.o_dtype == MLA_F32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o_lat) + o);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o_lat) + o);
#pragma unroll
          for (int c = 0; c < 4; ++c) dst[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(BAR_X_FULL));

    // ------------------------------------------------------------ epilogue
    if (warp < 6) {
      const bool done = __shfl_sync(0xffffffffu, lane == 0 ? (mbar_wait(bar(BAR_DONE), 0, lim) ? 1 : 0) : 0, 0) != 0;
      if (!done) {
        ok = false;
      } else {
        tc_fence_after();
        const int sub = warp & 3;
        const int v = sub * 32 + lane;      // output feature (TMEM lane)
        const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16);
        for (int c0 = 0; c0 < kRows; c0 += 16) {
          uint32_t d[16];
          tmem_ld16(tl + c0, d);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int bb = b0 + c0 + e;
            if (bb < p.B) {
              const int64_t o = ((int64_t)bb * p.h + s) * kDv + v;
              if (p.out_dtype == MLA_F32)
                static_cast<float*>(p.out)[o] = __uint_as_float(d[e]);
              else
                static_cast<uint16_t*>(p.out)[o] = f32_to_bf16_rn(__uint_as_float(d[e]));
            }
          }
        }
      }
    }
  }
  if (!ok && p.status != nullptr) set_status(p.status, MLA_DEV_WAIT_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_combine_out_proj(const float* o_part, const float* lse_part,
                                    const int32_t* seq_lens, int block_size, int max_blocks,
                                    int B, int h, int num_parts, const void* w_uv, void* out,
                                    int out_dtype, void* o_lat, int o_dtype, float* lse,
                                    int32_t* status, cudaStream_t s) {
  // A: W_UV as [h * 128 (s, v) rows, 512 (c) cols]; boxes of 64 c x 128 v
  auto fn = tensor_map_encoder();
  if (!fn) return cudaErrorInvalidValue;
  CUtensorMap ta;
  cuuint64_t dims[2] = {(cuuint64_t)kDc, (cuuint64_t)h * kDv};
  cuuint64_t strides[1] = {kDc * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  if (fn(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w_uv), dims, strides, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int r = device_registry().once(dev, kSetupCombineProj, []() {
    return (int)cudaFuncSetAttribute(combine_proj_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  });
  if (r != 0) return r < 0 ? cudaErrorInvalidDevice : (cudaError_t)r;
  CpParams p{o_part, lse_part, seq_lens, block_size, max_blocks, B, h, num_parts, out,
             out_dtype, o_lat, o_dtype, lse, status, 4000000000LL};
  dim3 grid(h, ceil_div(B, kRows));
  return launch_pdl(combine_proj_kernel, grid, dim3(kThreads), kSmemAlloc, s, ta, p);
}

}  // namespace mla
