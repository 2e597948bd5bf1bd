// Per-head GEMMs of the absorbed decode on the tensor cores (tcgen05 + TMEM +
// TMA), bf16 in, float32 accumulate:
//
//   mla_absorb_q  (kexue.fm "From MHA, MQA, GQA to MLA", section "Part 1" and
//                  its note 2; eq. mla-mqa, first block of q):
//     q_cat[b, s, c] = sum_d q_nope[b, s, d] W_UK[s, d, c]   (c < 512), and the
//     rotary part q_cat[b, s, 512 + j] = RoPE(q_rope[b, s, :], q_pos[b])[j].
//   mla_out_proj  (eq. mla-mqa, first line: o_t = [o^(s) W_v^(s)]):
//     out[b, s, v] = sum_c o_lat[b, s, c] W_UV[s, v, c].
//
// Both have the form D[m][n] = sum_k A_s[m][k] X_s[n][k] per head s, with m an
// output feature (the 128 TMEM lanes), n the batch row (TMEM columns, up to
// 256 per CTA) and k the contraction, streamed in 64-wide chunks by TMA:
//   absorb:   A_s[c][d] = W_UK[s][d][c]  (MN-major A: c is contiguous),
//             X_s[b][d] = q_nope[b][s][d] (K-major, a 3-D box over (d, s, b));
//   out_proj: A_s[v][c] = W_UV[s][v][c]  (K-major A),
//             X_s[b][c] = o_lat[b][s][c]  (K-major, a 3-D box over (c, s, b)).
// Grid (h, m tiles, batch tiles); 128 threads: warp 0 issues TMA, warp 1 owns
// TMEM and issues the MMAs, all four warps run the epilogue (thread = m).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "device_registry.h"
#include "tc_ptx.cuh"

namespace mla {

// defined in decode_tc.cu
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

namespace {

using namespace tc;

constexpr int kKChunk = 64;                 // contraction elements per stage
constexpr int kStagesG = 4;
constexpr int kABytes = 128 * kKChunk * 2;  // 16 KB: 128 m x 64 k
constexpr int kMaxN = 256;
constexpr int kGThreads = 128;

struct GemmParams {
  int K;            // contraction length (multiple of 64)
  int n_tile;       // batch rows per CTA (multiple of 16, <= 256)
  int nstage;       // pipeline stages (<= kStagesG)
  int stage_bytes;  // A chunk + X chunk, multiple of 1024
  int tmem_cols;    // power of two >= max(32, n_tile)
  int B, h;
  // K-major A: the tile of (s, m tile mt, chunk kc) starts at row
  // s * a_row_s + mt * 128, column s * a_col_s + kc * 64 of the 2-D A map
  // (per-head weights: rows advance with s; split contraction: columns do)
  int a_row_s, a_col_s;
  void* out;        // element (b, s, m) at out + (b * h + s) * out_ld + m
  int out_ld;
  int out_dtype;
  // rotary part of the absorbed query (absorb only)
  const uint16_t* q_rope;  // [B, h, 64] bf16 or null
  const int32_t* q_pos;
  double inv_freq[32];     // theta^(-2i/64), formed in float64 on the host
  float turn_hi[32];       // inv_freq / (2 pi) as a float32 head + tail
  float turn_lo[32];
  int32_t* status;
  long long wait_limit;
};

template <bool kAMajorMN>
__global__ void __launch_bounds__(kGThreads)
head_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_x,
                 const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int s = blockIdx.x, mt = blockIdx.y, nt = blockIdx.z;
  const int b0 = nt * p.n_tile;
  const int nk = p.K / kKChunk;
  const int nstage = p.nstage;
  const int kGStageBytes = p.stage_bytes;
  grid_dep_launch();

  const uint32_t bars = sbase + nstage * kGStageBytes;   // full[4], empty[4], done
  auto full = [&](int i) { return bars + 8 * i; };
  auto empty = [&](int i) { return bars + 8 * (kStagesG + i); };
  const uint32_t done = bars + 8 * (2 * kStagesG);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + nstage * kGStageBytes + 128);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesG; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const long long lim = p.wait_limit;
  bool ok = true;
  // this CTA's weight tiles into L2 while the previous grid of the stream
  // finishes (a prefetch brings nothing into the CTA, and L2 stays coherent
  // with that grid's writes); every read of memory comes after the wait
  if (warp == 0 && lane == 0) {
    for (int kc = 0; kc < nk; ++kc) {
      if (kAMajorMN) {
        tma_prefetch_2d(&tm_a, mt * 128, s * p.K + kc * kKChunk);
        tma_prefetch_2d(&tm_a, mt * 128 + 64, s * p.K + kc * kKChunk);
      } else {
        tma_prefetch_2d(&tm_a, s * p.a_col_s + kc * kKChunk, s * p.a_row_s + mt * 128);
      }
    }
  }
  grid_dep_wait();

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint32_t xbytes = (uint32_t)p.n_tile * kKChunk * 2;
    for (int kc = 0; kc < nk; ++kc) {
      const int st = kc % nstage;
      if (kc >= nstage && !mbar_wait(empty(st), ((kc / nstage) - 1) & 1, lim)) {
        ok = false;
        break;
      }
      const uint32_t a_dst = sbase + st * kGStageBytes;
      const uint32_t x_dst = a_dst + kABytes;
      mbar_arrive_expect_tx(full(st), kABytes + xbytes);
      if (kAMajorMN) {
        // two boxes of 64 m (contiguous) x 64 k rows
        tma_load_2d(a_dst, &tm_a, mt * 128, s * p.K + kc * kKChunk, full(st));
        tma_load_2d(a_dst + kABytes / 2, &tm_a, mt * 128 + 64, s * p.K + kc * kKChunk, full(st));
      } else {
        // one box of 64 k (contiguous) x 128 m rows
        tma_load_2d(a_dst, &tm_a, s * p.a_col_s + kc * kKChunk, s * p.a_row_s + mt * 128,
                    full(st));
      }
      tma_load_3d(x_dst, &tm_x, kc * kKChunk, s, b0, full(st));
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(128, p.n_tile, kAMajorMN, false);
    for (int kc = 0; kc < nk && ok; ++kc) {
      const int st = kc % nstage;
      if (!mbar_wait(full(st), (kc / nstage) & 1, lim)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a_st = sbase + st * kGStageBytes;
      const uint32_t x_st = a_st + kABytes;
#pragma unroll
      for (int kk = 0; kk < kKChunk / 16; ++kk) {
        const uint64_t ad = kAMajorMN ? smem_desc(a_st + kk * 2048, kABytes / 2, 1024, kSwizzle128B)
                                      : smem_desc(a_st + kk * 32, 16, 1024, kSwizzle128B);
        const uint64_t xd = smem_desc(x_st + kk * 32, 16, 1024, kSwizzle128B);
        mma_ss(tmem, ad, xd, idesc, (kc > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(empty(st));
    }
    mma_commit(done);
  }
  __syncwarp();

  // rotary query part (absorb): independent of the MMA; the (row, pair) items
  // of this head are spread over its m-tile CTAs.  A thread's items are
  // loaded together, then rotated, so their load latencies overlap.
  if (p.q_rope != nullptr) {
    const int nb = min(p.n_tile, p.B - b0);
    const int total = nb * 32;
    const int stride = kGThreads * (int)gridDim.y;
    uint16_t* q_cat = static_cast<uint16_t*>(p.out);
    constexpr int kU = 4;
    for (int i0 = threadIdx.x + mt * kGThreads; i0 < total; i0 += kU * stride) {
      uint32_t xr[kU];
      int32_t ps[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * stride;
        if (i < total) {
          const int bb = b0 + i / 32, pr = i % 32;
          ps[u] = p.q_pos[bb];
          xr[u] = *reinterpret_cast<const uint32_t*>(p.q_rope + ((int64_t)bb * p.h + s) * 64 +
                                                    2 * pr);
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * stride;
        if (i >= total) break;
        const int bb = b0 + i / 32, pr = i % 32;
        float cs, sn;
        if ((uint32_t)ps[u] < (1u << 24))
          rope_cos_sin_turns(ps[u], p.turn_hi[pr], p.turn_lo[pr], &cs, &sn);
        else
          rope_cos_sin((double)ps[u], p.inv_freq[pr], &cs, &sn);
        const float x0 = bf16_to_f32((uint16_t)(xr[u] & 0xffffu));
        const float x1 = bf16_to_f32((uint16_t)(xr[u] >> 16));
        const int64_t ob = ((int64_t)bb * p.h + s) * p.out_ld + 512 + 2 * pr;
        *reinterpret_cast<uint32_t*>(q_cat + ob) =
            (uint32_t)f32_to_bf16_rn(x0 * cs - x1 * sn) |
            ((uint32_t)f32_to_bf16_rn(x0 * sn + x1 * cs) << 16);
      }
    }
  }

  // ------------------------------------------------------------ epilogue
  // (every thread waits for the MMAs, even after a failure, so that TMEM is
  // never released under a running MMA)
  ok = __syncthreads_and(ok);
  const bool waited = __syncthreads_and(mbar_wait(done, 0, lim));
  if (!ok || !waited) {
    if (threadIdx.x == 0) set_status(p.status, MLA_DEV_WAIT_TIMEOUT);
  } else {
    tc_fence_after();
    const int m = warp * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    for (int c0 = 0; c0 < p.n_tile; c0 += 16) {
      uint32_t v[16];
      tmem_ld16(tl + c0, v);
      tmem_wait_ld();
      if (p.out_dtype == MLA_BF16) {
        // pairs of neighbouring m (lanes 2j, 2j+1) as one 4-byte store: the
        // even lane stores row e, the odd lane row e + 1
        uint16_t* out16 = static_cast<uint16_t*>(p.out);
        const bool odd = (lane & 1) != 0;
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float send = __uint_as_float(odd ? v[e] : v[e + 1]);
          const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
          const int b = b0 + c0 + e + (odd ? 1 : 0);
          if (b < p.B) {
            const float lo = odd ? recv : __uint_as_float(v[e]);
            const float hi = odd ? __uint_as_float(v[e + 1]) : recv;
            const int64_t o = ((int64_t)b * p.h + s) * p.out_ld + mt * 128 + (m & ~1);
            *reinterpret_cast<uint32_t*>(out16 + o) =
                (uint32_t)f32_to_bf16_rn(lo) | ((uint32_t)f32_to_bf16_rn(hi) << 16);
          }
        }
        continue;
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int b = b0 + c0 + e;
        if (b < p.B) {
          const int64_t o = ((int64_t)b * p.h + s) * p.out_ld + mt * 128 + m;
          if (p.out_dtype == MLA_F32)
            static_cast<float*>(p.out)[o] = __uint_as_float(v[e]);
          else
            static_cast<uint16_t*>(p.out)[o] = f32_to_bf16_rn(__uint_as_float(v[e]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

constexpr int kGSmemMax = kStagesG * (kABytes + kMaxN * kKChunk * 2) + 256 + 1024;

// y[b, n] = sum_s part[b, s, n] over the split partials, in split order
// (deterministic); four columns per thread.
__global__ void __launch_bounds__(256)
split_reduce_kernel(const float* __restrict__ part, int splits, int B, int N, void* y,
                    int y_dtype) {
  const int64_t i = ((int64_t)blockIdx.x * 256 + threadIdx.x) * 4;
  if (i >= (int64_t)B * N) return;
  const int b = (int)(i / N), n = (int)(i % N);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sp = 0; sp < splits; ++sp) {
    const float4 v = *reinterpret_cast<const float4*>(part + ((int64_t)b * splits + sp) * N + n);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  if (y_dtype == MLA_F32) {
    *reinterpret_cast<float4*>(static_cast<float*>(y) + i) = acc;
  } else {
    uint2 pk;
    pk.x = (uint32_t)f32_to_bf16_rn(acc.x) | ((uint32_t)f32_to_bf16_rn(acc.y) << 16);
    pk.y = (uint32_t)f32_to_bf16_rn(acc.z) | ((uint32_t)f32_to_bf16_rn(acc.w) << 16);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(y) + i) = pk;
  }
}

// Pipeline shape for a contraction of K and a batch tile of n rows.
void shape(GemmParams* p, int K, int n) {
  p->K = K;
  p->n_tile = n;
  const int nk = K / kKChunk;
  p->nstage = nk < kStagesG ? nk : kStagesG;
  p->stage_bytes = (kABytes + n * kKChunk * 2 + 1023) / 1024 * 1024;
  int c = 32;
  while (c < n) c *= 2;
  p->tmem_cols = c;
}

int smem_bytes(const GemmParams& p) { return p.nstage * p.stage_bytes + 256 + 1024; }

bool encode(CUtensorMap* m, int rank, const void* base, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// batch rows per CTA: at most cap (a multiple of 16), rounded up to 16
int n_tile_for(int B, int cap = kMaxN) {
  int n = B < cap ? B : cap;
  return (n + 15) / 16 * 16;
}

// the dynamic shared-memory limit is a per-device setting: once per device
template <bool kMN>
cudaError_t set_smem_attr() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int r = device_registry().once(dev, kMN ? kSetupGemmMN : kSetupGemmK, []() {
    return (int)cudaFuncSetAttribute(head_gemm_kernel<kMN>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmemMax);
  });
  if (r != 0) return r < 0 ? cudaErrorInvalidDevice : (cudaError_t)r;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_absorb_q_tc(const void* q_nope, const void* q_rope, const int32_t* q_pos,
                               const void* w_uk, void* q_cat, int B, int h, double theta,
                               cudaStream_t s) {
  // A: W_UK as [h * 128 (s, d) rows, 512 (c) cols]; boxes of 64 c x 64 d
  CUtensorMap ta, tx;
  cuuint64_t adims[2] = {512, (cuuint64_t)h * 128};
  cuuint64_t astr[1] = {512 * 2};
  cuuint32_t abox[2] = {64, 64};
  // X: q_nope as (d = 128, s = h, b = B); boxes of 64 d x 1 x n_tile
  const int nt = n_tile_for(B);
  cuuint64_t xdims[3] = {128, (cuuint64_t)h, (cuuint64_t)B};
  cuuint64_t xstr[2] = {128 * 2, (cuuint64_t)h * 128 * 2};
  cuuint32_t xbox[3] = {64, 1, (cuuint32_t)nt};
  if (!encode(&ta, 2, w_uk, adims, astr, abox) || !encode(&tx, 3, q_nope, xdims, xstr, xbox))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_attr<true>();
  if (e != cudaSuccess) return e;
  GemmParams p{};
  shape(&p, 128, nt);
  p.B = B;
  p.h = h;
  p.out = q_cat;
  p.out_ld = 576;
  p.out_dtype = MLA_BF16;
  p.q_rope = static_cast<const uint16_t*>(q_rope);
  p.q_pos = q_pos;
  for (int i = 0; i < 32; ++i) {
    p.inv_freq[i] = pow(theta, -2.0 * (double)i / 64.0);
    const double turns = p.inv_freq[i] / 6.283185307179586476925;
    p.turn_hi[i] = (float)turns;
    p.turn_lo[i] = (float)(turns - (double)p.turn_hi[i]);
  }
  p.status = nullptr;
  p.wait_limit = 4000000000LL;
  dim3 grid(h, 512 / 128, ceil_div(B, nt));
  return launch_pdl(head_gemm_kernel<true>, grid, dim3(kGThreads), smem_bytes(p), s, ta, tx, p);
}

cudaError_t launch_out_proj_tc(const void* o_lat, const void* w_uv, void* out, int B, int h,
                               int out_dtype, cudaStream_t s) {
  // A: W_UV as [h * 128 (s, v) rows, 512 (c) cols]; boxes of 64 c x 128 v
  CUtensorMap ta, tx;
  cuuint64_t adims[2] = {512, (cuuint64_t)h * 128};
  cuuint64_t astr[1] = {512 * 2};
  cuuint32_t abox[2] = {64, 128};
  // 32 batch rows per CTA: more CTAs stream W_UV (from L2 after the first) in parallel
  const int nt = n_tile_for(B, 32);
  cuuint64_t xdims[3] = {512, (cuuint64_t)h, (cuuint64_t)B};
  cuuint64_t xstr[2] = {512 * 2, (cuuint64_t)h * 512 * 2};
  cuuint32_t xbox[3] = {64, 1, (cuuint32_t)nt};
  if (!encode(&ta, 2, w_uv, adims, astr, abox) || !encode(&tx, 3, o_lat, xdims, xstr, xbox))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_attr<false>();
  if (e != cudaSuccess) return e;
  GemmParams p{};
  shape(&p, 512, nt);
  p.B = B;
  p.h = h;
  p.a_row_s = 128;
  p.a_col_s = 0;
  p.out = out;
  p.out_ld = 128;
  p.out_dtype = out_dtype;
  p.q_rope = nullptr;
  p.q_pos = nullptr;
  p.status = nullptr;
  p.wait_limit = 4000000000LL;
  dim3 grid(h, 1, ceil_div(B, nt));
  return launch_pdl(head_gemm_kernel<false>, grid, dim3(kGThreads), smem_bytes(p), s, ta, tx, p);
}

// ---------------------------------------------------------------------------
// plain linear layers and the W_UV / W_O fold
// ---------------------------------------------------------------------------

// Contraction splits of y = x W^T (M x K times N x K): enough CTAs to cover
// the GPU about once (148 SMs on this part), each split at least 512 long.
int linear_splits(int M, int K, int N) {
  const int tiles = (N / 128) * ceil_div(M, n_tile_for(M));
  int sp = 1;
  while (sp < 64 && tiles * sp < 148 && (K / 64) % (2 * sp) == 0 && K / (2 * sp) >= 512) sp *= 2;
  return sp;
}

cudaError_t launch_linear_tc(const void* x, const void* w, void* y, int M, int K, int N,
                             int y_dtype, float* part, cudaStream_t s) {
  const int sp = linear_splits(M, K, N);
  const int ks = K / sp;
  const int nt = n_tile_for(M);
  // A: W as [N rows, K cols]; boxes of 64 k x 128 n
  CUtensorMap ta, tx;
  cuuint64_t adims[2] = {(cuuint64_t)K, (cuuint64_t)N};
  cuuint64_t astr[1] = {(cuuint64_t)K * 2};
  cuuint32_t abox[2] = {64, 128};
  // X: x as (k within split, split, row); boxes of 64 k x 1 x n_tile
  cuuint64_t xdims[3] = {(cuuint64_t)ks, (cuuint64_t)sp, (cuuint64_t)M};
  cuuint64_t xstr[2] = {(cuuint64_t)ks * 2, (cuuint64_t)K * 2};
  cuuint32_t xbox[3] = {64, 1, (cuuint32_t)nt};
  if (!encode(&ta, 2, w, adims, astr, abox) || !encode(&tx, 3, x, xdims, xstr, xbox))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_attr<false>();
  if (e != cudaSuccess) return e;
  GemmParams p{};
  shape(&p, ks, nt);
  p.B = M;
  p.h = sp;
  p.a_row_s = 0;
  p.a_col_s = ks;
  // one split: straight into y; several: float32 partials [M, splits, N]
  p.out = sp == 1 ? y : static_cast<void*>(part);
  p.out_ld = N;
  p.out_dtype = sp == 1 ? y_dtype : MLA_F32;
  p.q_rope = nullptr;
  p.q_pos = nullptr;
  p.status = nullptr;
  p.wait_limit = 4000000000LL;
  dim3 grid(sp, N / 128, ceil_div(M, nt));
  head_gemm_kernel<false><<<grid, kGThreads, smem_bytes(p), s>>>(ta, tx, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || sp == 1) return e;
  const int64_t n4 = (int64_t)M * N / 4;
  split_reduce_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(part, sp, M, N, y, y_dtype);
  return cudaGetLastError();
}

cudaError_t launch_fold_uv_o_tc(const void* w_uv, const void* w_o, void* w_fold, int h,
                                int d_model, cudaStream_t s) {
  // W_fold[n, s, c] = sum_v W_O[n, s * 128 + v] W_UV[s, v, c]: per head s,
  // D[c][n] = sum_v A_s[c][v] X_s[n][v] with A_s[c][v] = W_UV[s][v][c]
  // (MN-major, as W_UK in the absorbed query) and X_s[n][v] = W_O[n][s][v]
  CUtensorMap ta, tx;
  cuuint64_t adims[2] = {512, (cuuint64_t)h * 128};
  cuuint64_t astr[1] = {512 * 2};
  cuuint32_t abox[2] = {64, 64};
  const int nt = n_tile_for(d_model);
  cuuint64_t xdims[3] = {128, (cuuint64_t)h, (cuuint64_t)d_model};
  cuuint64_t xstr[2] = {128 * 2, (cuuint64_t)h * 128 * 2};
  cuuint32_t xbox[3] = {64, 1, (cuuint32_t)nt};
  if (!encode(&ta, 2, w_uv, adims, astr, abox) || !encode(&tx, 3, w_o, xdims, xstr, xbox))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_attr<true>();
  if (e != cudaSuccess) return e;
  GemmParams p{};
  shape(&p, 128, nt);
  p.B = d_model;
  p.h = h;
  p.out = w_fold;
  p.out_ld = 512;
  p.out_dtype = MLA_BF16;
  p.q_rope = nullptr;
  p.q_pos = nullptr;
  p.status = nullptr;
  p.wait_limit = 4000000000LL;
  dim3 grid(h, 512 / 128, ceil_div(d_model, nt));
  head_gemm_kernel<true><<<grid, kGThreads, smem_bytes(p), s>>>(ta, tx, p);
  return cudaGetLastError();
}

}  // namespace mla
