// mla_prefill_fwd: causal attention of a whole prompt in the MHA form of MLA
// on the tensor cores (tcgen05 + TMEM + TMA), bf16 in, float32 accumulate.
//
// kexue.fm "From MHA, MQA, GQA to MLA", section "Part 3", eq. mla-mha (the
// form used for training and prefill): every head s has 192-d keys
// k_i = [c_i W_kc^(s), RoPE(k_R,i)] and 128-d values v_i = c_i W_v^(s), and
// token t attends to the tokens i <= t with its query [q_nope,t, RoPE(q_R,t)]
// and the scale 1/sqrt(192) (iotdigitaltwinplm.com "Prefill versus decode":
// at prefill the per-head keys and values are formed once and attention is
// compute-bound, so the absorbed form does not pay).  The per-head
// k_nope = C W_UK^T and v = C W_UV^T come from mla_linear; this kernel is the
// attention.
//
// One CTA per (128-query tile, head, sequence); 320 threads:
//   warp 0      TMA: the Q tile once (3 boxes of 64 dims x 128 tokens), then
//               the K (k_nope 2 boxes + the shared RoPE key 1 box) and V (2
//               boxes) tiles of 128 tokens into a ring of 2 stages;
//   warp 1      MMA issuer: S(j) = Q K(j)^T (12 K=16 steps, M = 128 queries,
//               N = 128 keys) into S buffer j % 2, and O += P(j) V(j) (8 steps,
//               P from TMEM, V as an MN-major operand);
//   warps 2..9  softmax: two warps per TMEM lane quarter split a row's 128
//               scores (64 each); online softmax with a lazily rescaled O
//               (only when the maximum grows by more than kTau, log2 units).
// TMEM columns: S x 2 [0, 256), O [256, 384), P (bf16 pairs) [384, 448).
// Key tiles past the query tile are skipped; the diagonal tile is masked to
// keys i <= t.  Every wait is bounded; a timeout is written to the status
// word and the kernel winds down.
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

constexpr int kTile = 128;                  // queries per CTA and keys per tile
constexpr int kBox = 128 * 128;             // 128 rows x 64 bf16, 128-byte swizzle (16 KB)
constexpr int kQBytes = 3 * kBox;           // 192 dims
constexpr int kKBytes = 3 * kBox;           // 128 nope dims + 64 RoPE dims
constexpr int kVBytes = 2 * kBox;           // 128 dims
constexpr int kStageBytes = kKBytes + kVBytes;
constexpr int kStages = 2;
constexpr int kThreads = 320;
constexpr int kSoftWarps = 8;
constexpr int kOffQ = 0;
constexpr int kOffStages = kOffQ + kQBytes;
constexpr int kOffHmax = kOffStages + kStages * kStageBytes;    // [2][128] float
constexpr int kOffLsum = kOffHmax + 2 * 128 * 4;                // [128] float
constexpr int kOffBar = kOffLsum + 128 * 4;
constexpr int kNumBars = 16;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 32;
constexpr int kSmemAlloc = kSmemBytes + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory budget");

constexpr uint32_t kColS = 0;     // [2] 128 columns each
constexpr uint32_t kColO = 256;
constexpr uint32_t kColP = 384;   // 64 columns: 128 keys as bf16 pairs
constexpr uint32_t kTmemCols = 512;

constexpr float kTau = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

enum {
  BAR_Q_FULL = 0,
  BAR_KV_FULL = 1,                // [2]
  BAR_KV_EMPTY = BAR_KV_FULL + 2, // [2]
  BAR_S_FULL = BAR_KV_EMPTY + 2,  // [2]
  BAR_S_EMPTY = BAR_S_FULL + 2,   // [2] softmax warps read S buffer j % 2
  BAR_P_FULL = BAR_S_EMPTY + 2,   // softmax warps stored P(j)
  BAR_O_DONE = BAR_P_FULL + 1,    // [2] O += P(j) V(j) done (by j % 2)
  BAR_DRAIN = BAR_O_DONE + 2,
  BAR_COUNT = BAR_DRAIN + 1,
};
static_assert(BAR_COUNT <= kNumBars, "barrier array");

struct PrefillParams {
  const int32_t* cu_seqlens;
  void* out;          // [T, h, 128], out_dtype
  int out_dtype;
  float* lse;         // [T, h] or null
  int h;
  float scale_log2;
  int32_t* status;
  long long wait_limit;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kn,
                  const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_v,
                  const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int qt = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
  const int row_begin = p.cu_seqlens[b];
  const int L = p.cu_seqlens[b + 1] - row_begin;
  const int q0 = qt * kTile;               // first query position of this CTA
  if (q0 >= L) return;                     // uniform for the whole CTA
  const int n_q = min(kTile, L - q0);      // live query rows
  const int ntiles = qt + 1;               // key tiles 0 .. qt (causal)
  const int r0 = row_begin + q0;           // global row of query 0 / of key tile qt

  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8 * i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_Q_FULL), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(BAR_KV_FULL + i), 1);
      mbar_init(bar(BAR_KV_EMPTY + i), 1);
      mbar_init(bar(BAR_S_FULL + i), 1);
      mbar_init(bar(BAR_S_EMPTY + i), kSoftWarps);
      mbar_init(bar(BAR_O_DONE + i), 1);
    }
    mbar_init(bar(BAR_P_FULL), kSoftWarps);
    mbar_init(bar(BAR_DRAIN), 1);
    *abort_flag = 0;
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
  bool timed_out = false;
  auto fail = [&]() {
    if (timed_out) set_status(p.status, MLA_DEV_WAIT_TIMEOUT);
    *abort_flag = 1;
  };
  auto warp_wait = [&](uint32_t bb, uint32_t parity) -> bool {
    bool ok = true;
    if (lane == 0) ok = mbar_wait_or_abort(bb, parity, lim, abort_flag, &timed_out);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(BAR_Q_FULL), kQBytes);
      for (int c = 0; c < 3; ++c)
        tma_load_3d(sbase + kOffQ + c * kBox, &tm_q, 64 * c, s, r0, bar(BAR_Q_FULL));
      int j = 0;
      for (; j < ntiles; ++j) {
        const int st = j % kStages;
        if (j >= kStages && !mbar_wait_or_abort(bar(BAR_KV_EMPTY + st), ((j / kStages) - 1) & 1,
                                                lim, abort_flag, &timed_out)) {
          fail();
          break;
        }
        const uint32_t dst = sbase + kOffStages + st * kStageBytes;
        const int kr = row_begin + j * kTile;   // global row of key 0 of tile j
        mbar_arrive_expect_tx(bar(BAR_KV_FULL + st), kStageBytes);
        tma_load_3d(dst, &tm_kn, 0, s, kr, bar(BAR_KV_FULL + st));
        tma_load_3d(dst + kBox, &tm_kn, 64, s, kr, bar(BAR_KV_FULL + st));
        tma_load_2d(dst + 2 * kBox, &tm_kr, 0, kr, bar(BAR_KV_FULL + st));
        tma_load_3d(dst + kKBytes, &tm_v, 0, s, kr, bar(BAR_KV_FULL + st));
        tma_load_3d(dst + kKBytes + kBox, &tm_v, 64, s, kr, bar(BAR_KV_FULL + st));
      }
      // every issued copy lands before the CTA may leave
      int never = 0;
      bool dummy = false;
      mbar_wait_or_abort(bar(BAR_Q_FULL), 0, lim, &never, &dummy);
      for (int st = 0; st < kStages; ++st) {
        const int n = (j - st + kStages - 1) / kStages;
        if (n > 0) mbar_wait_or_abort(bar(BAR_KV_FULL + st), (n - 1) & 1, lim, &never, &dummy);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // in order: S(j), then O += P(j-1) V(j-1); S(j) needs its stage and the
    // softmax's read of S(j-2); P(j-1) is written after O += P(j-2) V(j-2)
    const uint32_t idS = idesc_bf16_f32(128, 128, false, false);
    const uint32_t idO = idesc_bf16_f32(128, 128, false, true);
    bool ok = warp_wait(bar(BAR_Q_FULL), 0);
    auto issue_pv = [&](int jj) -> bool {
      if (!warp_wait(bar(BAR_P_FULL), jj & 1)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t v_st = sbase + kOffStages + (jj % kStages) * kStageBytes + kKBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = smem_desc(v_st + kk * 2048, kBox, 1024, kSwizzle128B);
          mma_ts(tmem + kColO, tmem + kColP + 8 * kk, bd, idO, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(BAR_O_DONE + (jj & 1)));
        mma_commit(bar(BAR_KV_EMPTY + (jj % kStages)));
      }
      __syncwarp();
      return true;
    };
    for (int j = 0; ok && j < ntiles; ++j) {
      const int st = j % kStages;
      if (!warp_wait(bar(BAR_KV_FULL + st), (j / kStages) & 1)) { ok = false; break; }
      if (j >= 2 && !warp_wait(bar(BAR_S_EMPTY + (j & 1)), ((j >> 1) - 1) & 1)) { ok = false; break; }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t k_st = sbase + kOffStages + st * kStageBytes;
        const uint32_t d = tmem + kColS + 128 * (j & 1);
#pragma unroll
        for (int kk = 0; kk < 12; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          const uint64_t ad = smem_desc(sbase + kOffQ + off, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(k_st + off, 16, 1024, kSwizzle128B);
          mma_ss(d, ad, bd, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(BAR_S_FULL + (j & 1)));
      }
      __syncwarp();
      if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
    }
    if (ok && !issue_pv(ntiles - 1)) ok = false;
    if (!ok) fail();
    if (lane == 0) {
      mma_commit(bar(BAR_DRAIN));
      int never = 0;
      bool dummy = false;
      mbar_wait_or_abort(bar(BAR_DRAIN), 0, lim, &never, &dummy);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int wg = warp - 2;              // 0..7
    const int hf = wg >> 2;               // column half: keys [64 hf, 64 hf + 64)
    const int sub = warp & 3;             // TMEM lane quarter
    const int row = sub * 32 + lane;      // query row of the tile
    const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16);
    float* hmax = reinterpret_cast<float*>(smem + kOffHmax);
    float* lsum = reinterpret_cast<float*>(smem + kOffLsum);
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(1 + sub) : "memory"); };
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles && ok; ++j) {
      if (!warp_wait(bar(BAR_S_FULL + (j & 1)), (j >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      uint32_t r[64];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_ld16(tl + kColS + 128 * (j & 1) + 64 * hf + 16 * c,
                  *reinterpret_cast<uint32_t(*)[16]>(&r[16 * c]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_S_EMPTY + (j & 1)));
      // scores in log2 units; the diagonal tile sees keys i <= t only
      const bool diag = j == qt;
      float mt = -INFINITY;
#pragma unroll
      for (int kk = 0; kk < 64; ++kk) {
        float x = __uint_as_float(r[kk]) * p.scale_log2;
        if (diag && 64 * hf + kk > row) x = -INFINITY;
        r[kk] = __float_as_uint(x);
        mt = fmaxf(mt, x);
      }
      // row maximum over both halves
      pair_sync();
      hmax[hf * 128 + row] = mt;
      pair_sync();
      mt = fmaxf(mt, hmax[(hf ^ 1) * 128 + row]);
      float m_new = m_run;
      bool resc = false;
      if (m_run == -INFINITY) {
        m_new = mt;
      } else if (mt > m_run + kTau) {
        m_new = mt;
        resc = true;
      }
      // P (bf16 pairs) in place, row sum of this half
      float psum = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float p0 = ex2(__uint_as_float(r[2 * e]) - m_new);
        const float p1 = ex2(__uint_as_float(r[2 * e + 1]) - m_new);
        psum += p0 + p1;
        r[e] = pack_bf16x2(p0, p1);
      }
      // P's TMEM columns and O are free once O += P(j-1) V(j-1) is done
      if (j >= 1) {
        const int jp = j - 1;
        if (!warp_wait(bar(BAR_O_DONE + (jp & 1)), (jp >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
      }
      if (resc) {
        const float alpha = exp2f(m_run - m_new);
        l_run *= alpha;
      }
      if (__any_sync(0xffffffffu, resc)) {
        const float alpha = resc ? exp2f(m_run - m_new) : 1.0f;
        for (int c = 0; c < 4; ++c) {
          uint32_t v[16];
          tmem_ld16(tl + kColO + 64 * hf + 16 * c, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tmem_st16(tl + kColO + 64 * hf + 16 * c, v);
        }
      }
      m_run = m_new;
      l_run += psum;
#pragma unroll
      for (int c = 0; c < 2; ++c)
        tmem_st16(tl + kColP + 32 * hf + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&r[16 * c]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_P_FULL));
    }
    if (ok) {
      // ---- epilogue: O / l -> out rows, lse
      const int jl = ntiles - 1;
      ok = warp_wait(bar(BAR_O_DONE + (jl & 1)), (jl >> 1) & 1);
      if (ok) {
        tc_fence_after();
        pair_sync();
        if (hf == 1) lsum[row] = l_run;
        pair_sync();
        const float l = hf == 0 ? l_run + lsum[row] : 0.f;
        pair_sync();
        if (hf == 0) lsum[row] = l;
        pair_sync();
        const float lt = lsum[row];
        const float inv = lt > 0.f ? 1.0f / lt : 0.f;
        const bool live = row < n_q;
        const int64_t orow = ((int64_t)(r0 + row) * p.h + s) * 128 + 64 * hf;
        for (int c = 0; c < 4; ++c) {
          uint32_t v[16];
          tmem_ld16(tl + kColO + 64 * hf + 16 * c, v);
          tmem_wait_ld();
          if (live) {
            if (p.out_dtype == MLA_F32) {
              float* o = static_cast<float*>(p.out) + orow + 16 * c;
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4)
                *reinterpret_cast<float4*>(o + 4 * q4) =
                    make_float4(__uint_as_float(v[4 * q4]) * inv, __uint_as_float(v[4 * q4 + 1]) * inv,
                                __uint_as_float(v[4 * q4 + 2]) * inv, __uint_as_float(v[4 * q4 + 3]) * inv);
            } else {
              uint16_t* o = static_cast<uint16_t*>(p.out) + orow + 16 * c;
              uint32_t w[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv);
              *reinterpret_cast<uint4*>(o) = make_uint4(w[0], w[1], w[2], w[3]);
              *reinterpret_cast<uint4*>(o + 8) = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
        }
        if (live && hf == 0 && p.lse != nullptr)
          p.lse[(int64_t)(r0 + row) * p.h + s] = lt > 0.f ? (m_run + log2f(lt)) * kLn2 : -INFINITY;
      }
    }
    if (!ok) {
      fail();
      // the partner warp of this lane quarter may wait at a pair meeting
      asm volatile("bar.arrive %0, 64;" ::"r"(1 + sub) : "memory");
      asm volatile("bar.arrive %0, 64;" ::"r"(1 + sub) : "memory");
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

bool encode_bf16(CUtensorMap* m, int rank, const void* base, const cuuint64_t* dims,
                 const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// q[t, s, 0:128] = q_nope[t, s, :]; q[t, s, 128 + 2i .. +1] = RoPE of the pair
// (2i, 2i+1) of q_rope[t, s, :] at the token's position in its sequence.
struct InvFreq64 {
  double v[32];
};

__global__ void __launch_bounds__(256)
prefill_query_kernel(const uint16_t* __restrict__ q_nope, const uint16_t* __restrict__ q_rope,
                     const int32_t* __restrict__ cu, int h, uint16_t* __restrict__ q,
                     const __grid_constant__ InvFreq64 f) {
  const int b = blockIdx.y;
  const int row0 = cu[b], L = cu[b + 1] - row0;
  const int t = blockIdx.x;                 // position in the sequence
  if (t >= L) return;
  const int64_t row = row0 + t;
  for (int i = threadIdx.x; i < h * 64; i += 256) {
    const int s = i / 64, d = i % 64;       // two nope elements per item
    const int64_t src = (row * h + s) * 128 + 2 * d;
    const int64_t dst = (row * h + s) * 192 + 2 * d;
    *reinterpret_cast<uint32_t*>(q + dst) = *reinterpret_cast<const uint32_t*>(q_nope + src);
  }
  for (int i = threadIdx.x; i < h * 32; i += 256) {
    const int s = i / 32, pr = i % 32;
    float cs, sn;
    rope_cos_sin((double)t, f.v[pr], &cs, &sn);
    const int64_t src = (row * h + s) * 64 + 2 * pr;
    const float x0 = bf16_to_f32(q_rope[src]), x1 = bf16_to_f32(q_rope[src + 1]);
    const int64_t dst = (row * h + s) * 192 + 128 + 2 * pr;
    q[dst] = f32_to_bf16_rn(x0 * cs - x1 * sn);
    q[dst + 1] = f32_to_bf16_rn(x0 * sn + x1 * cs);
  }
}

}  // namespace

cudaError_t launch_prefill_tc(const void* q, const void* k_nope, const void* k_rope,
                              const void* v, const int32_t* cu_seqlens, int B, int max_len,
                              int h, int64_t total_rows, float scale, void* out, int out_dtype,
                              float* lse, int32_t* status, cudaStream_t s) {
  CUtensorMap tq, tkn, tkr, tv;
  const cuuint64_t T = (cuuint64_t)total_rows;
  cuuint64_t qd[3] = {192, (cuuint64_t)h, T}, qs[2] = {192 * 2, (cuuint64_t)h * 192 * 2};
  cuuint64_t nd[3] = {128, (cuuint64_t)h, T}, ns[2] = {128 * 2, (cuuint64_t)h * 128 * 2};
  cuuint64_t rd[2] = {64, T}, rs[1] = {64 * 2};
  cuuint32_t box3[3] = {64, 1, 128}, box2[2] = {64, 128};
  if (!encode_bf16(&tq, 3, q, qd, qs, box3) || !encode_bf16(&tkn, 3, k_nope, nd, ns, box3) ||
      !encode_bf16(&tkr, 2, k_rope, rd, rs, box2) || !encode_bf16(&tv, 3, v, nd, ns, box3))
    return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int r = device_registry().once(dev, kSetupPrefill, []() {
    return (int)cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemAlloc);
  });
  if (r != 0) return r < 0 ? cudaErrorInvalidDevice : (cudaError_t)r;
  PrefillParams p{cu_seqlens, out, out_dtype, lse, h, scale * 1.4426950408889634f, status,
                  4000000000LL};
  dim3 grid(ceil_div(max_len, kTile), h, B);
  prefill_tc_kernel<<<grid, kThreads, kSmemAlloc, s>>>(tq, tkn, tkr, tv, p);
  return cudaGetLastError();
}

cudaError_t launch_prefill_query(const void* q_nope, const void* q_rope, const int32_t* cu_seqlens,
                                 int B, int max_len, int h, double theta, void* q, cudaStream_t s) {
  InvFreq64 f;
  for (int i = 0; i < 32; ++i) f.v[i] = pow(theta, -2.0 * (double)i / 64.0);
  dim3 grid(max_len, B);
  prefill_query_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(q_nope),
                                            static_cast<const uint16_t*>(q_rope), cu_seqlens, h,
                                            static_cast<uint16_t*>(q), f);
  return cudaGetLastError();
}

}  // namespace mla
