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
// One CTA per (128-query tile, head, sequence), 576 threads:
//   warp 0      TMA: K tiles of 128 keys (k_nope 2 boxes + the shared RoPE key
//               1 box, 48 KB) into a ring of 3 stages, running two tiles ahead
//               of the V tiles (2 boxes, 32 KB) in a ring of 2;
//   warp 1      MMA issuer: S(j) = Q K(j)^T (12 K=16 steps with the query in
//               TMEM, M = 128 queries, N = 128 keys) into S buffer j % 2, and
//               O += P(j) V(j) (8 steps, P from TMEM, V as an MN-major operand),
//               in the order S(0), S(1), PV(0), S(2), PV(1), S(3), ...;
//   warps 2..17 load the query tile into TMEM, then run the softmax: four warps
//               per TMEM lane quarter split a row's 128 scores (32 each); online
//               softmax with a lazily rescaled O (only when the maximum grows by
//               more than kTau, log2 units).
// TMEM columns: query (bf16 pairs) [0, 96), S x 2 [128, 384), O [384, 512).
// P(j) (bf16 pairs, 64 columns) is written over the first half of S buffer
// j % 2 once the whole row's scores are in registers; the MMAs of one issuing
// thread run in issue order, so S(j+2) overwrites P(j) only after O += P(j) V(j)
// has read it.  With the query in TMEM each score MMA reads only the key tile
// from shared memory.  Key tiles past the query tile are skipped; the diagonal
// tile is masked to keys i <= t.  Every wait is bounded; a timeout is written
// to the status word and the kernel winds down.
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

constexpr int kTile = 128;                  // queries per CTA and keys per key tile
constexpr int kBox = 128 * 128;             // 128 rows x 64 bf16, 128-byte swizzle (16 KB)
constexpr int kKBytes = 3 * kBox;           // 128 nope dims + 64 RoPE dims
constexpr int kVBytes = 2 * kBox;           // 128 dims
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kQuarterWarps = 4;            // softmax warps per TMEM lane quarter
constexpr int kSoftWarps = 4 * kQuarterWarps;
constexpr int kCols = kTile / kQuarterWarps;  // score columns per softmax thread
constexpr int kThreads = 64 + 32 * kSoftWarps;
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKStages * kKBytes;
constexpr int kOffHm = kOffV + kVStages * kVBytes;   // [2][kQuarterWarps][128] float
constexpr int kOffBar = kOffHm + 2 * kQuarterWarps * 128 * 4;
constexpr int kNumBars = 24;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 32;
constexpr int kSmemAlloc = kSmemBytes + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory budget");

constexpr uint32_t kColQ = 0;      // 96 columns
constexpr uint32_t kColS = 128;    // [2] 128 columns each; P(j) over the first 64 of buffer j % 2
constexpr uint32_t kColO = 384;
constexpr uint32_t kTmemCols = 512;

// waits on the critical path poll with test_wait (a suspended try_wait can
// resume hundreds of cycles after the phase completes)
constexpr float kTau = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

enum {
  BAR_Q_READY = 0,                      // softmax warps stored the query tile in TMEM
  BAR_K_FULL = 1,                       // [kKStages] TMA -> MMA
  BAR_K_EMPTY = BAR_K_FULL + kKStages,  // [kKStages] MMA -> TMA
  BAR_V_FULL = BAR_K_EMPTY + kKStages,  // [kVStages]
  BAR_V_EMPTY = BAR_V_FULL + kVStages,  // [kVStages]
  BAR_S_FULL = BAR_V_EMPTY + kVStages,  // [2] S(j) written into buffer j % 2
  BAR_P_FULL = BAR_S_FULL + 2,          // [2] softmax warps stored P(j) (by j % 2)
  BAR_O_DONE = BAR_P_FULL + 2,          // O += P(j) V(j) done (one phase per key tile)
  BAR_DRAIN = BAR_O_DONE + 1,
  BAR_COUNT = BAR_DRAIN + 1,
};
static_assert(BAR_COUNT <= kNumBars, "barrier array");

struct PrefillParams {
  const uint16_t* q;  // [T, h, 192] bf16
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
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_kn, const __grid_constant__ CUtensorMap tm_kr,
                  const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // the longest CTAs (last query tiles: most key tiles) are launched first
  const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;
  const int s = blockIdx.y, b = blockIdx.z;
  const int row_begin = p.cu_seqlens[b];
  const int L = p.cu_seqlens[b + 1] - row_begin;
  const int q0 = qt * kTile;               // first query position of this CTA
  if (q0 >= L) return;                     // uniform for the whole CTA
  const int n = qt + 1;                    // key tiles 0 .. qt (causal)

  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8 * i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_Q_READY), 12);     // the warps of column quarters 0..2
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(bar(BAR_K_FULL + i), 1);
      mbar_init(bar(BAR_K_EMPTY + i), 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(bar(BAR_V_FULL + i), 1);
      mbar_init(bar(BAR_V_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(BAR_S_FULL + i), 1);
      mbar_init(bar(BAR_P_FULL + i), kSoftWarps);
    }
    mbar_init(bar(BAR_O_DONE), 1);
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
  auto warp_spin = [&](uint32_t bb, uint32_t parity) -> bool {
    bool ok = true;
    if (lane == 0) ok = mbar_spin_or_abort(bb, parity, lim, abort_flag, &timed_out);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // order K(0), K(1), then K(j+2), V(j): the issuer needs K two tiles ahead
    if (lane == 0) {
      int nk = 0, nv = 0;
      bool ok = true;
      auto load_k = [&](int j) -> bool {
        const int st = j % kKStages;
        if (j >= kKStages && !mbar_wait_or_abort(bar(BAR_K_EMPTY + st), ((j / kKStages) - 1) & 1,
                                                 lim, abort_flag, &timed_out))
          return false;
        const uint32_t dst = sbase + kOffK + st * kKBytes;
        const int kr = row_begin + j * kTile;
        mbar_arrive_expect_tx(bar(BAR_K_FULL + st), kKBytes);
        tma_load_3d(dst, &tm_kn, 0, s, kr, bar(BAR_K_FULL + st));
        tma_load_3d(dst + kBox, &tm_kn, 64, s, kr, bar(BAR_K_FULL + st));
        tma_load_2d(dst + 2 * kBox, &tm_kr, 0, kr, bar(BAR_K_FULL + st));
        ++nk;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int st = j % kVStages;
        if (j >= kVStages && !mbar_wait_or_abort(bar(BAR_V_EMPTY + st), ((j / kVStages) - 1) & 1,
                                                 lim, abort_flag, &timed_out))
          return false;
        const uint32_t dst = sbase + kOffV + st * kVBytes;
        const int kr = row_begin + j * kTile;
        mbar_arrive_expect_tx(bar(BAR_V_FULL + st), kVBytes);
        tma_load_3d(dst, &tm_v, 0, s, kr, bar(BAR_V_FULL + st));
        tma_load_3d(dst + kBox, &tm_v, 64, s, kr, bar(BAR_V_FULL + st));
        ++nv;
        return true;
      };
      for (int j = 0; j < 2 && j < n && ok; ++j) ok = load_k(j);
      for (int j = 0; j < n && ok; ++j) {
        if (j + 2 < n && !(ok = load_k(j + 2))) break;
        ok = load_v(j);
      }
      if (!ok) fail();
      // every issued copy lands before the CTA may leave
      int never = 0;
      bool dummy = false;
      for (int st = 0; st < kKStages; ++st) {
        const int c = (nk - st + kKStages - 1) / kKStages;   // loads into stage st
        if (c > 0) mbar_wait_or_abort(bar(BAR_K_FULL + st), (c - 1) & 1, lim, &never, &dummy);
      }
      for (int st = 0; st < kVStages; ++st) {
        const int c = (nv - st + kVStages - 1) / kVStages;
        if (c > 0) mbar_wait_or_abort(bar(BAR_V_FULL + st), (c - 1) & 1, lim, &never, &dummy);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // one thread runs the whole loop: a warp-wide loop (the other lanes waiting
    // at warp reconvergence and a broadcast after every wait) was measured to
    // add several hundred cycles per key tile to the MMA issue
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      const uint32_t idO = idesc_bf16_f32(128, 128, false, true);
      auto wait = [&](uint32_t bb, uint32_t parity) -> bool {
        return mbar_spin_or_abort(bb, parity, lim, abort_flag, &timed_out);
      };
      auto issue_s = [&](int j) -> bool {
        const int st = j % kKStages;
        if (!wait(bar(BAR_K_FULL + st), (j / kKStages) & 1)) return false;
        tc_fence_after();
        const uint32_t k_st = sbase + kOffK + st * kKBytes;
        const uint32_t d = tmem + kColS + 128 * (j & 1);
#pragma unroll
        for (int kk = 0; kk < 12; ++kk) {
          const uint64_t bd = smem_desc(k_st + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024,
                                        kSwizzle128B);
          mma_ts(d, tmem + kColQ + 8 * kk, bd, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(BAR_S_FULL + (j & 1)));
        mma_commit(bar(BAR_K_EMPTY + st));
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        const int st = j % kVStages;
        if (!wait(bar(BAR_V_FULL + st), (j / kVStages) & 1)) return false;
        if (!wait(bar(BAR_P_FULL + (j & 1)), (j >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t v_st = sbase + kOffV + st * kVBytes;
        const uint32_t a = tmem + kColS + 128 * (j & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = smem_desc(v_st + kk * 2048, kBox, 1024, kSwizzle128B);
          mma_ts(tmem + kColO, a + 8 * kk, bd, idO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(BAR_O_DONE));
        mma_commit(bar(BAR_V_EMPTY + st));
        return true;
      };
      bool ok = wait(bar(BAR_Q_READY), 0);
      for (int j = 0; ok && j < 2 && j < n; ++j) ok = issue_s(j);
      for (int j = 0; ok && j < n; ++j) {
        if (!(ok = issue_pv(j))) break;
        if (j + 2 < n) ok = issue_s(j + 2);
      }
      if (!ok) fail();
      mma_commit(bar(BAR_DRAIN));
      int never = 0;
      bool dummy = false;
      mbar_wait_or_abort(bar(BAR_DRAIN), 0, lim, &never, &dummy);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int w = warp - 2;                // 0..15
    const int cq = w >> 2;                 // column quarter: keys [32 cq, 32 cq + 32)
    const int sub = warp & 3;              // TMEM lane quarter
    const int row = sub * 32 + lane;       // query row of the tile
    const int qpos = q0 + row;
    const bool live = qpos < L;
    const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16);
    float* hm = reinterpret_cast<float*>(smem + kOffHm);   // [2][kQuarterWarps][128]
    const int barid = 1 + sub;
    auto quarter_sync = [&]() {
      asm volatile("bar.sync %0, %1;" ::"r"(barid), "r"(32 * kQuarterWarps) : "memory");
    };
    bool ok = true;

    // ---- the query row into TMEM: warps of column quarter cq < 3 store dims
    //      [64 cq, 64 cq + 64) as bf16 pairs at columns [32 cq, 32 cq + 32)
    if (cq < 3) {
      uint32_t qv[32];
      if (live) {
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + ((int64_t)(row_begin + qpos) * p.h + s) * 192 + 64 * cq);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = src[i];
          qv[4 * i] = v.x;
          qv[4 * i + 1] = v.y;
          qv[4 * i + 2] = v.z;
          qv[4 * i + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) qv[i] = 0u;
      }
      tmem_st16(tl + kColQ + 32 * cq, *reinterpret_cast<uint32_t(*)[16]>(&qv[0]));
      tmem_st16(tl + kColQ + 32 * cq + 16, *reinterpret_cast<uint32_t(*)[16]>(&qv[16]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_Q_READY));
    }

    const float sl2 = p.scale_log2;
    float m_run = -INFINITY;   // running row maximum of the raw scores
    float l_run = 0.f;         // this thread's share of the row sum
    for (int j = 0; j < n && ok; ++j) {
      const int sb = j & 1;
      if (!warp_spin(bar(BAR_S_FULL + sb), (j >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      uint32_t r[kCols];
      tmem_ld16(tl + kColS + 128 * sb + 32 * cq, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
      tmem_ld16(tl + kColS + 128 * sb + 32 * cq + 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16]));
      tmem_wait_ld();
      // raw-score maximum (the scale is positive); the diagonal tile sees keys i <= t only
      if (j == qt) {
#pragma unroll
        for (int kk = 0; kk < kCols; ++kk)
          if (32 * cq + kk > row) r[kk] = __float_as_uint(-INFINITY);
      }
      // four independent chains, then a tree (the maximum is exact in any order)
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int kk = 0; kk < kCols; ++kk) m4[kk & 3] = fmaxf(m4[kk & 3], __uint_as_float(r[kk]));
      float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      // the four quarters of the row meet (buffer j % 2, so one meeting per tile)
      float* hmb = hm + sb * kQuarterWarps * 128;
      hmb[cq * 128 + row] = mt;
      quarter_sync();
#pragma unroll
      for (int c = 0; c < kQuarterWarps; ++c) mt = fmaxf(mt, hmb[c * 128 + row]);
      float m_new = m_run;
      bool resc = false;
      if (m_run == -INFINITY) {
        m_new = mt;
      } else if ((mt - m_run) * sl2 > kTau) {
        m_new = mt;
        resc = true;
      }
      const float mb = m_new * sl2;
      // P = 2^(x * scale_log2 - m * scale_log2) as bf16 pairs, row sum share
      float ps4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < kCols / 2; ++e) {
        const float p0 = ex2(fmaf(__uint_as_float(r[2 * e]), sl2, -mb));
        const float p1 = ex2(fmaf(__uint_as_float(r[2 * e + 1]), sl2, -mb));
        ps4[e & 3] += p0 + p1;
        r[e] = pack_bf16x2(p0, p1);
      }
      const float psum = (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
      if (__any_sync(0xffffffffu, resc)) {
        // O must hold P(j-1) V(j-1) before it is rescaled
        if (j >= 1) {
          if (!warp_wait(bar(BAR_O_DONE), (j - 1) & 1)) { ok = false; break; }
          tc_fence_after();
        }
        const float alpha = resc ? ex2((m_run - m_new) * sl2) : 1.0f;
        for (int c = 0; c < kCols / 16; ++c) {
          uint32_t v[16];
          tmem_ld16(tl + kColO + 32 * cq + 16 * c, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tmem_st16(tl + kColO + 32 * cq + 16 * c, v);
        }
        if (resc) l_run *= alpha;
      }
      m_run = m_new;
      l_run += psum;
      // P(j) over the first half of S buffer j % 2: every quarter of the row has
      // read its scores (they met above)
      tmem_st16(tl + kColS + 128 * sb + 16 * cq, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_P_FULL + sb));
    }
    if (ok) {
      // ---- epilogue: O / l -> out rows, lse
      ok = warp_wait(bar(BAR_O_DONE), (n - 1) & 1);
      if (ok) {
        tc_fence_after();
        float* hmb = hm + (n & 1) * kQuarterWarps * 128;
        hmb[cq * 128 + row] = l_run;
        quarter_sync();
        float lt = 0.f;
#pragma unroll
        for (int c = 0; c < kQuarterWarps; ++c) lt += hmb[c * 128 + row];
        const float inv = lt > 0.f ? 1.0f / lt : 0.f;
        const int64_t orow = ((int64_t)(row_begin + qpos) * p.h + s) * 128 + 32 * cq;
        for (int c = 0; c < kCols / 16; ++c) {
          uint32_t v[16];
          tmem_ld16(tl + kColO + 32 * cq + 16 * c, v);
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
              uint32_t w8[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                w8[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv);
              *reinterpret_cast<uint4*>(o) = make_uint4(w8[0], w8[1], w8[2], w8[3]);
              *reinterpret_cast<uint4*>(o + 8) = make_uint4(w8[4], w8[5], w8[6], w8[7]);
            }
          }
        }
        if (live && cq == 0 && p.lse != nullptr)
          p.lse[(int64_t)(row_begin + qpos) * p.h + s] =
              lt > 0.f ? (m_run * sl2 + log2f(lt)) * kLn2 : -INFINITY;
      }
    }
    if (!ok) {
      fail();
      // the other warps of this lane quarter may wait at a quarter meeting
      asm volatile("bar.arrive %0, %1;" ::"r"(barid), "r"(32 * kQuarterWarps) : "memory");
      asm volatile("bar.arrive %0, %1;" ::"r"(barid), "r"(32 * kQuarterWarps) : "memory");
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
  CUtensorMap tkn, tkr, tv;
  const cuuint64_t T = (cuuint64_t)total_rows;
  cuuint64_t nd[3] = {128, (cuuint64_t)h, T}, ns[2] = {128 * 2, (cuuint64_t)h * 128 * 2};
  cuuint64_t rd[2] = {64, T}, rs[1] = {64 * 2};
  cuuint32_t box3[3] = {64, 1, 128}, box2[2] = {64, 128};
  if (!encode_bf16(&tkn, 3, k_nope, nd, ns, box3) || !encode_bf16(&tkr, 2, k_rope, rd, rs, box2) ||
      !encode_bf16(&tv, 3, v, nd, ns, box3))
    return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int r = device_registry().once(dev, kSetupPrefill, []() {
    return (int)cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemAlloc);
  });
  if (r != 0) return r < 0 ? cudaErrorInvalidDevice : (cudaError_t)r;
  PrefillParams p{static_cast<const uint16_t*>(q), cu_seqlens, out, out_dtype, lse, h,
                  scale * 1.4426950408889634f, status, 4000000000LL};
  dim3 grid(ceil_div(max_len, kTile), h, B);
  prefill_tc_kernel<<<grid, kThreads, kSmemAlloc, s>>>(tkn, tkr, tv, p);
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
