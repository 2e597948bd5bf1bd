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
// One CTA per (256 queries, head, sequence): two query tiles of 128 rows, A
// (the first 128) and B (the next), 576 threads:
//   warp 0      TMA: both query tiles once (3 boxes of 64 dims x 128 tokens
//               each), then per key tile of 128 tokens the K boxes (k_nope 2 +
//               the shared RoPE key 1) and the V boxes (2) into a ring of 8
//               slots of 16 KB (a V tile takes two neighbouring slots);
//   warp 1      MMA issuer: S_t(j) = Q_t K(j)^T (12 K=16 steps, M = 128
//               queries, N = 128 keys) and O_t += P_t(j) V(j) (8 steps, P from
//               TMEM, V as an MN-major operand), in the order PV_A(j),
//               S_A(j+1), PV_B(j), S_B(j+1): while one tile's softmax runs, the
//               tensor cores work on the other tile;
//   warps 2..17 softmax, 8 warps per query tile: two warps per TMEM lane
//               quarter split a row's 128 scores (64 each); online softmax
//               with a lazily rescaled O (only when the maximum grows by more
//               than kTau, log2 units).
// TMEM columns: tile t holds S_t at [256 t, 256 t + 128) and O_t at
// [256 t + 128, 256 t + 256); P_t (bf16 pairs, 64 columns) is written over
// the first half of S_t once the scores are in registers.  The MMAs of one
// issuing thread run in issue order, so S_t(j+1) overwrites P_t(j) only after
// O_t += P_t(j) V(j) has read it.  Key tiles past a query tile are skipped; the
// diagonal tile is masked to keys i <= t.  Every wait is bounded; a timeout
// is written to the status word and the kernel winds down.
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

constexpr int kTile = 128;                  // queries per tile and keys per key tile
constexpr int kQTiles = 2;                  // query tiles per CTA
constexpr int kBox = 128 * 128;             // 128 rows x 64 bf16, 128-byte swizzle (16 KB)
constexpr int kQBytes = 3 * kBox;           // one query tile, 192 dims
constexpr int kSlots = 8;                   // K/V ring slots of one box each
constexpr int kSoftWarps = 8;               // per query tile
constexpr int kThreads = 64 + 32 * kSoftWarps * kQTiles;
constexpr int kOffQ = 0;                    // [kQTiles] query tiles
constexpr int kOffRing = kOffQ + kQTiles * kQBytes;
constexpr int kOffHm = kOffRing + kSlots * kBox;   // [kQTiles][128] float: row max / row sum meeting
constexpr int kOffBar = kOffHm + kQTiles * 128 * 4;
constexpr int kNumBars = 32;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 32;
constexpr int kSmemAlloc = kSmemBytes + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory budget");

constexpr uint32_t kTmemCols = 512;        // tile t: S_t / P_t at 256 t, O_t at 256 t + 128

constexpr float kTau = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

enum {
  BAR_Q_FULL = 0,
  BAR_FULL = 1,                         // [kSlots] TMA -> MMA
  BAR_EMPTY = BAR_FULL + kSlots,        // [kSlots] MMA -> TMA
  BAR_S_FULL = BAR_EMPTY + kSlots,      // [kQTiles] S_t(j) written
  BAR_P_FULL = BAR_S_FULL + kQTiles,    // [kQTiles] softmax warps of tile t stored P_t(j)
  BAR_O_DONE = BAR_P_FULL + kQTiles,    // [kQTiles] last O_t += P_t V done
  BAR_DRAIN = BAR_O_DONE + kQTiles,
  BAR_COUNT = BAR_DRAIN + 1,
};
static_assert(BAR_COUNT <= kNumBars, "barrier array");

// Slot sequence of the K/V ring, walked identically by the TMA producer and
// the MMA issuer: per key tile three single slots (K) and one pair of
// neighbouring slots (V; a pair never starts on the last slot, which is then
// skipped).  phase bit s = parity of slot s's fills so far, used bit s = slot
// s filled before (its refill waits for the previous use to end).
struct Ring {
  int pos = 0;
  uint32_t phase = 0, used = 0;
  __device__ __forceinline__ int next(bool pair) {
    int s = pos % kSlots;
    if (pair && s == kSlots - 1) {
      ++pos;
      s = 0;
    }
    pos += pair ? 2 : 1;
    return s;
  }
  __device__ __forceinline__ uint32_t parity(int s) const { return (phase >> s) & 1u; }
  __device__ __forceinline__ bool was_used(int s) const { return (used >> s) & 1u; }
  __device__ __forceinline__ void advance(int s) {
    phase ^= 1u << s;
    used |= 1u << s;
  }
};

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
  // the longest CTAs (last query tiles: most key tiles) are launched first
  const int m = (int)gridDim.x - 1 - (int)blockIdx.x;
  const int s = blockIdx.y, b = blockIdx.z;
  const int row_begin = p.cu_seqlens[b];
  const int L = p.cu_seqlens[b + 1] - row_begin;
  const int q0 = m * kQTiles * kTile;      // first query position of this CTA
  if (q0 >= L) return;                     // uniform for the whole CTA
  // key tiles of query tile t: 0 .. 2m + t (causal); tile B may be past the end
  const int ntk0 = kQTiles * m + 1;
  const int ntk1 = q0 + kTile < L ? kQTiles * m + 2 : 0;
  auto ntk = [&](int t) { return t == 0 ? ntk0 : ntk1; };
  const int nkt = ntk1 > ntk0 ? ntk1 : ntk0;

  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8 * i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_Q_FULL), 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(bar(BAR_FULL + i), 1);
      mbar_init(bar(BAR_EMPTY + i), 1);
    }
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(bar(BAR_S_FULL + t), 1);
      mbar_init(bar(BAR_P_FULL + t), kSoftWarps);
      mbar_init(bar(BAR_O_DONE + t), 1);
    }
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
  const uint32_t ring = sbase + kOffRing;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const int r0 = row_begin + q0;
      mbar_arrive_expect_tx(bar(BAR_Q_FULL), kQTiles * kQBytes);
      for (int t = 0; t < kQTiles; ++t)
        for (int c = 0; c < 3; ++c)
          tma_load_3d(sbase + kOffQ + t * kQBytes + c * kBox, &tm_q, 64 * c, s, r0 + t * kTile,
                      bar(BAR_Q_FULL));
      Ring rg;
      bool ok = true;
      auto fill = [&](int slot) -> bool {
        if (rg.was_used(slot) && !mbar_wait_or_abort(bar(BAR_EMPTY + slot), rg.parity(slot) ^ 1u,
                                                     lim, abort_flag, &timed_out))
          return false;
        mbar_arrive_expect_tx(bar(BAR_FULL + slot), kBox);
        return true;
      };
      for (int j = 0; ok && j < nkt; ++j) {
        const int kr = row_begin + j * kTile;   // global row of key 0 of tile j
        for (int c = 0; c < 3 && ok; ++c) {
          const int sl = rg.next(false);
          if (!(ok = fill(sl))) break;
          if (c < 2)
            tma_load_3d(ring + sl * kBox, &tm_kn, 64 * c, s, kr, bar(BAR_FULL + sl));
          else
            tma_load_2d(ring + sl * kBox, &tm_kr, 0, kr, bar(BAR_FULL + sl));
          rg.advance(sl);
        }
        if (!ok) break;
        const int sv = rg.next(true);
        for (int c = 0; c < 2 && ok; ++c) {
          if (!(ok = fill(sv + c))) break;
          tma_load_3d(ring + (sv + c) * kBox, &tm_v, 64 * c, s, kr, bar(BAR_FULL + sv + c));
          rg.advance(sv + c);
        }
      }
      if (!ok) fail();
      // every issued copy lands before the CTA may leave
      int never = 0;
      bool dummy = false;
      mbar_wait_or_abort(bar(BAR_Q_FULL), 0, lim, &never, &dummy);
      for (int sl = 0; sl < kSlots; ++sl)
        if (rg.was_used(sl))
          mbar_wait_or_abort(bar(BAR_FULL + sl), rg.parity(sl) ^ 1u, lim, &never, &dummy);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idS = idesc_bf16_f32(128, 128, false, false);
    const uint32_t idO = idesc_bf16_f32(128, 128, false, true);
    Ring rg;
    int ks0 = 0, ks1 = 0, ks2 = 0, sv = 0;
    auto ks = [&](int c) { return c == 0 ? ks0 : (c == 1 ? ks1 : ks2); };
    bool ok = warp_wait(bar(BAR_Q_FULL), 0);
    auto acquire_k = [&]() -> bool {
      ks0 = rg.next(false);
      ks1 = rg.next(false);
      ks2 = rg.next(false);
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        if (!warp_wait(bar(BAR_FULL + ks(c)), rg.parity(ks(c)))) return false;
        rg.advance(ks(c));
      }
      return true;
    };
    auto acquire_v = [&]() -> bool {
      sv = rg.next(true);
      for (int c = 0; c < 2; ++c) {
        if (!warp_wait(bar(BAR_FULL + sv + c), rg.parity(sv + c))) return false;
        rg.advance(sv + c);
      }
      return true;
    };
    auto release = [&](int sl) {
      if (lane == 0) mma_commit(bar(BAR_EMPTY + sl));
    };
    auto issue_s = [&](int t) {
      tc_fence_after();
      if (lane == 0) {
        const uint32_t q_t = sbase + kOffQ + t * kQBytes;
#pragma unroll
        for (int kk = 0; kk < 12; ++kk) {
          const uint32_t off = (kk & 3) * 32;
          const uint64_t ad = smem_desc(q_t + (kk >> 2) * kBox + off, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(ring + ks(kk >> 2) * kBox + off, 16, 1024, kSwizzle128B);
          mma_ss(tmem + 256 * t, ad, bd, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(BAR_S_FULL + t));
      }
      __syncwarp();
    };
    auto issue_pv = [&](int t, int j) -> bool {
      if (!warp_wait(bar(BAR_P_FULL + t), j & 1)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t v_st = ring + sv * kBox;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = smem_desc(v_st + kk * 2048, kBox, 1024, kSwizzle128B);
          mma_ts(tmem + 256 * t + 128, tmem + 256 * t + 8 * kk, bd, idO,
                 (j > 0 || kk > 0) ? 1u : 0u);
        }
        if (j == ntk(t) - 1) mma_commit(bar(BAR_O_DONE + t));
      }
      __syncwarp();
      return true;
    };
    if (ok) ok = acquire_k();
    if (ok) {
      for (int t = 0; t < kQTiles; ++t)
        if (ntk(t) > 0) issue_s(t);
      for (int c = 0; c < 3; ++c) release(ks(c));
    }
    for (int j = 0; ok && j < nkt; ++j) {
      if (!(ok = acquire_v())) break;
      const bool more = j + 1 < nkt;
      bool have_k = false;
      for (int t = 0; t < kQTiles && ok; ++t) {
        if (j < ntk(t) && !(ok = issue_pv(t, j))) break;
        if (j + 1 < ntk(t)) {
          if (!have_k) {
            if (!(ok = acquire_k())) break;
            have_k = true;
          }
          issue_s(t);
        }
      }
      if (!ok) break;
      for (int c = 0; c < 2; ++c) release(sv + c);
      if (more && have_k)
        for (int c = 0; c < 3; ++c) release(ks(c));
    }
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
    const int w = warp - 2;               // 0..15
    const int t = w / kSoftWarps;         // query tile
    const int hf = (w % kSoftWarps) >> 2; // column half: keys [64 hf, 64 hf + 64)
    const int sub = warp & 3;             // TMEM lane quarter
    const int row = sub * 32 + lane;      // query row of the tile
    const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16);
    const uint32_t colS = 256 * t, colO = 256 * t + 128;
    float* hm = reinterpret_cast<float*>(smem + kOffHm) + t * 128;
    const int barid = 1 + t * 4 + sub;
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(barid) : "memory"); };
    // the two halves of a row meet in hm[row]: half 1 writes, half 0 combines
    // and writes back, half 1 reads (two meetings)
    auto meet = [&](float v, bool is_max) -> float {
      if (hf == 1) hm[row] = v;
      pair_sync();
      if (hf == 0) {
        v = is_max ? fmaxf(v, hm[row]) : v + hm[row];
        hm[row] = v;
      }
      pair_sync();
      if (hf == 1) v = hm[row];
      return v;
    };
    const int n = ntk(t);
    const int qt_diag = kQTiles * m + t;  // key tile on the diagonal
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n && ok; ++j) {
      if (!warp_wait(bar(BAR_S_FULL + t), j & 1)) { ok = false; break; }
      tc_fence_after();
      uint32_t r[64];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_ld16(tl + colS + 64 * hf + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&r[16 * c]));
      tmem_wait_ld();
      // scores in log2 units; the diagonal tile sees keys i <= t only
      const bool diag = j == qt_diag;
      float mt = -INFINITY;
#pragma unroll
      for (int kk = 0; kk < 64; ++kk) {
        float x = __uint_as_float(r[kk]) * p.scale_log2;
        if (diag && 64 * hf + kk > row) x = -INFINITY;
        r[kk] = __float_as_uint(x);
        mt = fmaxf(mt, x);
      }
      mt = meet(mt, true);
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
      // O_t is final for P_t(j-1) here: S_t(j) was issued after O_t += P_t(j-1) V
      if (resc) l_run *= exp2f(m_run - m_new);
      if (__any_sync(0xffffffffu, resc)) {
        const float alpha = resc ? exp2f(m_run - m_new) : 1.0f;
        for (int c = 0; c < 4; ++c) {
          uint32_t v[16];
          tmem_ld16(tl + colO + 64 * hf + 16 * c, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tmem_st16(tl + colO + 64 * hf + 16 * c, v);
        }
      }
      m_run = m_new;
      l_run += psum;
      // P over the first half of S: both halves of every row have read their
      // scores (they met above)
#pragma unroll
      for (int c = 0; c < 2; ++c)
        tmem_st16(tl + colS + 32 * hf + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&r[16 * c]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_P_FULL + t));
    }
    if (ok && n > 0) {
      // ---- epilogue: O / l -> out rows, lse
      ok = warp_wait(bar(BAR_O_DONE + t), 0);
      if (ok) {
        tc_fence_after();
        const float lt = meet(l_run, false);
        const float inv = lt > 0.f ? 1.0f / lt : 0.f;
        const int qpos = q0 + t * kTile + row;
        const bool live = qpos < L;
        const int64_t orow = ((int64_t)(row_begin + qpos) * p.h + s) * 128 + 64 * hf;
        for (int c = 0; c < 4; ++c) {
          uint32_t v[16];
          tmem_ld16(tl + colO + 64 * hf + 16 * c, v);
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
        if (live && hf == 0 && p.lse != nullptr)
          p.lse[(int64_t)(row_begin + qpos) * p.h + s] =
              lt > 0.f ? (m_run + log2f(lt)) * kLn2 : -INFINITY;
      }
    }
    if (!ok) {
      fail();
      // the partner warp of this lane quarter may wait at a pair meeting
      asm volatile("bar.arrive %0, 64;" ::"r"(barid) : "memory");
      asm volatile("bar.arrive %0, 64;" ::"r"(barid) : "memory");
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
  dim3 grid(ceil_div(max_len, kQTiles * kTile), h, B);
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
