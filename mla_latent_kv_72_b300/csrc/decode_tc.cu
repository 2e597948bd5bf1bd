// mla_decode_fwd, tensor-core kernel for sm_103a (tcgen05 + TMEM + TMA + a
// 2-CTA cluster), bf16 latent cache, d_c = 512, d_r = 64, 64-token blocks,
// up to 128 heads.
//
// What it computes is the decode-time MQA form of MLA (kexue.fm "From MHA,
// MQA, GQA to MLA", eq. mla-mqa): for each head s, scores
// q_cat^(s) . [c_i, k_R,i] over the cached rows, softmax, and the
// probability-weighted sum of the latents c_i.  All heads share each cache
// row, so the score tile S = Q K^T (M = 128 heads, N = 64 tokens, K = 576)
// and the output O += P C (M = 128 heads, N = 512 latent, K = 64 tokens) are
// dense contractions on the tensor cores.
//
// Work split.  One float32 accumulator for 128 heads x 512 latent columns
// fills the whole 512-column tensor memory of an SM, so a pair of CTAs (a
// cluster of 2) shares each (sequence, split) work item:
//   CTA r owns output columns [256 r, 256 r + 256) of the latent (O_r in TMEM)
//   and the matching slice of the 576-d score contraction: CTA 0 the latent
//   columns 0..255 plus the 64 RoPE columns, CTA 1 the latent columns 256..511.
//   Each CTA TMA-loads exactly its own columns of every cache block (the pair
//   reads each byte of the cache once), computes its partial score tile
//   S_r = Q[:, K_r] K[:, K_r]^T, and the two partial tiles are exchanged
//   through distributed shared memory; both CTAs then hold the same
//   S = S_0 + S_1 (float addition commutes, so both run a bit-identical online
//   softmax) and write the same P, which each multiplies into its own O_r.
//
// Roles (192 threads): warp 0 issues TMA loads, warp 1 allocates TMEM and
// issues tcgen05.mma (one elected lane), warps 2..5 (thread = head row)
// load the query into TMEM, run the online softmax and the epilogue.
//
// TMEM columns: O_r [0, 256), S [256, 320), Q_r [320, 320 + 160) as the MMA
// A operand (bf16 pairs).  Every wait is bounded; on a timeout the kernel
// writes MLA_DEV_WAIT_TIMEOUT to the status word and winds down.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int kTok = 64;                    // tokens per tile (= cache block)
constexpr int kStages = 3;
constexpr int kBoxBytes = 64 * 128;         // 64 rows x 64 bf16, 128-byte swizzle
constexpr int kStageBytes = 5 * kBoxBytes;  // CTA 0: 4 latent boxes + the RoPE box
constexpr int kPBytes = 128 * 128;          // P: 128 rows x 64 bf16
constexpr int kRecvBytes = 128 * 64 * 4;    // partial S of the peer, float32

constexpr int kOffStages = 0;
constexpr int kOffP = kOffStages + kStages * kStageBytes;
constexpr int kOffRecv = kOffP + 2 * kPBytes;
constexpr int kOffBar = kOffRecv + kRecvBytes;
constexpr int kNumBars = 16;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16;
constexpr int kSmemAlloc = kSmemBytes + 1024;  // alignment slack

constexpr uint32_t kColO = 0;
constexpr uint32_t kColS = 256;
constexpr uint32_t kColQ = 320;
constexpr uint32_t kTmemCols = 512;

constexpr int kThreads = 192;
constexpr float kTau = 8.0f;  // lazy rescale threshold (log2 units): P stays <= 2^8
constexpr float kLn2 = 0.69314718055994530942f;

// barrier indices
enum {
  BAR_KV_FULL = 0,   // [kStages]
  BAR_KV_EMPTY = 3,  // [kStages]
  BAR_S_FULL = 6,
  BAR_S_EMPTY = 7,
  BAR_P_FULL = 8,    // [2]
  BAR_O_DONE = 10,   // [2]
  BAR_Q_READY = 12,
  BAR_RECV_FULL = 13,
  BAR_RECV_FREE = 14,
  BAR_DRAIN = 15,
};

struct TcParams {
  const uint16_t* q_cat;        // [B, h, 576] bf16
  const int32_t* block_table;   // [B, max_blocks]
  const int32_t* seq_lens;      // [B]
  float* o_part;                // [B, S, h, 512]
  float* lse_part;              // [B, S, h]
  int32_t* status;
  int max_blocks, B, h, num_splits, num_blocks;
  float scale_log2;
  long long wait_limit;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_lat,
                 const __grid_constant__ CUtensorMap tm_rope, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int work = blockIdx.x / 2;
  const int b = work / p.num_splits, j = work % p.num_splits;

  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8 * i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(BAR_KV_FULL + s), 1);
      mbar_init(bar(BAR_KV_EMPTY + s), 1);
    }
    mbar_init(bar(BAR_S_FULL), 1);
    mbar_init(bar(BAR_S_EMPTY), 128);
    mbar_init(bar(BAR_P_FULL + 0), 128);
    mbar_init(bar(BAR_P_FULL + 1), 128);
    mbar_init(bar(BAR_O_DONE + 0), 1);
    mbar_init(bar(BAR_O_DONE + 1), 1);
    mbar_init(bar(BAR_Q_READY), 128);
    mbar_init(bar(BAR_RECV_FULL), 128);
    mbar_init(bar(BAR_RECV_FREE), 128);
    mbar_init(bar(BAR_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_lat);
    prefetch_tmap(&tm_rope);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  int L = p.seq_lens[b];
  if (L > p.max_blocks * kTok) {
    if (threadIdx.x == 0 && rank == 0) set_status(p.status, MLA_DEV_BAD_LENGTH);
    L = p.max_blocks * kTok;
  }
  if (L < 0) L = 0;
  int blo, bhi;
  split_range(ceil_div(L, kTok), p.num_splits, j, &blo, &bhi);
  const int T = bhi - blo;
  const long long lim = p.wait_limit;

  auto fail = [&]() {
    set_status(p.status, MLA_DEV_WAIT_TIMEOUT);
    *abort_flag = 1;
  };

  if (T > 0 && warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t tx = rank == 0 ? 5 * kBoxBytes : 4 * kBoxBytes;
      int issued[kStages] = {0, 0, 0};
      for (int i = 0; i < T; ++i) {
        if (*abort_flag) break;
        const int st = i % kStages;
        if (i >= kStages && !mbar_wait(bar(BAR_KV_EMPTY + st), ((i / kStages) - 1) & 1, lim)) {
          fail();
          break;
        }
        int pb = p.block_table[(int64_t)b * p.max_blocks + blo + i];
        if (pb < 0 || pb >= p.num_blocks) {
          set_status(p.status, MLA_DEV_BAD_BLOCK);
          pb = 0;  // load a valid block instead; the result is flagged as wrong
        }
        const uint32_t dst = sbase + kOffStages + st * kStageBytes;
        const uint32_t fb = bar(BAR_KV_FULL + st);
        mbar_arrive_expect_tx(fb, tx);
        const int y = pb * kTok;
        for (int k = 0; k < 4; ++k)
          tma_load_2d(dst + k * kBoxBytes, &tm_lat, (int)(rank * 4 + k) * 64, y, fb);
        if (rank == 0) tma_load_2d(dst + 4 * kBoxBytes, &tm_rope, 0, y, fb);
        issued[st]++;
      }
      // wait for every issued load to land before the CTA may exit
      for (int st = 0; st < kStages; ++st)
        if (issued[st] > 0) mbar_wait(bar(BAR_KV_FULL + st), (issued[st] - 1) & 1, lim);
    }
  } else if (T > 0 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idS = idesc_bf16_f32(128, 64, false, false);
    const uint32_t idO = idesc_bf16_f32(128, 256, false, true);
    const int nK = rank == 0 ? 20 : 16;     // 16-wide K steps of the partial score
    const int nbox = rank == 0 ? 5 : 4;
    bool ok = __all_sync(0xffffffffu, mbar_wait(bar(BAR_Q_READY), 0, lim));
    if (!ok) fail();
    tc_fence_after();

    auto issue_o = [&](int t) -> bool {
      bool w = __all_sync(0xffffffffu, mbar_wait(bar(BAR_P_FULL + (t & 1)), (t >> 1) & 1, lim));
      if (!w) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t stage = sbase + kOffStages + (t % kStages) * kStageBytes;
        const uint32_t pbuf = sbase + kOffP + (t & 1) * kPBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = smem_desc(pbuf + k * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(stage + k * 2048, kBoxBytes, 1024, kSwizzle128B);
          mma_ss(tmem + kColO, ad, bd, idO, (t > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(bar(BAR_O_DONE + (t & 1)));
        mma_commit(bar(BAR_KV_EMPTY + (t % kStages)));
      }
      __syncwarp();
      return true;
    };

    for (int i = 0; i < T && ok; ++i) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
      const int st = i % kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_KV_FULL + st), (i / kStages) & 1, lim))) {
        ok = false;
        break;
      }
      const uint32_t stage = sbase + kOffStages + st * kStageBytes;
      const int n_valid = min(kTok, L - (blo + i) * kTok);
      if (n_valid < kTok) {
        // slots past the sequence end: zero them so that P = 0 meets finite values
        uint8_t* sp = smem + kOffStages + st * kStageBytes;
        const int nrow = kTok - n_valid;
        for (int e = lane; e < nbox * nrow * 8; e += 32) {
          const int box = e / (nrow * 8), rr = (e / 8) % nrow, ch = e % 8;
          *reinterpret_cast<uint4*>(sp + box * kBoxBytes + (n_valid + rr) * 128 + ch * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (i > 0 &&
          !__all_sync(0xffffffffu, mbar_wait(bar(BAR_S_EMPTY), (i - 1) & 1, lim))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (lane == 0) {
        for (int k = 0; k < nK; ++k) {
          const uint64_t bd = smem_desc(stage + (k >> 2) * kBoxBytes + (k & 3) * 32, 16, 1024,
                                        kSwizzle128B);
          mma_ts(tmem + kColS, tmem + kColQ + 8 * k, bd, idS, k > 0 ? 1u : 0u);
        }
        mma_commit(bar(BAR_S_FULL));
      }
      __syncwarp();
      if (i > 0 && !issue_o(i - 1)) { ok = false; break; }
    }
    if (ok && !__any_sync(0xffffffffu, *abort_flag != 0)) ok = issue_o(T - 1);
    if (!ok) fail();
    // drain: every MMA issued by this thread has completed
    if (lane == 0) mma_commit(bar(BAR_DRAIN));
    __syncwarp();
    mbar_wait(bar(BAR_DRAIN), 0, lim);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ softmax / epilogue
    const int sub = warp & 3;                 // TMEM sub-partition of this warp
    const int row = sub * 32 + lane;          // head
    const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16);
    const bool live = row < p.h;
    float* orow = p.o_part + (((int64_t)b * p.num_splits + j) * p.h + row) * 512 + rank * 256;

    if (T == 0) {
      if (live) {
        for (int c = 0; c < 256; c += 4)
          *reinterpret_cast<float4*>(orow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (rank == 0) p.lse_part[((int64_t)b * p.num_splits + j) * p.h + row] = -INFINITY;
      }
    } else {
      // query slice -> TMEM (A operand): CTA 0 dims [0,256) ++ [512,576), CTA 1 dims [256,512)
      {
        const uint4* q = reinterpret_cast<const uint4*>(p.q_cat + ((int64_t)b * p.h + (live ? row : 0)) * 576);
        const int nq = rank == 0 ? 160 : 128;
        for (int c0 = 0; c0 < nq; c0 += 16) {
          uint32_t w[16];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int g = c0 / 4 + u;  // 8-dim group index within this CTA's slice
            const int gsrc = rank == 0 ? (g < 32 ? g : 64 + (g - 32)) : 32 + g;
            uint4 v = live ? q[gsrc] : make_uint4(0, 0, 0, 0);
            w[4 * u + 0] = v.x;
            w[4 * u + 1] = v.y;
            w[4 * u + 2] = v.z;
            w[4 * u + 3] = v.w;
          }
          tmem_st16(tl + kColQ + c0, w);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(BAR_Q_READY));
      }

      const uint32_t peer_recv = mapa(sbase + kOffRecv + row * 256, peer);
      const uint32_t peer_recv_full = mapa(bar(BAR_RECV_FULL), peer);
      const uint32_t peer_recv_free = mapa(bar(BAR_RECV_FREE), peer);
      const uint8_t* my_recv = smem + kOffRecv + row * 256;
      const int sw16 = row & 15, sw8 = row & 7;

      float m_run = -INFINITY, l = 0.f;
      bool ok = true;
      for (int i = 0; i < T; ++i) {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
        const int n_valid = min(kTok, L - (blo + i) * kTok);
        // partial scores of this CTA
        if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_S_FULL), i & 1, lim))) { ok = false; break; }
        tc_fence_after();
        uint32_t r[64];
        tmem_ld16(tl + kColS + 0, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
        tmem_ld16(tl + kColS + 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16]));
        tmem_ld16(tl + kColS + 32, *reinterpret_cast<uint32_t(*)[16]>(&r[32]));
        tmem_ld16(tl + kColS + 48, *reinterpret_cast<uint32_t(*)[16]>(&r[48]));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(BAR_S_EMPTY));

        // exchange partial scores with the peer CTA
        if (i > 0 && !__all_sync(0xffffffffu, mbar_wait<true>(bar(BAR_RECV_FREE), (i - 1) & 1, lim))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int c = 0; c < 16; ++c)
          st_cluster_v4(peer_recv + ((c ^ sw16) << 4), __uint_as_float(r[4 * c]),
                        __uint_as_float(r[4 * c + 1]), __uint_as_float(r[4 * c + 2]),
                        __uint_as_float(r[4 * c + 3]));
        mbar_arrive_remote(peer_recv_full);
        if (!__all_sync(0xffffffffu, mbar_wait<true>(bar(BAR_RECV_FULL), i & 1, lim))) {
          ok = false;
          break;
        }
        float x[64];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float4 v = *reinterpret_cast<const float4*>(my_recv + ((c ^ sw16) << 4));
          x[4 * c + 0] = __uint_as_float(r[4 * c + 0]) + v.x;
          x[4 * c + 1] = __uint_as_float(r[4 * c + 1]) + v.y;
          x[4 * c + 2] = __uint_as_float(r[4 * c + 2]) + v.z;
          x[4 * c + 3] = __uint_as_float(r[4 * c + 3]) + v.w;
        }
        mbar_arrive_remote(peer_recv_free);

        // online softmax (log2 domain) with lazy rescaling of O
        float mt = -INFINITY;
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          x[k] = k < n_valid ? x[k] * p.scale_log2 : -INFINITY;
          mt = fmaxf(mt, x[k]);
        }
        bool need = false;
        float m_new = m_run;
        if (i == 0) {
          m_run = mt;
        } else if (mt > m_run + kTau) {
          need = true;
          m_new = mt;
        }
        if (__any_sync(0xffffffffu, need)) {
          const int t = i - 1;
          if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_O_DONE + (t & 1)), (t >> 1) & 1, lim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = need ? exp2f(m_run - m_new) : 1.0f;
          for (int c = 0; c < 16; ++c) {
            uint32_t v[16];
            tmem_ld16(tl + kColO + 16 * c, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st16(tl + kColO + 16 * c, v);
          }
          tmem_wait_st();
          l *= alpha;
          m_run = m_new;
        }

        // P (bf16) for this tile; its buffer was last read by the O MMA of tile i-2
        if (i >= 2 &&
            !__all_sync(0xffffffffu, mbar_wait(bar(BAR_O_DONE + (i & 1)), ((i - 2) >> 1) & 1, lim))) {
          ok = false;
          break;
        }
        uint8_t* prow = smem + kOffP + (i & 1) * kPBytes + row * 128;
        float psum = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float p0 = exp2f(x[8 * c + 2 * e] - m_run);
            const float p1 = exp2f(x[8 * c + 2 * e + 1] - m_run);
            psum += p0 + p1;
            pk[e] = pack_bf16x2(p0, p1);
          }
          *reinterpret_cast<uint4*>(prow + ((c ^ sw8) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        l += psum;
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(BAR_P_FULL + (i & 1)));
      }

      if (!ok) fail();
      // epilogue: O_r / l -> o_part, lse (CTA 0)
      if (ok && !__any_sync(0xffffffffu, *abort_flag != 0)) {
        const int t = T - 1;
        const bool w = __all_sync(0xffffffffu, mbar_wait(bar(BAR_O_DONE + (t & 1)), (t >> 1) & 1, lim));
        if (!w) {
          fail();
        } else {
          tc_fence_after();
          const float inv = 1.0f / l;
          for (int c = 0; c < 16; ++c) {
            uint32_t v[16];
            tmem_ld16(tl + kColO + 16 * c, v);
            tmem_wait_ld();
            if (live) {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4)
                *reinterpret_cast<float4*>(orow + 16 * c + 4 * q4) =
                    make_float4(__uint_as_float(v[4 * q4]) * inv, __uint_as_float(v[4 * q4 + 1]) * inv,
                                __uint_as_float(v[4 * q4 + 2]) * inv, __uint_as_float(v[4 * q4 + 3]) * inv);
            }
          }
          if (live && rank == 0)
            p.lse_part[((int64_t)b * p.num_splits + j) * p.h + row] = (m_run + log2f(l)) * kLn2;
        }
      }
    }
  }

  // teardown: TMEM free after every reader is done; the cluster stays up until
  // neither CTA touches the other's shared memory any more
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D bf16 view [rows, cols] with the given row pitch, 64 x 64 boxes, 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
               uint64_t row_pitch_bytes) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_pitch_bytes};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int device_major() {
  static int major = -1;
  if (major < 0) {
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaGetDeviceProperties(&prop, dev) == cudaSuccess)
      major = prop.major;
    else
      major = 0;
  }
  return major;
}

}  // namespace

bool decode_tc_supported(int q_dtype, const mla_kv_cache& kv, int h) {
  return q_dtype == MLA_BF16 && kv.latent_dtype == MLA_BF16 && kv.rope_dtype == MLA_BF16 &&
         kv.d_c == 512 && kv.d_r == 64 && kv.block_size == kTok && h >= 1 && h <= 128 &&
         device_major() >= 10 && get_encode_fn() != nullptr;
}

cudaError_t launch_decode_tc(const void* q_cat, const mla_kv_cache& kv,
                             const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                             int B, int h, int num_splits, float scale, float* o_part,
                             float* lse_part, int32_t* status, cudaStream_t s) {
  CUtensorMap tm_lat, tm_rope;
  const uint64_t rows = (uint64_t)kv.num_blocks * kv.block_size;
  if (!make_tmap(&tm_lat, kv.latent, 512, rows, (uint64_t)kv.latent_stride * 2) ||
      !make_tmap(&tm_rope, kv.rope, 64, rows, (uint64_t)kv.rope_stride * 2))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  TcParams prm;
  prm.q_cat = static_cast<const uint16_t*>(q_cat);
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.o_part = o_part;
  prm.lse_part = lse_part;
  prm.status = status;
  prm.max_blocks = max_blocks;
  prm.B = B;
  prm.h = h;
  prm.num_splits = num_splits;
  prm.num_blocks = kv.num_blocks;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.wait_limit = 4000000000LL;  // about 2 s of SM clock
  dim3 grid(2 * B * num_splits);
  decode_tc_kernel<<<grid, kThreads, kSmemAlloc, s>>>(tm_lat, tm_rope, prm);
  return cudaGetLastError();
}

}  // namespace mla
