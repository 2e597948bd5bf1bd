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
// cluster of 2) shares each piece of work.  CTA r owns latent output columns
// [256 r, 256 r + 256) (O_r in TMEM) and the matching slice of the 576-d
// score contraction: latent columns [256 r, 256 r + 256) plus RoPE dims
// [32 r, 32 r + 32).  Each CTA TMA-loads exactly its own columns of every
// cache block (four 64x64 latent boxes, 128-byte swizzle, and one 32x64 RoPE
// box, 64-byte swizzle), so the pair reads each byte of the cache once.  Its
// partial score tile (128 heads x 64 tokens) goes to the peer through
// distributed shared memory: both CTAs keep the top 24 bits of every partial
// (their own and the peer's) and use the freed low byte of each value sent
// as a per-use tag, which the receiver polls for; both then hold the same
// S = S_0 + S_1 (the addition commutes), run a bit-identical online softmax
// and write the same P, which each multiplies into its own O_r.
//
// Schedule.  The grid is persistent: pair p runs part p of the balanced
// partition of the whole block stream (all sequences' blocks in order, see
// common.cuh), one segment (the part's blocks of one sequence) after another,
// and writes one partial (o, lse) per segment into slot p + b.
//
// Roles of the bf16 variant (19 warps, 608 threads):
//   warp 0       TMA producer: a ring of 4 stages (36 KB each) plus an L2
//                prefetch of the tile one ahead of the load;
//   warp 1       score MMA issuer: S = Q K^T, 16 TS steps (query latent slice
//                in TMEM) + 2 SS steps (query RoPE slice in shared memory),
//                M = 128 heads, N = 64 tokens;
//   warps 2..17  two softmax groups of 8 warps, tile k to group k % 2; two
//                warps per TMEM lane quarter split a row's 64 scores (32
//                each) and meet on a 64-thread named barrier for the row max;
//   warp 18      P.C MMA issuer: O_r += P C_r, 4 TS steps (P in TMEM, the
//                latent boxes as an MN-major B operand), N = 256.
// The FP8-latent variant has 3 bf16 stages, 2 e4m3 landing buffers, four
// converter warps (e4m3 x block scale -> bf16 into the swizzled stage) and a
// single event-driven MMA warp for both kinds of MMA.
//
// The running maximum is handed from one group to the other per tile; O is
// rescaled only when the maximum grows by more than kTau (log2 units), so
// P <= 2^kTau in bf16.
//
// TMEM columns: O_r [0, 256), S [256, 320), query latent slice [320, 448)
// (bf16 pairs, the A operand of the score MMA), P x 2 [448, 512) (bf16
// pairs, the A operand of the P.C MMA).  Every wait is bounded; on a timeout
// the kernel writes MLA_DEV_WAIT_TIMEOUT to the status word and winds down.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "device_registry.h"
#include "tc_ptx.cuh"

namespace mla {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

namespace {

using namespace tc;

constexpr int kTok = 64;                    // tokens per tile (= cache block)
constexpr int kMaxStages = 4;              // stage count of the bf16 variant (the larger)
constexpr int kPrefetchAhead = 1;           // L2 prefetch: tiles ahead of the TMA load
constexpr int kLandBytes = 64 * 256;        // FP8 variant: 64 tokens x 256 e4m3 codes
constexpr int kGroups = 2;                  // softmax groups (tile k goes to group k % kGroups)
// warps per TMEM lane quarter in a softmax group: with 2, a row's 64 scores are
// split between two warps (columns [32 hf, 32 hf + 32)), which halves each
// thread's share of the per-tile chain; the row maximum then meets in shared memory
constexpr int kHalves = 2;
constexpr int kCols = 64 / kHalves;         // score columns per softmax thread
constexpr int kGroupWarps = 4 * kHalves;
constexpr int kSoftWarps = kGroups * kGroupWarps;
// 1: the softmax warps poll for their scores without suspending (faster
// wake-up, at the cost of issue slots the other group's warps could use)
constexpr int kSpinSoftmax = 0;
constexpr int kBoxBytes = 64 * 128;         // 64 rows x 64 bf16, 128-byte swizzle
constexpr int kRopeBoxBytes = 64 * 64;      // 64 rows x 32 bf16, 64-byte swizzle
constexpr int kStageBytes = 4 * kBoxBytes + kRopeBoxBytes;  // 4 latent boxes + half the RoPE dims
constexpr int kQRopeBytes = 128 * 64;       // query RoPE slice: 128 heads x 32 bf16
// partial S of the peer: 64 scores per row, each the top 24 bits of a float32
// (sign, exponent, 15 mantissa bits) with a use tag in the low byte, so that
// the receiver can tell fresh values from the previous use's by looking at them
constexpr int kXChunks = 16;                // 16-byte chunks per row
constexpr int kRecvBytes = 128 * kXChunks * 16;

constexpr int kNumBars = 40;
// FP8 variant: warps that widen the e4m3 codes of each tile to bf16
constexpr int kConvWarps = 4;

// Layout of one variant: the bf16 cache (4 stages) or the FP8 latent cache (3
// bf16 stages filled by converter warps from 2 FP8 landing buffers).
template <bool kFp8>
struct Cfg {
  static constexpr int kStages = kFp8 ? 3 : kMaxStages;
  static constexpr int kLand = kFp8 ? 2 : 0;
  // bf16: one more warp issues the P.C MMAs (warp 2 + kSoftWarps); FP8: kConvWarps converter warps
  static constexpr bool kSplitMma = !kFp8;
  static constexpr int kThreads = 64 + 32 * kSoftWarps + (kFp8 ? 32 * kConvWarps : 32);
  static constexpr int kOffStages = 0;
  static constexpr int kOffLand = kOffStages + kStages * kStageBytes;
  static constexpr int kOffRecv = kOffLand + kLand * kLandBytes;
  static constexpr int kOffQRope = kOffRecv + kGroups * kRecvBytes;  // 1024-aligned
  static constexpr int kOffMpub = kOffQRope + kQRopeBytes;       // [2][128] float
  static constexpr int kOffLm = kOffMpub + 2 * 128 * 4;          // [2 seg][kGroups][128] float: m
  static constexpr int kOffLs = kOffLm + 2 * kGroups * 128 * 4;  // [2 seg][kGroups][kHalves][128] l
  static constexpr int kOffHmax = kOffLs + 2 * kGroups * kHalves * 128 * 4;  // [kGroups][kHalves][128]
  static constexpr int kOffBar = kOffHmax + (kHalves > 1 ? kGroups * kHalves * 128 * 4 : 0);
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 64;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;  // alignment slack
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
  static_assert(kStages <= kMaxStages, "barrier array");
};

constexpr uint32_t kColO = 0;
constexpr uint32_t kColS = 256;
constexpr uint32_t kColQ = 320;   // latent query slice (bf16 pairs), 128 columns
constexpr uint32_t kColP = 448;   // [2] P (bf16 pairs, 32 columns each), A of the P.C MMA
constexpr uint32_t kTmemCols = 512;

constexpr float kTau = 8.0f;  // lazy rescale threshold (log2 units): P stays <= 2^8
constexpr float kLn2 = 0.69314718055994530942f;

// barrier indices (derived from kStages so that the arrays never overlap)
enum {
  BAR_KV_FULL = 0,                      // [kStages] TMA (+ FP8 converters) -> MMA
  BAR_KV_EMPTY = BAR_KV_FULL + kMaxStages,  // [kStages] MMA (commit after P.C) -> TMA
  BAR_LAND_FULL = BAR_KV_EMPTY + kMaxStages,  // [2] FP8: TMA -> converters
  BAR_LAND_EMPTY = BAR_LAND_FULL + 2,   // [2] FP8: converters (2 warps) -> TMA
  BAR_S_FULL = BAR_LAND_EMPTY + 2,      // [kGroups] MMA -> softmax group k % kGroups; one
                                        //     barrier per group so that a group's parity
                                        //     waits never alias another group's phases
  BAR_S_EMPTY = BAR_S_FULL + kGroups,   // softmax (a group's warps) -> MMA
  BAR_P_FULL = BAR_S_EMPTY + 1,         // [2] softmax (a group's warps) -> MMA, by P buffer k & 1
  BAR_O_DONE = BAR_P_FULL + 2,          // [4] MMA -> softmax, by k & 3 (P buffer free, O final);
                                        //     four so that no waiter can be two phases off
  BAR_PEER_FREE = BAR_O_DONE + 4,       // [kGroups] peer group's warps have read what we sent
  BAR_MREADY = BAR_PEER_FREE + kGroups, // [2] running maximum of tile k published and the
                                        //     previous one read by every warp of the group
  BAR_Q_FREE = BAR_MREADY + 2,          // MMA: last score MMA of a segment done
  BAR_Q_READY = BAR_Q_FREE + 1,         // softmax (all warps) + TMA of the RoPE query slice
  BAR_O_FREE = BAR_Q_READY + 1,         // softmax (all warps): O of a segment read out
  BAR_SEG = BAR_O_FREE + 1,             // softmax (all warps): end-of-segment rendezvous
  BAR_DRAIN = BAR_SEG + 1,
  BAR_DRAIN_O = BAR_DRAIN + 1,          // bf16 variant: the P.C issuer's own drain
  BAR_NEVER = BAR_DRAIN_O + 1,          // signalled by nothing (diagnostic timeout wait)
  BAR_QTMA = BAR_NEVER + 1,             // TMA of the query RoPE slice landed (its issuer waits)
  BAR_COUNT = BAR_QTMA + 1,
};
static_assert(BAR_COUNT <= kNumBars, "barrier array");

struct TcParams {
  const uint16_t* q_cat;        // [B, h, 576] bf16
  const int32_t* block_table;   // [B, max_blocks]
  const int32_t* seq_lens;      // [B]
  float* o_part;                // [B + P - 1, h, 512]
  float* lse_part;              // [B + P - 1, h]
  int32_t* status;
  const float* kv_scale;        // FP8 variant: per-block dequantisation scale [num_blocks]
  // rows of a sequence: h = q_len * heads query rows (token j, head s) at
  // row j * heads + s; a CTA pair takes 128 of them (row group)
  int max_blocks, B, h, num_parts, num_blocks;
  int heads, q_len;
  float scale_log2;
  long long wait_limit;
  // diagnostic: the MMA issuer's first wait is made on BAR_NEVER with this
  // limit (SM clocks), so that the kernel takes its timeout path; 0 = off
  long long test_wait_limit;
};

// 2^x on the SFU (subnormal results flush to zero: P values that small do not
// change the sums)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32-byte global accesses (sm_100 family): one sector per thread, half the
// instructions of 16-byte ones; the address must be 32-byte aligned
__device__ __forceinline__ void ldg_nc_v8(const void* ptr, uint32_t* w) {
  asm volatile("ld.global.nc.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                 "=r"(w[6]), "=r"(w[7])
               : "l"(ptr));
}
__device__ __forceinline__ void stg_v8(void* ptr, const float* v) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "f"(v[0]),
               "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}

// packed pairs of float32 (lo, hi) for the sm_100-family f32x2 arithmetic
typedef unsigned long long f2_t;
__device__ __forceinline__ f2_t f2_make(float lo, float hi) {
  f2_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f2_split(f2_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2_t f2_add(f2_t a, f2_t b) {
  f2_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_sub(f2_t a, f2_t b) {
  f2_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_mul(f2_t a, f2_t b) {
  f2_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_fma(f2_t a, f2_t b, f2_t c) {
  f2_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Optional per-tile event timestamps for pipeline analysis (compiled only with
// -DMLA_TRACE; the product build has none of it).
#ifdef MLA_TRACE
constexpr int kTraceTiles = 128;
constexpr int kTraceEv = 24;
__device__ unsigned long long* g_trace = nullptr;
#define MLA_TR(k, ev)                                                                   \
  do {                                                                                  \
    if (g_trace != nullptr && part < 2 && (k) < kTraceTiles)                            \
      g_trace[((part * 2 + rank) * kTraceTiles + (k)) * kTraceEv + (ev)] = clock64();   \
  } while (0)
#define MLA_TRMAX(k, ev)                                                                \
  do {                                                                                  \
    if (g_trace != nullptr && part < 2 && (k) < kTraceTiles)                            \
      atomicMax(&g_trace[((part * 2 + rank) * kTraceTiles + (k)) * kTraceEv + (ev)],    \
                (unsigned long long)clock64());                                         \
  } while (0)
#define MLA_TRMIN(k, ev)                                                                \
  do {                                                                                  \
    if (g_trace != nullptr && part < 2 && (k) < kTraceTiles)                            \
      atomicMax(&g_trace[((part * 2 + rank) * kTraceTiles + (k)) * kTraceEv + (ev)],    \
                ~(unsigned long long)clock64());                                        \
  } while (0)
#define MLA_SITE(site)                                                                  \
  do {                                                                                  \
    if (g_trace != nullptr && part < 2)                                                 \
      g_trace[((part * 2 + rank) * kTraceTiles + kTraceTiles - 1) * kTraceEv + 11] = (site); \
  } while (0)
#else
#define MLA_TR(k, ev) \
  do {                \
  } while (0)
#define MLA_TRMAX(k, ev) \
  do {                   \
  } while (0)
#define MLA_TRMIN(k, ev) \
  do {                   \
  } while (0)
#define MLA_SITE(site) \
  do {                 \
  } while (0)
#endif

// Walks the part's tiles (sequence b, logical block blk) in stream order.  The
// current sequence's clamped length is kept, so that a tile's valid length
// needs no memory access (the length is loaded once, when the walk enters the
// sequence).
struct TileIter {
  const int32_t* lens;
  int maxb, b, blk, nb, L;
  __device__ static int clamp_len(int L, int maxb) {
    return L < 0 ? 0 : (L > maxb * kTok ? maxb * kTok : L);
  }
  __device__ void init(const int32_t* l, int max_blocks, int b0, int blk0) {
    lens = l;
    maxb = max_blocks;
    b = b0;
    blk = blk0;
    L = clamp_len(lens[b], maxb);
    nb = (L + kTok - 1) / kTok;
  }
  // only called while another tile of the part follows, so b stays < B
  __device__ void next() {
    if (++blk >= nb) {
      blk = 0;
      do {
        ++b;
        L = clamp_len(lens[b], maxb);
        nb = (L + kTok - 1) / kTok;
      } while (nb == 0);
    }
  }
  __device__ int len() const { return L; }
  __device__ int valid() const {
    const int n = L - blk * kTok;
    return n < kTok ? n : kTok;
  }
};

template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<kFp8>::kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_lat,
                 const __grid_constant__ CUtensorMap tm_rope,
                 const __grid_constant__ CUtensorMap tm_q, const TcParams p) {
  using C = Cfg<kFp8>;
  constexpr int kStages = C::kStages, kThreads = C::kThreads;
  constexpr int kOffStages = C::kOffStages, kOffLand = C::kOffLand, kOffRecv = C::kOffRecv;
  constexpr int kOffQRope = C::kOffQRope, kOffMpub = C::kOffMpub;
  constexpr int kOffBar = C::kOffBar, kOffMisc = C::kOffMisc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int part = (blockIdx.x / 2) % p.num_parts;  // part of the block stream
  const int row0 = (blockIdx.x / 2) / p.num_parts * 128;  // first query row of this pair
  // scheduled while the previous grid of the stream finishes; nothing is read
  // from memory before that grid has completed
  grid_dep_launch();
  grid_dep_wait();

  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8 * i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* info = reinterpret_cast<int*>(smem + kOffMisc + 16);  // b0, blk0, ntiles

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(BAR_KV_FULL + s), kFp8 ? 1 + kConvWarps : 1);   // FP8: + the converter warps
      mbar_init(bar(BAR_KV_EMPTY + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(BAR_LAND_FULL + i), 1);
      mbar_init(bar(BAR_LAND_EMPTY + i), kConvWarps);
    }
    mbar_init(bar(BAR_S_EMPTY), kGroupWarps);
    for (int i = 0; i < kGroups; ++i) {
      mbar_init(bar(BAR_S_FULL + i), 1);
      mbar_init(bar(BAR_PEER_FREE + i), kGroupWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(BAR_P_FULL + i), kGroupWarps);
      mbar_init(bar(BAR_MREADY + i), kGroupWarps);
    }
    for (int i = 0; i < 4; ++i) mbar_init(bar(BAR_O_DONE + i), 1);
    mbar_init(bar(BAR_Q_FREE), 1);
    mbar_init(bar(BAR_Q_READY), kSoftWarps);
    mbar_init(bar(BAR_QTMA), 1);
    mbar_init(bar(BAR_O_FREE), kSoftWarps);
    mbar_init(bar(BAR_SEG), kSoftWarps);
    mbar_init(bar(BAR_DRAIN), 1);
    mbar_init(bar(BAR_DRAIN_O), 1);
    mbar_init(bar(BAR_NEVER), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    // this part's range of the block stream (both CTAs compute the same)
    const long long T = warp_stream_scan(p.seq_lens, p.B, kTok, p.max_blocks, -1, -1, nullptr,
                                         nullptr, nullptr);
    const int P = (int)(T < p.num_parts ? T : p.num_parts);
    int b0 = -1;
    long long g0 = 0, g1 = 0, sb = 0;
    if (part < P) {
      g0 = part_begin(T, P, part);
      g1 = part_begin(T, P, part + 1);
      warp_stream_scan(p.seq_lens, p.B, kTok, p.max_blocks, -1, g0, nullptr, &b0, &sb);
    }
    if (lane == 0) {
      info[0] = b0;
      info[1] = (int)(g0 - sb);
      info[2] = (int)(g1 - g0);
      prefetch_tmap(&tm_lat);
      prefetch_tmap(&tm_rope);
      prefetch_tmap(&tm_q);
      if (part == 0 && rank == 0)
        for (int b = 0; b < p.B; ++b)
          if (p.seq_lens[b] > p.max_blocks * kTok) set_status(p.status, MLA_DEV_BAD_LENGTH);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  // exchange buffers start with tag 0, which no use carries
  for (int i = threadIdx.x; i < kGroups * kRecvBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + kOffRecv)[i] = make_uint4(0, 0, 0, 0);
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated, part known
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int b_first = info[0], blk_first = info[1], ntiles = info[2];
  const long long lim = p.wait_limit;
  bool timed_out = false;

  auto fail = [&]() {
    if (timed_out) set_status(p.status, MLA_DEV_WAIT_TIMEOUT);
    *abort_flag = 1;
  };
  // lane 0 waits, the warp learns the result
  auto warp_wait = [&](uint32_t b, uint32_t parity) -> bool {
    bool ok = true;
    if (lane == 0) {
      ok = mbar_wait_or_abort(b, parity, lim, abort_flag, &timed_out);
      if (!ok && timed_out) MLA_SITE(1000 + warp * 100 + (int)((b - bar(0)) / 8));
    }
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  };
  // the same for the MMA issuer warps, polling without suspending
  auto warp_spin = [&](uint32_t b, uint32_t parity) -> bool {
    bool ok = true;
    if (lane == 0) {
      ok = mbar_spin_or_abort(b, parity, lim, abort_flag, &timed_out);
      if (!ok && timed_out) MLA_SITE(1000 + warp * 100 + (int)((b - bar(0)) / 8));
    }
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  };
  auto warp_wait_cluster = [&](uint32_t b, uint32_t parity) -> bool {
    bool ok = true;
    if (lane == 0) {
      ok = mbar_wait_or_abort<true>(b, parity, lim, abort_flag, &timed_out);
      if (!ok && timed_out) MLA_SITE(1000 + warp * 100 + (int)((b - bar(0)) / 8));
    }
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  };

  if (b_first >= 0 && ntiles > 0 && warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      TileIter it;
      it.init(p.seq_lens, p.max_blocks, b_first, blk_first);
      const uint32_t tx = kStageBytes;
      // L2 prefetch of the tiles whose loads come next (kPrefetchAhead tiles
      // ahead of the load), so that a stage freed late (after its P.C MMA)
      // refills partly from L2; running further ahead lets the cache stream
      // evict prefetched lines before their load, which then reads them from
      // HBM a second time
      TileIter pf;
      pf.init(p.seq_lens, p.max_blocks, b_first, blk_first);
      int kp = 0;
      auto prefetch_upto = [&](int kend) {
        for (; kp < kend && kp < ntiles; ++kp) {
          const int pb = p.block_table[(int64_t)pf.b * p.max_blocks + pf.blk];
          if (pb >= 0 && pb < p.num_blocks) {
            if constexpr (kFp8) {
              tma_prefetch_2d(&tm_lat, (int)rank * 256, pb * kTok);
            } else {
              for (int c = 0; c < 4; ++c)
                tma_prefetch_2d(&tm_lat, (int)(rank * 4 + c) * 64, pb * kTok);
            }
            tma_prefetch_2d(&tm_rope, (int)rank * 32, pb * kTok);
          }
          if (pf.blk == 0 && kp > 0) {
            // a later segment starts here: its query rows (this CTA's latent
            // slice and RoPE dims) go to L2 ahead of the segment's query load
            for (int j = 0; j < 8; ++j)
              tma_prefetch_2d(&tm_q, 256 * (int)rank + 32 * j, pf.b * p.h + row0);
            tma_prefetch_2d(&tm_q, 512 + 32 * (int)rank, pf.b * p.h + row0);
          }
          if (kp + 1 < ntiles) pf.next();
        }
      };
      int k = 0;
      for (; k < ntiles; ++k) {
        prefetch_upto(k + 1 + kPrefetchAhead);
        if (*abort_flag) break;
        const int st = k % kStages;
        if (k >= kStages &&
            !mbar_spin_or_abort(bar(BAR_KV_EMPTY + st), ((k / kStages) - 1) & 1, lim, abort_flag,
                                &timed_out)) {
          fail();
          break;
        }
        int pb = p.block_table[(int64_t)it.b * p.max_blocks + it.blk];
        if (pb < 0 || pb >= p.num_blocks) {
          set_status(p.status, MLA_DEV_BAD_BLOCK);
          pb = 0;  // load a valid block instead; the result is flagged as wrong
        }
        MLA_TR(k, 0);
        const uint32_t dst = sbase + kOffStages + st * kStageBytes;
        const uint32_t fb = bar(BAR_KV_FULL + st);
        const int y = pb * kTok;
        if constexpr (kFp8) {
          // e4m3 codes of this CTA's 256 latent columns -> landing buffer j; the
          // converter warps write the bf16 latent boxes of stage st from it
          const int j = k % 2;
          if (k >= 2 && !mbar_wait_or_abort(bar(BAR_LAND_EMPTY + j), ((k / 2) - 1) & 1, lim,
                                            abort_flag, &timed_out)) {
            fail();
            break;
          }
          reinterpret_cast<volatile int*>(smem + kOffMisc + 32)[j] = pb;
          mbar_arrive_expect_tx(fb, kRopeBoxBytes);
          tma_load_2d(dst + 4 * kBoxBytes, &tm_rope, (int)rank * 32, y, fb);
          mbar_arrive_expect_tx(bar(BAR_LAND_FULL + j), kLandBytes);
          tma_load_2d(sbase + kOffLand + j * kLandBytes, &tm_lat, (int)rank * 256, y,
                      bar(BAR_LAND_FULL + j));
        } else {
          mbar_arrive_expect_tx(fb, tx);
          for (int c = 0; c < 4; ++c)
            tma_load_2d(dst + c * kBoxBytes, &tm_lat, (int)(rank * 4 + c) * 64, y, fb);
          tma_load_2d(dst + 4 * kBoxBytes, &tm_rope, (int)rank * 32, y, fb);
        }
        if (k + 1 < ntiles) it.next();
      }
      // every issued load must land before the CTA may exit
      bool dummy = false;
      for (int st = 0; st < kStages; ++st) {
        const int n = (k - st + kStages - 1) / kStages;  // loads issued into stage st
        if (n > 0) {
          int never = 0;
          mbar_wait_or_abort(bar(BAR_KV_FULL + st), (n - 1) & 1, lim, &never, &dummy);
        }
      }
      if constexpr (kFp8) {
        for (int j = 0; j < 2; ++j) {
          const int n = (k - j + 1) / 2;  // loads issued into landing buffer j
          if (n > 0) {
            int never = 0;
            mbar_wait_or_abort(bar(BAR_LAND_FULL + j), (n - 1) & 1, lim, &never, &dummy);
          }
        }
      }
    }
  } else if (C::kSplitMma && b_first >= 0 && ntiles > 0 && warp == 1) {
    // ------------------------------------------------------------ score MMA issuer (bf16)
    // S(k) needs its stage (KV_FULL), the previous tile's scores loaded out
    // (S_EMPTY) and, at a segment start, the segment's query; blocking waits,
    // so the warp sleeps until its inputs are there.  The P.C MMAs come from
    // their own warp: a P.C never waits behind a score MMA being issued.
    const uint32_t idS = idesc_bf16_f32(128, 64, false, false);
    TileIter its;
    its.init(p.seq_lens, p.max_blocks, b_first, blk_first);
    int seg_s = 0;
    bool ok = true;
    if (p.test_wait_limit > 0) {
      // diagnostic: a wait that nothing ends, with a short limit
      bool fin = true;
      if (lane == 0)
        fin = mbar_spin_or_abort(bar(BAR_NEVER), 0, p.test_wait_limit, abort_flag, &timed_out);
      if (!__shfl_sync(0xffffffffu, fin ? 1 : 0, 0)) ok = false;
    }
    for (int ks = 0; ok && ks < ntiles; ++ks) {
      const int st = ks % kStages;
      const bool first = (ks == 0) || (its.blk == 0);
      const bool last = (ks == ntiles - 1) || (its.blk == its.nb - 1);
      // the tile's length first: its global load then overlaps the waits
      const int n_valid = its.valid();
      if (first && !warp_spin(bar(BAR_Q_READY), seg_s & 1)) { ok = false; break; }
      if (!warp_spin(bar(BAR_KV_FULL + st), (ks / kStages) & 1)) { ok = false; break; }
      if (lane == 0) MLA_TR(ks, 16);
      if (ks > 0 && !warp_spin(bar(BAR_S_EMPTY), (ks - 1) & 1)) { ok = false; break; }
      if (lane == 0) MLA_TR(ks, 17);
      if (n_valid < kTok) {
        // slots past the sequence end: zero them so that P = 0 meets finite values
        uint8_t* sp = smem + kOffStages + st * kStageBytes;
        const int nrow = kTok - n_valid;
        for (int e = lane; e < 4 * nrow * 8; e += 32) {
          const int box = e / (nrow * 8), rr = (e / 8) % nrow, ch = e % 8;
          *reinterpret_cast<uint4*>(sp + box * kBoxBytes + (n_valid + rr) * 128 + ch * 16) =
              make_uint4(0, 0, 0, 0);
        }
        for (int e = lane; e < nrow * 4; e += 32)
          *reinterpret_cast<uint4*>(sp + 4 * kBoxBytes + (n_valid + e / 4) * 64 + (e % 4) * 16) =
              make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      __syncwarp();
      tc_fence_after();
      if (lane == 0) {
        MLA_TR(ks, 1);
        const uint32_t stage = sbase + kOffStages + st * kStageBytes;
        for (int kk = 0; kk < 16; ++kk) {
          const uint64_t bd = smem_desc(stage + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024,
                                        kSwizzle128B);
          mma_ts(tmem + kColS, tmem + kColQ + 8 * kk, bd, idS, kk > 0 ? 1u : 0u);
        }
        for (int kk = 0; kk < 2; ++kk) {
          const uint64_t ad = smem_desc(sbase + kOffQRope + kk * 32, 16, 512, kSwizzle64B);
          const uint64_t bd = smem_desc(stage + 4 * kBoxBytes + kk * 32, 16, 512, kSwizzle64B);
          mma_ss(tmem + kColS, ad, bd, idS, 1u);
        }
        mma_commit(bar(BAR_S_FULL + (ks % kGroups)));
        if (last) mma_commit(bar(BAR_Q_FREE));
      }
      __syncwarp();
      if (last) ++seg_s;
      if (ks + 1 < ntiles) its.next();
    }
    if (!ok) fail();
    if (lane == 0) {
      mma_commit(bar(BAR_DRAIN));
      int never = 0;
      bool dummy = false;
      mbar_wait_or_abort(bar(BAR_DRAIN), 0, lim, &never, &dummy);
    }
    __syncwarp();
  } else if (C::kSplitMma && b_first >= 0 && ntiles > 0 && warp == 2 + kSoftWarps) {
    // ------------------------------------------------------------ P.C MMA issuer (bf16)
    // O(k) += P(k) C(k) once P(k) is in TMEM (S(k) is complete by then, so the
    // commit after O(k) also covers the last reader of the stage); the first
    // tile of a segment overwrites O after the previous segment's epilogue.
    const uint32_t idO = idesc_bf16_f32(128, 256, false, true);
    TileIter ito;
    ito.init(p.seq_lens, p.max_blocks, b_first, blk_first);
    int seg_o = 0;
    bool ok = true;
    for (int ko = 0; ko < ntiles; ++ko) {
      const bool first = (ko == 0) || (ito.blk == 0);
      const bool last = (ko == ntiles - 1) || (ito.blk == ito.nb - 1);
      if (first && seg_o > 0 && !warp_spin(bar(BAR_O_FREE), (seg_o - 1) & 1)) { ok = false; break; }
      if (!warp_spin(bar(BAR_P_FULL + (ko & 1)), (ko >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      if (lane == 0) {
        MLA_TR(ko, 2);
        const uint32_t stage = sbase + kOffStages + (ko % kStages) * kStageBytes;
        const uint32_t pcol = kColP + 32 * (ko & 1);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint64_t bd = smem_desc(stage + c * 2048, kBoxBytes, 1024, kSwizzle128B);
          mma_ts(tmem + kColO, tmem + pcol + 8 * c, bd, idO, (first && c == 0) ? 0u : 1u);
        }
        mma_commit(bar(BAR_O_DONE + (ko & 3)));
        mma_commit(bar(BAR_KV_EMPTY + (ko % kStages)));
      }
      __syncwarp();
      if (last) ++seg_o;
      if (ko + 1 < ntiles) ito.next();
    }
    if (!ok) fail();
    if (lane == 0) {
      mma_commit(bar(BAR_DRAIN_O));
      int never = 0;
      bool dummy = false;
      mbar_wait_or_abort(bar(BAR_DRAIN_O), 0, lim, &never, &dummy);
    }
    __syncwarp();
  } else if (b_first >= 0 && ntiles > 0 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Event-driven: whichever of the next score MMA S(ks) and the next P.C MMA
    // O(ko) has its inputs ready is issued first, so a late P never holds back
    // the next score tile (lane 0 probes, the warp follows its decision).
    const uint32_t idS = idesc_bf16_f32(128, 64, false, false);
    const uint32_t idO = idesc_bf16_f32(128, 256, false, true);
    const int nbox = 5;                     // boxes a ragged tile zero-fills (4 latent + RoPE)
    TileIter its, ito;
    its.init(p.seq_lens, p.max_blocks, b_first, blk_first);
    ito.init(p.seq_lens, p.max_blocks, b_first, blk_first);
    int ks = 0, ko = 0, seg_s = 0, seg_o = 0;
    int nv_s = its.valid();  // valid tokens of tile ks
    long long idle_since = clock64();
    bool ok = true;
    if (p.test_wait_limit > 0) {
      // diagnostic: a wait that nothing ends, with a short limit
      bool fin = true;
      if (lane == 0)
        fin = mbar_spin_or_abort(bar(BAR_NEVER), 0, p.test_wait_limit, abort_flag, &timed_out);
      if (!__shfl_sync(0xffffffffu, fin ? 1 : 0, 0)) ok = false;
    }
    // lane 0: issue O(ko) if its P is ready (state is advanced by advance_o on all lanes)
    auto try_issue_o_lane0 = [&]() -> bool {
      if (ko >= ks) return false;
      const bool first = (ko == 0) || (ito.blk == 0);
      const bool ready =
          (!(first && seg_o > 0) || mbar_test_wait(bar(BAR_O_FREE), (seg_o - 1) & 1)) &&
          mbar_test_wait(bar(BAR_P_FULL + (ko & 1)), (ko >> 1) & 1);
      if (!ready) return false;
      tc_fence_after();
      MLA_TR(ko, 2);
      const uint32_t stage = sbase + kOffStages + (ko % kStages) * kStageBytes;
      const uint32_t pcol = kColP + 32 * (ko & 1);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint64_t bd = smem_desc(stage + c * 2048, kBoxBytes, 1024, kSwizzle128B);
        mma_ts(tmem + kColO, tmem + pcol + 8 * c, bd, idO, (first && c == 0) ? 0u : 1u);
      }
      mma_commit(bar(BAR_O_DONE + (ko & 3)));
      mma_commit(bar(BAR_KV_EMPTY + (ko % kStages)));
      return true;
    };
    auto advance_o = [&]() {
      const bool last = (ko == ntiles - 1) || (ito.blk == ito.nb - 1);
      if (last) ++seg_o;
      if (ko + 1 < ntiles) ito.next();
      ++ko;
    };
    while (ok && ko < ntiles) {
      bool did = false;
      // O(ko) first: it frees a P buffer and a stage
      {
        bool issued = false;
        if (lane == 0) issued = try_issue_o_lane0();
        if (__shfl_sync(0xffffffffu, issued ? 1 : 0, 0)) {
          advance_o();
          did = true;
        }
      }
      if (ks < ntiles) {
        const int st = ks % kStages;
        const bool first = (ks == 0) || (its.blk == 0);
        const bool last = (ks == ntiles - 1) || (its.blk == its.nb - 1);
        bool ready = true;
        if (lane == 0) {
          const bool q_ok = !first || mbar_test_wait(bar(BAR_Q_READY), seg_s & 1);
          const bool kv_ok = mbar_test_wait(bar(BAR_KV_FULL + st), (ks / kStages) & 1);
          const bool s_ok = ks == 0 || mbar_test_wait(bar(BAR_S_EMPTY), (ks - 1) & 1);
#ifdef MLA_TRACE
          if (kv_ok && g_trace != nullptr && part < 2 && ks < kTraceTiles &&
              g_trace[((part * 2 + rank) * kTraceTiles + ks) * kTraceEv + 12] == 0)
            MLA_TR(ks, 12);
          if (s_ok && g_trace != nullptr && part < 2 && ks < kTraceTiles &&
              g_trace[((part * 2 + rank) * kTraceTiles + ks) * kTraceEv + 13] == 0)
            MLA_TR(ks, 13);
#endif
          ready = q_ok && kv_ok && s_ok;
        }
        if (__shfl_sync(0xffffffffu, ready ? 1 : 0, 0)) {
          const int n_valid = nv_s;
          if (n_valid < kTok) {
            // slots past the sequence end: zero them so that P = 0 meets finite values
            uint8_t* sp = smem + kOffStages + st * kStageBytes;
            const int nrow = kTok - n_valid;
            for (int e = lane; e < 4 * nrow * 8; e += 32) {
              const int box = e / (nrow * 8), rr = (e / 8) % nrow, ch = e % 8;
              *reinterpret_cast<uint4*>(sp + box * kBoxBytes + (n_valid + rr) * 128 + ch * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            for (int e = lane; e < nrow * 4; e += 32)
              *reinterpret_cast<uint4*>(sp + 4 * kBoxBytes + (n_valid + e / 4) * 64 + (e % 4) * 16) =
                  make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
          }
          __syncwarp();
          tc_fence_after();
          bool o_issued_inside = false;
          if (lane == 0) {
            MLA_TR(ks, 1);
            const uint32_t stage = sbase + kOffStages + st * kStageBytes;
            for (int kk = 0; kk < 16; ++kk) {
              const uint64_t bd = smem_desc(stage + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16,
                                            1024, kSwizzle128B);
              mma_ts(tmem + kColS, tmem + kColQ + 8 * kk, bd, idS, kk > 0 ? 1u : 0u);
              // a P.C MMA that became ready meanwhile goes in between (the two
              // accumulators are independent), so its stage is freed sooner
              if (kk == 7 && try_issue_o_lane0()) o_issued_inside = true;
            }
            // this CTA's 32 RoPE dims: query slice and keys in shared memory (64-byte swizzle)
            for (int kk = 0; kk < 2; ++kk) {
              const uint64_t ad = smem_desc(sbase + kOffQRope + kk * 32, 16, 512, kSwizzle64B);
              const uint64_t bd = smem_desc(stage + 4 * kBoxBytes + kk * 32, 16, 512, kSwizzle64B);
              mma_ss(tmem + kColS, ad, bd, idS, 1u);
            }
            mma_commit(bar(BAR_S_FULL + (ks % kGroups)));
            if (last) mma_commit(bar(BAR_Q_FREE));
          }
          if (__shfl_sync(0xffffffffu, o_issued_inside ? 1 : 0, 0)) advance_o();
          __syncwarp();
          if (last) ++seg_s;
          if (ks + 1 < ntiles) {
            its.next();
            nv_s = its.valid();  // loaded now, needed only at the next score MMA
          }
          ++ks;
          did = true;
        }
      }
      if (did) {
        idle_since = clock64();
      } else {
        // back off: a spinning MMA warp would take issue slots from the
        // softmax warps that share its SM sub-partition
        __nanosleep(64);
        if (*abort_flag) { ok = false; break; }
        if (clock64() - idle_since > lim) {
          timed_out = true;
          ok = false;
          if (lane == 0) MLA_SITE(2000 + ks * 0 + (ko < 1000 ? ko : 999));
          break;
        }
      }
    }
    if (!ok) fail();
    // drain: every MMA issued by this thread has completed
    if (lane == 0) {
      mma_commit(bar(BAR_DRAIN));
      int never = 0;
      bool dummy = false;
      mbar_wait_or_abort(bar(BAR_DRAIN), 0, lim, &never, &dummy);
    }
    __syncwarp();
  } else if (kFp8 && b_first >= 0 && ntiles > 0 && warp >= 2 + kSoftWarps) {
    // ------------------------------------------------------------ FP8 converters
    // Landing buffer j holds the e4m3 codes of 64 tokens x this CTA's 256 latent
    // columns (row-major, 256 B per token).  Each code becomes
    // bf16(e4m3 value x block scale) in the 128-byte-swizzled bf16 boxes of
    // stage st, where the MMAs read it (kexue.fm / iotdigitaltwinplm: the
    // latent is stored in FP8; one float32 scale per 64-token block).
    const int ct = threadIdx.x - 32 * (2 + kSoftWarps);  // 0 .. 32 kConvWarps - 1
    const volatile int* land_pb = reinterpret_cast<const volatile int*>(smem + kOffMisc + 32);
    bool ok = true;
    for (int k = 0; k < ntiles; ++k) {
      const int j = k % 2, st = k % kStages;
      if (!warp_wait(bar(BAR_LAND_FULL + j), (k / 2) & 1)) { ok = false; break; }
      if (ct == 0) MLA_TR(k, 22);
      const float sc = p.kv_scale[land_pb[j]];
      const uint8_t* src = smem + kOffLand + j * kLandBytes;
      uint8_t* dst = smem + kOffStages + st * kStageBytes;
      const f2_t sc2 = f2_make(sc, sc);
#pragma unroll 2
      for (int i = ct; i < 64 * 16; i += 32 * kConvWarps) {
        const int r = i >> 4, q = i & 15;           // token row, 16-code group
        const uint4 v = *reinterpret_cast<const uint4*>(src + r * 256 + q * 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
                static_cast<__nv_fp8x2_storage_t>((w[e] >> (16 * hh)) & 0xFFFFu), __NV_E4M3);
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
            float x0, x1;
            f2_split(f2_mul(f2_make(f.x, f.y), sc2), x0, x1);
            o[2 * e + hh] = pack_bf16x2(x0, x1);
          }
        }
        // codes 16q .. 16q+15 = latent columns of box q / 4, chunks 2 (q % 4) and +1
        const int box = q >> 2, c0 = 2 * (q & 3);
        uint8_t* rowp = dst + box * kBoxBytes + r * 128;
        *reinterpret_cast<uint4*>(rowp + ((c0 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(rowp + (((c0 + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        MLA_TRMAX(k, 23);
        mbar_arrive(bar(BAR_LAND_EMPTY + j));
        mbar_arrive(bar(BAR_KV_FULL + st));
      }
    }
    if (!ok) fail();
  } else if (b_first >= 0 && ntiles > 0 && warp >= 2 && warp < 2 + kSoftWarps) {
    // ------------------------------------------------------------ softmax groups
    const int wg = (warp - 2) % kGroupWarps;  // warp within the group
    const int g = (warp - 2) / kGroupWarps;   // group: tiles k with k % kGroups == g
    const int hf = wg >> 2;                   // column half: score columns [kCols hf, +kCols)
    const int sub = warp & 3;                 // TMEM sub-partition of this warp
    const int row = sub * 32 + lane;          // TMEM lane: query row row0 + row
    const int grow = row0 + row;
    const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16);
    const bool live = grow < p.h;
    // query token j = grow / heads sits q_len - 1 - j positions before the
    // last cached row and sees the rows up to its own position
    const int c_row = live ? p.q_len - 1 - grow / p.heads : 0;
    const bool group_lead = wg == 0 && lane == 0;
    float* mpub = reinterpret_cast<float*>(smem + kOffMpub);
    float* lm = reinterpret_cast<float*>(smem + C::kOffLm);
    float* lsum = reinterpret_cast<float*>(smem + C::kOffLs);
    float* hmax = reinterpret_cast<float*>(smem + C::kOffHmax);
    // the two warps of this group that share TMEM lane quarter sub meet on
    // named barrier 1 + 4 g + sub (64 threads)
    auto pair_sync = [&]() {
      if constexpr (kHalves > 1)
        asm volatile("bar.sync %0, 64;" ::"r"(1 + 4 * g + sub) : "memory");
    };
    // exchange buffers: chunk c (16 B) of row sub * 32 + lane at
    // (sub * kXChunks + c) * 512 + lane * 16, so that a warp's stores and loads
    // are contiguous 512-byte runs; this thread owns chunks [kCols/4 hf, +kCols/4)
    constexpr int kMyChunks = kCols / 4;
    const uint32_t xoff = (uint32_t)((sub * kXChunks + kMyChunks * hf) * 512 + lane * 16);
    const uint8_t* my_recv = smem + kOffRecv + g * kRecvBytes + xoff;
    const uint32_t my_recv_u32 = sbase + kOffRecv + g * kRecvBytes + xoff;
    const uint32_t peer_recv = mapa(sbase + kOffRecv + g * kRecvBytes + xoff, peer);
    const uint32_t peer_free = mapa(bar(BAR_PEER_FREE + g), peer);

    // query slice of sequence b -> TMEM (A operand).  CTA r holds latent dims
    // [256 r, 256 r + 256) (TMEM) and RoPE dims [512 + 32 r, +32) (shared
    // memory); the eight 16-column chunks (32 dims each) are split between
    // the softmax threads of a row.
    constexpr int kQChunks = 8 / (kGroups * kHalves);
    // 32-byte accesses need 32-byte aligned bases (the interface asks for 16)
    const bool q32 = (reinterpret_cast<uintptr_t>(p.q_cat) & 31u) == 0;
    const bool o32 = (reinterpret_cast<uintptr_t>(p.o_part) & 31u) == 0;
    static_assert(kQChunks * kGroups * kHalves == 8, "query chunks per thread");
    int n_qtma = 0;  // query RoPE loads issued by this thread (group lead of group 0)
    auto load_q = [&](int b) {
      if (group_lead && g == 0) {
        // RoPE dims [512 + 32 rank, +32) of the 128 query rows of sequence b
        mbar_arrive_expect_tx(bar(BAR_QTMA), kQRopeBytes);
        tma_load_2d(sbase + kOffQRope, &tm_q, 512 + 32 * (int)rank, b * p.h + row0, bar(BAR_QTMA));
      }
      const uint4* q = reinterpret_cast<const uint4*>(p.q_cat + ((int64_t)b * p.h + (live ? grow : 0)) * 576);
      const int qc0 = (g * kHalves + hf) * kQChunks;
      // all loads first (one memory round trip), then the TMEM stores; rows
      // are 1152 bytes apart, so each load instruction touches 32 lines:
      // 32-byte loads where q_cat allows them halve that traffic
      uint32_t w[kQChunks][16];
#pragma unroll
      for (int cc = 0; cc < kQChunks; ++cc) {
        const int dim0 = 256 * (int)rank + 32 * (qc0 + cc);
        if (!live) {
#pragma unroll
          for (int e = 0; e < 16; ++e) w[cc][e] = 0u;
        } else if (q32) {
          ldg_nc_v8(q + dim0 / 8, &w[cc][0]);
          ldg_nc_v8(q + dim0 / 8 + 2, &w[cc][8]);
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 v = __ldg(q + dim0 / 8 + u);
            w[cc][4 * u + 0] = v.x;
            w[cc][4 * u + 1] = v.y;
            w[cc][4 * u + 2] = v.z;
            w[cc][4 * u + 3] = v.w;
          }
        }
      }
#pragma unroll
      for (int cc = 0; cc < kQChunks; ++cc) tmem_st16(tl + kColQ + 16 * (qc0 + cc), w[cc]);
      tmem_wait_st();
      tc_fence_before();
      if (group_lead && g == 0) {
        // the issuer sees its own copy land before it signals the MMA warp, so
        // no copy into this CTA's shared memory is in flight once the role
        // ends, whatever the other roles do (no abort: the copy always lands)
        int never = 0;
        bool dummy = false;
        mbar_wait_or_abort(bar(BAR_QTMA), n_qtma & 1, lim, &never, &dummy);
        ++n_qtma;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_Q_READY));
    };

    TileIter it;
    it.init(p.seq_lens, p.max_blocks, b_first, blk_first);
    float m_g = -INFINITY, l_g = 0.f;   // running max / sum (this thread's columns) of this group's tiles
    int seg = 0;
    bool ok = true;
    load_q(it.b);

    for (int k = 0; k < ntiles && ok; ++k) {
      const bool first = (k == 0) || (it.blk == 0);
      const bool last = (k == ntiles - 1) || (it.blk == it.nb - 1);

      if (k % kGroups == g) {
        const int u = k / kGroups;  // use index of this group's exchange buffers
        const int n_valid = it.valid();
        // ---- partial scores of this CTA, this thread's columns
        if (!(kSpinSoftmax ? warp_spin(bar(BAR_S_FULL + g), u & 1)
                           : warp_wait(bar(BAR_S_FULL + g), u & 1))) { ok = false; break; }
        if (group_lead) MLA_TR(k, 3);
        if (lane == 0) { MLA_TRMAX(k, 19); MLA_TRMIN(k, 20); }
        tc_fence_after();
        uint32_t r[kCols];
#pragma unroll
        for (int c = 0; c < kCols / 16; ++c)
          tmem_ld16(tl + kColS + kCols * hf + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&r[16 * c]));
        tmem_wait_ld();
        if (group_lead) MLA_TR(k, 9);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) { MLA_TRMAX(k, 18); mbar_arrive(bar(BAR_S_EMPTY)); }

        // ---- exchange with the peer CTA
        // (no data comes back with this signal, so a CTA-scope wait suffices)
        if (u >= 1 && !warp_wait(bar(BAR_PEER_FREE + g), (u - 1) & 1)) { ok = false; break; }
        if (group_lead) MLA_TR(k, 10);
        // both CTAs keep only the top 24 bits of each partial (their own and
        // the peer's), so the two sums stay bit-identical; the freed low byte
        // of every value sent carries the use tag (1..255)
        const uint32_t tag = (uint32_t)(u % 255) + 1u;
#pragma unroll
        for (int i = 0; i < kCols; ++i) r[i] &= 0xFFFFFF00u;
#pragma unroll
        for (int c = 0; c < kMyChunks; ++c)
          st_cluster_v4(peer_recv + c * 512, __uint_as_float(r[4 * c] | tag),
                        __uint_as_float(r[4 * c + 1] | tag), __uint_as_float(r[4 * c + 2] | tag),
                        __uint_as_float(r[4 * c + 3] | tag));
        if (group_lead) MLA_TR(k, 11);
        if (group_lead) MLA_TR(k, 4);
        // poll the local buffer until all of this thread's values carry the tag
        // (each 4-byte value is written atomically, so a tagged value is whole)
        {
          const long long t0 = clock64();
          bool got = false;
          // watch one chunk until it carries the tag (one load per round),
          // then check them all
          while (true) {
            uint32_t v0, v1, v2, v3;
            asm volatile("ld.volatile.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                         : "r"(my_recv_u32 + (kMyChunks - 1) * 512)
                         : "memory");
            const bool seen = ((v0 & 0xFFu) == tag) & ((v1 & 0xFFu) == tag) &
                              ((v2 & 0xFFu) == tag) & ((v3 & 0xFFu) == tag);
            if (__all_sync(0xffffffffu, seen)) break;
            if (*abort_flag || clock64() - t0 > lim) break;
          }
          while (true) {
            bool mine = true;
#pragma unroll
            for (int c = 0; c < kMyChunks; ++c) {
              uint32_t v0, v1, v2, v3;
              asm volatile("ld.volatile.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                           : "r"(my_recv_u32 + c * 512)
                           : "memory");
              mine &= ((v0 & 0xFFu) == tag) & ((v1 & 0xFFu) == tag) & ((v2 & 0xFFu) == tag) &
                      ((v3 & 0xFFu) == tag);
            }
            if (__all_sync(0xffffffffu, mine)) { got = true; break; }
            if (*abort_flag) break;
            if (clock64() - t0 > lim) {
              timed_out = true;
              if (lane == 0) MLA_SITE(3000 + warp);
              break;
            }
          }
          if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        }
        if (group_lead) MLA_TR(k, 5);
        // full score (log2 domain) in place: r <- (own partial + peer's) * scale
        float mt = -INFINITY;
        const f2_t scale2 = f2_make(p.scale_log2, p.scale_log2);
#pragma unroll
        for (int c = 0; c < kMyChunks; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(my_recv + c * 512);
          const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int kk = 4 * c + e;
            const f2_t own = f2_make(__uint_as_float(r[kk]), __uint_as_float(r[kk + 1]));
            const f2_t oth = f2_make(__uint_as_float(vv[e] & 0xFFFFFF00u),
                                     __uint_as_float(vv[e + 1] & 0xFFFFFF00u));
            float x0, x1;
            f2_split(f2_mul(f2_add(own, oth), scale2), x0, x1);
            r[kk] = __float_as_uint(x0);
            r[kk + 1] = __float_as_uint(x1);
          }
        }
        // the buffer may be refilled: tell the peer (the values are consumed)
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_relaxed(peer_free);
        // slots past the sequence end, and past this row's own position, get -inf
        const int lim = min(n_valid, it.len() - it.blk * kTok - c_row);
        if (lim < kTok) {
#pragma unroll
          for (int kk = 0; kk < kCols; ++kk)
            if (kCols * hf + kk >= lim) r[kk] = __float_as_uint(-INFINITY);
        }
#pragma unroll
        for (int kk = 0; kk < kCols; ++kk) mt = fmaxf(mt, __uint_as_float(r[kk]));
        if constexpr (kHalves > 1) {
          // row maximum over both halves: the first meeting makes sure that the
          // partner has read what this thread wrote for the group's previous tile
          pair_sync();
          hmax[(g * kHalves + hf) * 128 + row] = mt;
          pair_sync();
          mt = fmaxf(mt, hmax[(g * kHalves + (hf ^ 1)) * 128 + row]);
        }

        // ---- running maximum, handed over from the previous tile's group
        float m_prev = -INFINITY;
        if (!first) {
          const int kp = k - 1;
          if (!warp_wait(bar(BAR_MREADY + (kp & 1)), (kp >> 1) & 1)) { ok = false; break; }
          m_prev = mpub[(kp & 1) * 128 + row];
        }
        if (group_lead) MLA_TR(k, 6);
        float m_k = m_prev;
        bool resc = false;
        if (m_prev == -INFINITY) {
          m_k = mt;
        } else if (mt > m_prev + kTau) {
          m_k = mt;
          resc = true;
        }
        // every warp of the group arrives once it has read m_prev, so the
        // next writer of this slot (tile k + 1's group) cannot overwrite it early
        if (hf == 0) mpub[(k & 1) * 128 + row] = m_k;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_MREADY + (k & 1)));
        if (m_g != m_k) {
          if (m_g != -INFINITY) l_g *= exp2f(m_g - m_k);
          m_g = m_k;
        }

        // ---- P (bf16 pairs) in registers first, packed in place into r[0..kCols/2)
        f2_t psum2 = f2_make(0.f, 0.f);
        // a row that sees no slot yet keeps m = -inf: its P is 0
        const float nm = m_k == -INFINITY ? 0.f : -m_k;
        const f2_t negm = f2_make(nm, nm);
#pragma unroll
        for (int e = 0; e < kCols / 2; ++e) {
          const f2_t y = f2_add(f2_make(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1])), negm);
          float y0, y1;
          f2_split(y, y0, y1);
          const float p0 = ex2(y0), p1 = ex2(y1);
          psum2 = f2_add(psum2, f2_make(p0, p1));
          r[e] = pack_bf16x2(p0, p1);
        }
        {
          float s0, s1;
          f2_split(psum2, s0, s1);
          l_g += s0 + s1;
        }

        // ---- P buffer (k & 1) was read by the P.C MMA of tile k-2; waiting for it
        // also makes O(k-3) complete, so the rescale's wait on the other group's
        // barrier below cannot alias an older phase
        if (k >= 2 && !warp_wait(bar(BAR_O_DONE + ((k - 2) & 3)), ((k - 2) >> 2) & 1)) { ok = false; break; }
        if (group_lead) MLA_TR(k, 7);

        // ---- rescale O between P(k-1) C and P(k) C (rare); each half takes
        // its share of the 16 chunks of 16 columns
        if (__any_sync(0xffffffffu, resc)) {
          const int kp = k - 1;
          if (!warp_wait(bar(BAR_O_DONE + (kp & 3)), (kp >> 2) & 1)) { ok = false; break; }
          tc_fence_after();
          const float alpha = resc ? exp2f(m_prev - m_k) : 1.0f;
          for (int c = (16 / kHalves) * hf; c < (16 / kHalves) * (hf + 1); ++c) {
            uint32_t v[16];
            tmem_ld16(tl + kColO + 16 * c, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st16(tl + kColO + 16 * c, v);
          }
        }
        tc_fence_after();
        const uint32_t pcol = kColP + 32 * (k & 1) + (kCols / 2) * hf;
#pragma unroll
        for (int c = 0; c < kCols / 32; ++c)
          tmem_st16(tl + pcol + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&r[16 * c]));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) { MLA_TRMAX(k, 21); mbar_arrive(bar(BAR_P_FULL + (k & 1))); }
        if (group_lead) MLA_TR(k, 8);
      }

      if (last) {
        // ---- end of a segment: every softmax warp
        float* lms = lm + (seg & 1) * (kGroups * 128);
        float* lss = lsum + (seg & 1) * (kGroups * kHalves * 128);
        if (hf == 0) lms[g * 128 + row] = m_g;
        lss[(g * kHalves + hf) * 128 + row] = l_g;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_SEG));
        if (!warp_wait(bar(BAR_SEG), seg & 1)) { ok = false; break; }
        if (group_lead && g == 0) MLA_TR(k, 12);
        float M = -INFINITY;
#pragma unroll
        for (int gg = 0; gg < kGroups; ++gg) M = fmaxf(M, lms[gg * 128 + row]);
        float l = 0.f;
#pragma unroll
        for (int gg = 0; gg < kGroups; ++gg) {
          const float mg = lms[gg * 128 + row];
          if (mg != -INFINITY) {
            float lg = 0.f;
#pragma unroll
            for (int hh = 0; hh < kHalves; ++hh) lg += lss[(gg * kHalves + hh) * 128 + row];
            l += lg * exp2f(mg - M);
          }
        }
        const int b = it.b;
        // query of the next segment first: the next score MMA can start while
        // this segment's output is read out
        if (k + 1 < ntiles) {
          TileIter nx = it;
          nx.next();
          if (!warp_wait(bar(BAR_Q_FREE), seg & 1)) { ok = false; break; }
          tc_fence_after();
          load_q(nx.b);
          if (group_lead && g == 0) MLA_TR(k, 13);
        }
        // epilogue: O_r / l -> o_part slot (part + b); 16 chunks of 16 columns
        // split between the softmax threads of the row
        if (!warp_wait(bar(BAR_O_DONE + (k & 3)), (k >> 2) & 1)) { ok = false; break; }
        if (group_lead && g == 0) MLA_TR(k, 14);
        tc_fence_after();
        const int64_t slot = (int64_t)part + b;
        float* orow = p.o_part + (slot * p.h + (live ? grow : 0)) * 512 + rank * 256;
        // a row that saw no slot of this segment: output 0, lse -inf (weight 0)
        const float inv = l > 0.f ? 1.0f / l : 0.f;
        constexpr int kEpiChunks = 16 / (kGroups * kHalves);
        const int ec0 = (g * kHalves + hf) * kEpiChunks;
        for (int c = ec0; c < ec0 + kEpiChunks; ++c) {
          uint32_t v[16];
          tmem_ld16(tl + kColO + 16 * c, v);
          tmem_wait_ld();
          if (live) {
            float o[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __uint_as_float(v[e]) * inv;
            if (o32) {
              stg_v8(orow + 16 * c, o);
              stg_v8(orow + 16 * c + 8, o + 8);
            } else {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4)
                *reinterpret_cast<float4*>(orow + 16 * c + 4 * q4) =
                    make_float4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
            }
          }
        }
        if (live && rank == 0 && g == 0 && hf == 0)
          p.lse_part[slot * p.h + grow] = l > 0.f ? (M + log2f(l)) * kLn2 : -INFINITY;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_O_FREE));
        if (group_lead && g == 0) MLA_TR(k, 15);
        m_g = -INFINITY;
        l_g = 0.f;
        ++seg;
      }
      if (k + 1 < ntiles) it.next();
    }
    if (!ok) {
      fail();
      // the partner warp of this lane quarter may be held at one of the two
      // pair meetings of a tile: arrive twice so that it reaches a wait that
      // sees the abort flag
      if constexpr (kHalves > 1) {
        asm volatile("bar.arrive %0, 64;" ::"r"(1 + 4 * g + sub) : "memory");
        asm volatile("bar.arrive %0, 64;" ::"r"(1 + 4 * g + sub) : "memory");
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

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() { return tensor_map_encoder(); }

// 2-D bf16 view [rows, cols] with the given row pitch; box_cols x box_rows boxes,
// 128-byte swizzle for 64-column boxes and 64-byte swizzle for 32-column boxes.
bool make_tmap(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
               uint64_t row_pitch_bytes, uint32_t box_cols, uint32_t box_rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_pitch_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw =
      box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// compute capability major of the current device (0 if there is none)
int device_major() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return device_registry().value(
      dev,
      [dev]() {
        int major = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) {
          cudaGetLastError();
          major = 0;
        }
        return major;
      },
      0);
}

}  // namespace

#ifdef MLA_TRACE
extern "C" int mla_debug_set_trace(void* p) {
  return cudaMemcpyToSymbol(g_trace, &p, sizeof(p)) == cudaSuccess ? 0 : -1;
}
#endif

DeviceRegistry& device_registry() {
  static DeviceRegistry reg;
  return reg;
}

// The driver's tensor-map encoder (one entry point for every device of the
// process), looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag flag;
  std::call_once(flag, []() {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

bool tc_device() { return device_major() >= 10 && get_encode_fn() != nullptr; }

bool decode_tc_supported(int q_dtype, const mla_kv_cache& kv, int rows) {
  const bool lat_ok = kv.latent_dtype == MLA_BF16 || (kv.latent_dtype == MLA_FP8E4M3 && kv.scale);
  return q_dtype == MLA_BF16 && lat_ok && kv.rope_dtype == MLA_BF16 && kv.d_c == 512 &&
         kv.d_r == 64 && kv.block_size == kTok && rows >= 1 && tc_device();
}

namespace {

// e4m3 latent view [rows, 512] (bytes), boxes of 256 codes x 64 rows, no swizzle.
bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t row_pitch_bytes) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {512, rows};
  cuuint64_t strides[1] = {row_pitch_bytes};
  cuuint32_t box[2] = {256, 64};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool kFp8>
cudaError_t launch_variant(const CUtensorMap& tm_lat, const CUtensorMap& tm_rope,
                           const CUtensorMap& tm_q, const TcParams& prm, int num_pairs,
                           cudaStream_t s) {
  // the dynamic shared-memory limit is a per-device setting: once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int r = device_registry().once(dev, kFp8 ? kSetupDecodeFp8 : kSetupDecodeBf16, []() {
    return (int)cudaFuncSetAttribute(decode_tc_kernel<kFp8>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Cfg<kFp8>::kSmemAlloc);
  });
  if (r != 0) return r < 0 ? cudaErrorInvalidDevice : (cudaError_t)r;
  dim3 grid(2 * num_pairs);
  return launch_pdl(decode_tc_kernel<kFp8>, grid, dim3(Cfg<kFp8>::kThreads), Cfg<kFp8>::kSmemAlloc,
                    s, tm_lat, tm_rope, tm_q, prm);
}

}  // namespace

cudaError_t launch_decode_tc(const void* q_cat, const mla_kv_cache& kv,
                             const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                             int B, int q_len, int heads, int num_parts, float scale,
                             float* o_part, float* lse_part, int32_t* status, bool test_timeout,
                             cudaStream_t s) {
  const int h = q_len * heads;                 // query rows per sequence
  const int groups = (h + 127) / 128;          // CTA pairs per part
  const bool fp8 = kv.latent_dtype == MLA_FP8E4M3;
  CUtensorMap tm_lat, tm_rope, tm_q;
  const uint64_t rows = (uint64_t)kv.num_blocks * kv.block_size;
  const bool lat_ok =
      fp8 ? make_tmap_u8(&tm_lat, kv.latent, rows, (uint64_t)kv.latent_stride)
          : make_tmap(&tm_lat, kv.latent, 512, rows, (uint64_t)kv.latent_stride * 2, 64, 64);
  if (!lat_ok || !make_tmap(&tm_rope, kv.rope, 64, rows, (uint64_t)kv.rope_stride * 2, 32, 64) ||
      !make_tmap(&tm_q, q_cat, 576, (uint64_t)B * h, 576 * 2, 32, 128))
    return cudaErrorInvalidValue;
  TcParams prm;
  prm.q_cat = static_cast<const uint16_t*>(q_cat);
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.o_part = o_part;
  prm.lse_part = lse_part;
  prm.status = status;
  prm.kv_scale = kv.scale;
  prm.max_blocks = max_blocks;
  prm.B = B;
  prm.h = h;
  prm.heads = heads;
  prm.q_len = q_len;
  prm.num_parts = num_parts;
  prm.num_blocks = kv.num_blocks;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.wait_limit = 4000000000LL;  // about 2 s of SM clock
  prm.test_wait_limit = test_timeout ? 20000 : 0;  // about 10 us
  return fp8 ? launch_variant<true>(tm_lat, tm_rope, tm_q, prm, num_parts * groups, s)
             : launch_variant<false>(tm_lat, tm_rope, tm_q, prm, num_parts * groups, s);
}

}  // namespace mla
