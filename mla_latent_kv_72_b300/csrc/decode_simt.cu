// mla_decode_fwd, CUDA-core (SIMT) kernel: float32 arithmetic for every
// supported cache dtype.  It is the kernel of the float32 workload and the
// general fallback for shapes the tensor-core kernel does not take.
//
// Attention of one query token over the latent cache in the decode-time MQA
// form (kexue.fm "From MHA, MQA, GQA to MLA", eq. mla-mqa), online softmax over
// 32-token tiles, one warp per head, over the same balanced part partition of
// the block stream as the tensor-core kernel.
#include <math.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;          // heads per CTA
constexpr int kTile = 32;          // tokens per tile (one per lane)

struct SimtArgs {
  const void* q_cat;
  int q_dtype;
  mla_kv_cache kv;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* seq_lens;
  int B, h, num_parts;   // h = q_len * heads query rows per sequence (row j * heads + s)
  int heads, q_len;
  float scale;
  float* o_part;
  float* lse_part;
  int32_t* status;
};

// grid: (num_parts, ceil(h / kWarps)); block: 32 * kWarps threads.  CTA (p, hg)
// runs part p of the block stream for heads hg * kWarps .. + kWarps - 1, one
// segment (the part's blocks of one sequence) after another.
// smem: q [kWarps][dqk] and the current tile K [kTile][dqk + 1], both float32.
__global__ void __launch_bounds__(32 * kWarps) decode_simt_kernel(SimtArgs a) {
  extern __shared__ float smem[];
  __shared__ long long s_info[4];
  const int d_c = a.kv.d_c, d_r = a.kv.d_r, dqk = d_c + d_r;
  const int ks = dqk + 1;
  float* sq = smem;                       // [kWarps][dqk]
  float* sk = smem + kWarps * dqk;        // [kTile][ks]
  const int p = blockIdx.x, hg = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int s = hg * kWarps + warp;
  const int bs = a.kv.block_size;

  if (warp == 0) {
    long long T = warp_stream_scan(a.seq_lens, a.B, bs, a.max_blocks, -1, -1, nullptr, nullptr,
                                   nullptr);
    const int P = (int)(T < a.num_parts ? T : a.num_parts);
    long long g0 = 0, g1 = 0, sb = 0;
    int b0 = -1;
    if (p < P) {
      g0 = part_begin(T, P, p);
      g1 = part_begin(T, P, p + 1);
      warp_stream_scan(a.seq_lens, a.B, bs, a.max_blocks, -1, g0, nullptr, &b0, &sb);
    }
    if (lane == 0) {
      s_info[0] = b0;
      s_info[1] = g0 - sb;  // first logical block within sequence b0
      s_info[2] = g1 - g0;  // blocks of this part
      if (p == 0)
        for (int b = 0; b < a.B; ++b)
          if (a.seq_lens[b] > a.max_blocks * bs) set_status(a.status, MLA_DEV_BAD_LENGTH);
    }
  }
  __syncthreads();
  int b = (int)s_info[0];
  if (b < 0) return;
  int blk = (int)s_info[1];
  long long left = s_info[2];

  for (int i = threadIdx.x; i < kWarps * dqk; i += blockDim.x) sq[i] = 0.f;

  constexpr int kMaxPerLane = 32;     // d_c / 32 <= 32
  const int per_lane = d_c / 32;
  int loaded_b = -1;
  while (left > 0) {
    const int nb = seq_blocks(a.seq_lens, b, bs, a.max_blocks);
    if (nb == 0) { ++b; continue; }
    const int take = (int)((long long)(nb - blk) < left ? (nb - blk) : left);
    const int L = min(max(a.seq_lens[b], 0), a.max_blocks * bs);
    const int t_begin = blk * bs;
    const int t_end = min((blk + take) * bs, L);

    if (loaded_b != b) {
      __syncthreads();  // previous segment's readers of sq are done
      for (int i = threadIdx.x; i < kWarps * dqk; i += blockDim.x) {
        int w = i / dqk, d = i % dqk;
        int hs = hg * kWarps + w;
        sq[i] = hs < a.h ? load_as_f32(a.q_cat, a.q_dtype, ((int64_t)b * a.h + hs) * dqk + d) : 0.f;
      }
      loaded_b = b;
    }

    float o[kMaxPerLane];
#pragma unroll
    for (int k = 0; k < kMaxPerLane; ++k) o[k] = 0.f;
    float m = -INFINITY, l = 0.f;

    for (int t0 = t_begin; t0 < t_end; t0 += kTile) {
      __syncthreads();  // previous tile consumed (and q written on the first pass)
      for (int r = warp; r < kTile; r += kWarps) {
        int t = t0 + r;
        float* row = sk + r * ks;
        if (t < t_end) {
          int pb = a.block_table[(int64_t)b * a.max_blocks + t / bs];
          if (pb < 0 || pb >= a.kv.num_blocks) {
            set_status(a.status, MLA_DEV_BAD_BLOCK);
            for (int d = lane; d < dqk; d += 32) row[d] = 0.f;
            continue;
          }
          int64_t slot = (int64_t)pb * bs + (t % bs);
          float sc = 1.f;
          if (a.kv.latent_dtype == MLA_FP8E4M3) sc = a.kv.scale[pb];
          for (int d = lane; d < d_c; d += 32)
            row[d] = load_as_f32(a.kv.latent, a.kv.latent_dtype, slot * a.kv.latent_stride + d) * sc;
          for (int d = lane; d < d_r; d += 32)
            row[d_c + d] = load_as_f32(a.kv.rope, a.kv.rope_dtype, slot * a.kv.rope_stride + d);
        } else {
          for (int d = lane; d < dqk; d += 32) row[d] = 0.f;
        }
      }
      __syncthreads();
      if (s < a.h) {
        // score of token (t0 + lane)
        const float* qv = sq + warp * dqk;
        const float* kr = sk + lane * ks;
        float acc = 0.f;
        for (int d = 0; d < dqk; ++d) acc = fmaf(qv[d], kr[d], acc);
        // slots past the sequence end, and past this row's own position
        // (token j = s / heads sits q_len - 1 - j before the last row), get -inf
        const int lim = min(t_end, L - (a.q_len - 1 - s / a.heads));
        float sc = (t0 + lane < lim) ? acc * a.scale : -INFINITY;
        float tmax = sc;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
        float m_new = fmaxf(m, tmax);
        float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
        float pr_ = (sc == -INFINITY) ? 0.f : expf(sc - m_new);
        float psum = pr_;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
        l = l * alpha + psum;
        m = m_new;
#pragma unroll
        for (int k = 0; k < kMaxPerLane; ++k) o[k] *= alpha;
        for (int r = 0; r < kTile; ++r) {
          float pr = __shfl_sync(0xffffffffu, pr_, r);
          const float* row = sk + r * ks;
#pragma unroll
          for (int k = 0; k < kMaxPerLane; ++k)
            if (k < per_lane) o[k] = fmaf(pr, row[lane + 32 * k], o[k]);
        }
      }
    }

    if (s < a.h) {
      const int64_t slot = (int64_t)p + b;
      int64_t ob = (slot * a.h + s) * d_c;
      float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int k = 0; k < kMaxPerLane; ++k)
        if (k < per_lane) a.o_part[ob + lane + 32 * k] = o[k] * inv;
      if (lane == 0) a.lse_part[slot * a.h + s] = l > 0.f ? m + logf(l) : -INFINITY;
    }
    left -= take;
    ++b;
    blk = 0;
  }
}

}  // namespace

cudaError_t launch_decode_simt(const void* q_cat, int q_dtype, const mla_kv_cache& kv,
                               const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                               int B, int q_len, int heads, int num_parts, float scale,
                               float* o_part, float* lse_part, int32_t* status, cudaStream_t s) {
  const int h = q_len * heads;
  SimtArgs a{q_cat, q_dtype, kv, block_table, max_blocks, seq_lens, B, h, num_parts,
             heads, q_len, scale, o_part, lse_part, status};
  const int dqk = kv.d_c + kv.d_r;
  size_t smem = sizeof(float) * ((size_t)kWarps * dqk + (size_t)kTile * (dqk + 1));
  cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(num_parts, ceil_div(h, kWarps));
  decode_simt_kernel<<<grid, 32 * kWarps, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
