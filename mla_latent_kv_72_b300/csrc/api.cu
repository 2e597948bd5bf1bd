// C ABI of the MLA decode library: host-side argument checks and dispatch.
// Every check runs before any launch; a failing call launches nothing.
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool is_float_dtype(int dt) { return dt == MLA_F32 || dt == MLA_BF16; }

inline int from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return MLA_OK;
  cudaGetLastError();  // clear a sticky launch-configuration error so later calls are unaffected
  return MLA_ERR_LAUNCH;
}

int check_cache(const mla_kv_cache* kv) {
  if (!kv || !kv->latent || !kv->rope) return MLA_ERR_ARG;
  if (kv->num_blocks <= 0 || kv->block_size <= 0 || kv->d_c <= 0 || kv->d_r <= 0)
    return MLA_ERR_ARG;
  if (kv->d_c % 32 != 0 || kv->d_c > 1024 || kv->d_r % 2 != 0 || kv->d_r > 256)
    return MLA_ERR_SHAPE;
  if (kv->latent_dtype == MLA_FP8E4M3) {
    if (!kv->scale) return MLA_ERR_ARG;
    if (kv->rope_dtype != MLA_BF16) return MLA_ERR_DTYPE;
  } else if (!is_float_dtype(kv->latent_dtype) || kv->rope_dtype != kv->latent_dtype) {
    return MLA_ERR_DTYPE;
  }
  if (kv->latent_stride < kv->d_c || kv->rope_stride < kv->d_r) return MLA_ERR_SHAPE;
  const int lb = mla::dtype_bytes(kv->latent_dtype), rb = mla::dtype_bytes(kv->rope_dtype);
  if (!aligned16(kv->latent) || !aligned16(kv->rope) || (kv->latent_stride * lb) % 16 != 0 ||
      (kv->rope_stride * rb) % 16 != 0)
    return MLA_ERR_ALIGN;
  return MLA_OK;
}

}  // namespace

namespace mla {
// defined in combine_proj.cu
cudaError_t launch_combine_out_proj(const float* o_part, const float* lse_part,
                                    const int32_t* seq_lens, int block_size, int max_blocks,
                                    int B, int h, int num_parts, const void* w_uv, void* out,
                                    int out_dtype, void* o_lat, int o_dtype, float* lse,
                                    int32_t* status, cudaStream_t s);
}  // namespace mla

extern "C" {

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_ARG: return "invalid argument (null pointer, non-positive size or bad enum)";
    case MLA_ERR_ALIGN: return "pointer or row stride not 16-byte aligned";
    case MLA_ERR_DTYPE: return "unsupported dtype combination";
    case MLA_ERR_SHAPE: return "dimensions outside the supported range";
    case MLA_ERR_LAUNCH: return "CUDA launch error";
    case MLA_ERR_DEVICE: return "no usable CUDA device";
    default: return "unknown status";
  }
}

int mla_version(void) { return 100; }

double mla_cache_bytes_per_token(int latent_dtype, int rope_dtype, int d_c, int d_r,
                                 int block_size) {
  if (d_c <= 0 || d_r < 0 || block_size <= 0) return -1.0;
  if (latent_dtype < MLA_F32 || latent_dtype > MLA_FP8E4M3) return -1.0;
  if (!is_float_dtype(rope_dtype)) return -1.0;
  double b = (double)d_c * mla::dtype_bytes(latent_dtype) + (double)d_r * mla::dtype_bytes(rope_dtype);
  if (latent_dtype == MLA_FP8E4M3) b += 4.0 / block_size;
  return b;
}

int mla_absorb_q(const void* q_nope, const void* q_rope, const int32_t* q_pos, const void* w_uk,
                 void* q_cat, int B, int h, int d_nope, int d_c, int d_r, int dtype,
                 double rope_theta, void* stream) {
  if (!q_nope || !q_rope || !q_pos || !w_uk || !q_cat) return MLA_ERR_ARG;
  if (B <= 0 || h <= 0 || d_nope <= 0 || d_c <= 0 || d_r <= 0 || !(rope_theta > 0.0))
    return MLA_ERR_ARG;
  if (!is_float_dtype(dtype)) return MLA_ERR_DTYPE;
  if (d_c % 64 != 0 || d_c > 1024 || d_r % 2 != 0 || d_r > 256 || d_nope > 512)
    return MLA_ERR_SHAPE;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(q_cat))
    return MLA_ERR_ALIGN;
  if (dtype == MLA_BF16 && d_nope == 128 && d_c == 512 && d_r == 64 && mla::tc_device())
    return from_cuda(mla::launch_absorb_q_tc(q_nope, q_rope, q_pos, w_uk, q_cat, B, h, rope_theta,
                                             static_cast<cudaStream_t>(stream)));
  return from_cuda(mla::launch_absorb_q_simt(q_nope, q_rope, q_pos, w_uk, q_cat, B, h, d_nope,
                                             d_c, d_r, dtype, rope_theta,
                                             static_cast<cudaStream_t>(stream)));
}

int mla_decode_num_partials(int B, int num_parts) {
  if (B <= 0 || num_parts <= 0 || num_parts > MLA_MAX_PARTS) return MLA_ERR_ARG;
  return B + num_parts - 1;
}

}  // extern "C"

namespace {

// Checks and dispatch shared by the one-token and the multi-token decode.
int decode_impl(const void* q_cat, int q_dtype, const mla_kv_cache* kv,
                const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                int B, int q_len, int h, int num_parts, float softmax_scale, float* o_part,
                float* lse_part, int32_t* dev_status, unsigned flags, void* stream) {
  if (!q_cat || !block_table || !seq_lens || !o_part || !lse_part) return MLA_ERR_ARG;
  if (B <= 0 || h <= 0 || q_len <= 0 || num_parts <= 0 || max_blocks_per_seq <= 0)
    return MLA_ERR_ARG;
  if (flags != MLA_DECODE_AUTO && flags != MLA_DECODE_FORCE_SIMT &&
      flags != MLA_DECODE_TEST_WAIT_TIMEOUT)
    return MLA_ERR_ARG;
  int st = check_cache(kv);
  if (st != MLA_OK) return st;
  if (!is_float_dtype(q_dtype)) return MLA_ERR_DTYPE;
  if (q_dtype == MLA_F32 && kv->latent_dtype != MLA_F32) return MLA_ERR_DTYPE;
  if (q_dtype == MLA_BF16 && kv->latent_dtype == MLA_F32) return MLA_ERR_DTYPE;
  if (num_parts > MLA_MAX_PARTS || q_len > MLA_MAX_Q_LEN || (int64_t)q_len * h > 4096)
    return MLA_ERR_SHAPE;
  if (!aligned16(q_cat) || !aligned16(o_part)) return MLA_ERR_ALIGN;
  float scale = softmax_scale > 0.f ? softmax_scale : (float)(1.0 / sqrt(128.0 + kv->d_r));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool tc =
      flags != MLA_DECODE_FORCE_SIMT && mla::decode_tc_supported(q_dtype, *kv, q_len * h);
  // the diagnostic timeout exists only in the pipelined tensor-core kernel
  if (flags == MLA_DECODE_TEST_WAIT_TIMEOUT && !tc) return MLA_ERR_ARG;
  if (tc) {
    return from_cuda(mla::launch_decode_tc(q_cat, *kv, block_table, max_blocks_per_seq, seq_lens,
                                           B, q_len, h, num_parts, scale, o_part, lse_part,
                                           dev_status, flags == MLA_DECODE_TEST_WAIT_TIMEOUT, s));
  }
  return from_cuda(mla::launch_decode_simt(q_cat, q_dtype, *kv, block_table, max_blocks_per_seq,
                                           seq_lens, B, q_len, h, num_parts, scale, o_part,
                                           lse_part, dev_status, s));
}

}  // namespace

extern "C" {

int mla_decode_fwd(const void* q_cat, int q_dtype, const mla_kv_cache* kv,
                   const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                   int B, int h, int num_parts, float softmax_scale, float* o_part,
                   float* lse_part, int32_t* dev_status, unsigned flags, void* stream) {
  return decode_impl(q_cat, q_dtype, kv, block_table, max_blocks_per_seq, seq_lens, B, 1, h,
                     num_parts, softmax_scale, o_part, lse_part, dev_status, flags, stream);
}

int mla_decode_fwd_multi(const void* q_cat, int q_dtype, const mla_kv_cache* kv,
                         const int32_t* block_table, int max_blocks_per_seq,
                         const int32_t* seq_lens, int B, int q_len, int h, int num_parts,
                         float softmax_scale, float* o_part, float* lse_part,
                         int32_t* dev_status, unsigned flags, void* stream) {
  return decode_impl(q_cat, q_dtype, kv, block_table, max_blocks_per_seq, seq_lens, B, q_len, h,
                     num_parts, softmax_scale, o_part, lse_part, dev_status, flags, stream);
}

int mla_combine(const float* o_part, const float* lse_part, const int32_t* seq_lens,
                int block_size, int max_blocks_per_seq, int B, int h, int d_c, int num_parts,
                void* o_lat, int o_dtype, float* lse, void* stream) {
  if (!o_part || !lse_part || !o_lat || !seq_lens) return MLA_ERR_ARG;
  if (B <= 0 || h <= 0 || d_c <= 0 || num_parts <= 0 || block_size <= 0 ||
      max_blocks_per_seq <= 0)
    return MLA_ERR_ARG;
  if (!is_float_dtype(o_dtype)) return MLA_ERR_DTYPE;
  if (d_c % 4 != 0 || d_c > 2048 || num_parts > MLA_MAX_PARTS) return MLA_ERR_SHAPE;
  if (!aligned16(o_part) || !aligned16(o_lat)) return MLA_ERR_ALIGN;
  return from_cuda(mla::launch_combine(o_part, lse_part, seq_lens, block_size,
                                       max_blocks_per_seq, B, h, d_c, num_parts, o_lat, o_dtype,
                                       lse, static_cast<cudaStream_t>(stream)));
}

int mla_combine_out_proj(const float* o_part, const float* lse_part, const int32_t* seq_lens,
                         int block_size, int max_blocks_per_seq, int B, int h, int d_c,
                         int num_parts, const void* w_uv, int d_v, void* out, int out_dtype,
                         void* o_lat, int o_dtype, float* lse, int32_t* dev_status,
                         void* stream) {
  if (!o_part || !lse_part || !seq_lens || !w_uv || !out) return MLA_ERR_ARG;
  if (B <= 0 || h <= 0 || num_parts <= 0 || block_size <= 0 || max_blocks_per_seq <= 0)
    return MLA_ERR_ARG;
  if (!is_float_dtype(out_dtype) || (o_lat && !is_float_dtype(o_dtype))) return MLA_ERR_DTYPE;
  if (d_c != 512 || d_v != 128 || h > 65535 || num_parts > MLA_MAX_PARTS) return MLA_ERR_SHAPE;
  if (!aligned16(o_part) || !aligned16(w_uv) || (o_lat && !aligned16(o_lat)))
    return MLA_ERR_ALIGN;
  if (!mla::tc_device()) return MLA_ERR_DEVICE;
  return from_cuda(mla::launch_combine_out_proj(
      o_part, lse_part, seq_lens, block_size, max_blocks_per_seq, B, h, num_parts, w_uv, out,
      out_dtype, o_lat, o_dtype, lse, dev_status, static_cast<cudaStream_t>(stream)));
}

int mla_out_proj(const void* o_lat, const void* w_uv, void* out, int B, int h, int d_c, int d_v,
                 int in_dtype, int out_dtype, void* stream) {
  if (!o_lat || !w_uv || !out) return MLA_ERR_ARG;
  if (B <= 0 || h <= 0 || d_c <= 0 || d_v <= 0) return MLA_ERR_ARG;
  if (!is_float_dtype(in_dtype) || !is_float_dtype(out_dtype)) return MLA_ERR_DTYPE;
  if (d_c % 64 != 0 || d_c > 1024 || d_v > 1024) return MLA_ERR_SHAPE;
  if (!aligned16(o_lat) || !aligned16(w_uv) || !aligned16(out)) return MLA_ERR_ALIGN;
  if (in_dtype == MLA_BF16 && d_c == 512 && d_v == 128 && mla::tc_device())
    return from_cuda(mla::launch_out_proj_tc(o_lat, w_uv, out, B, h, out_dtype,
                                             static_cast<cudaStream_t>(stream)));
  return from_cuda(mla::launch_out_proj_simt(o_lat, w_uv, out, B, h, d_c, d_v, in_dtype,
                                             out_dtype, static_cast<cudaStream_t>(stream)));
}

size_t mla_linear_workspace_bytes(int M, int K, int N) {
  if (M <= 0 || K <= 0 || N <= 0 || K % 64 != 0 || N % 128 != 0) return 0;
  const int sp = mla::linear_splits(M, K, N);
  return sp > 1 ? (size_t)sp * (size_t)M * (size_t)N * sizeof(float) : 0;
}

int mla_linear(const void* x, const void* w, void* y, int M, int K, int N, int y_dtype,
               void* workspace, size_t workspace_bytes, void* stream) {
  if (!x || !w || !y) return MLA_ERR_ARG;
  if (M <= 0 || K <= 0 || N <= 0) return MLA_ERR_ARG;
  if (!is_float_dtype(y_dtype)) return MLA_ERR_DTYPE;
  if (K % 64 != 0 || N % 128 != 0 || K > (1 << 20) || N > (1 << 20)) return MLA_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return MLA_ERR_ALIGN;
  const size_t need = mla_linear_workspace_bytes(M, K, N);
  if (need > 0 && (!workspace || workspace_bytes < need)) return MLA_ERR_ARG;
  if (need > 0 && !aligned16(workspace)) return MLA_ERR_ALIGN;
  if (!mla::tc_device()) return MLA_ERR_DEVICE;
  return from_cuda(mla::launch_linear_tc(x, w, y, M, K, N, y_dtype,
                                         static_cast<float*>(workspace),
                                         static_cast<cudaStream_t>(stream)));
}

int mla_fold_uv_into_o(const void* w_uv, const void* w_o, void* w_fold, int h, int d_c, int d_v,
                       int d_model, void* stream) {
  if (!w_uv || !w_o || !w_fold) return MLA_ERR_ARG;
  if (h <= 0 || d_c <= 0 || d_v <= 0 || d_model <= 0) return MLA_ERR_ARG;
  if (d_c != 512 || d_v != 128) return MLA_ERR_SHAPE;
  if (!aligned16(w_uv) || !aligned16(w_o) || !aligned16(w_fold)) return MLA_ERR_ALIGN;
  if (!mla::tc_device()) return MLA_ERR_DEVICE;
  return from_cuda(mla::launch_fold_uv_o_tc(w_uv, w_o, w_fold, h, d_model,
                                            static_cast<cudaStream_t>(stream)));
}

int mla_prefill_query(const void* q_nope, const void* q_rope, const int32_t* cu_seqlens, int B,
                      int max_len, int h, double rope_theta, void* q, void* stream) {
  if (!q_nope || !q_rope || !cu_seqlens || !q) return MLA_ERR_ARG;
  if (B <= 0 || max_len < 0 || h <= 0 || !(rope_theta > 0.0)) return MLA_ERR_ARG;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(q)) return MLA_ERR_ALIGN;
  if (max_len == 0) return MLA_OK;
  return from_cuda(mla::launch_prefill_query(q_nope, q_rope, cu_seqlens, B, max_len, h,
                                             rope_theta, q, static_cast<cudaStream_t>(stream)));
}

int mla_prefill_fwd(const void* q, const void* k_nope, const void* k_rope, const void* v,
                    const int32_t* cu_seqlens, int B, int max_len, int64_t total_rows, int h,
                    float softmax_scale, void* out, int out_dtype, float* lse,
                    int32_t* dev_status, void* stream) {
  if (!q || !k_nope || !k_rope || !v || !cu_seqlens || !out) return MLA_ERR_ARG;
  if (B <= 0 || max_len < 0 || total_rows <= 0 || h <= 0) return MLA_ERR_ARG;
  if (!is_float_dtype(out_dtype)) return MLA_ERR_DTYPE;
  if (h > 65535 || B > 65535 || total_rows > (int64_t)1 << 31) return MLA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k_nope) || !aligned16(k_rope) || !aligned16(v) ||
      !aligned16(out))
    return MLA_ERR_ALIGN;
  if (!mla::tc_device()) return MLA_ERR_DEVICE;
  if (max_len == 0) return MLA_OK;
  const float scale = softmax_scale > 0.f ? softmax_scale : (float)(1.0 / sqrt(192.0));
  return from_cuda(mla::launch_prefill_tc(q, k_nope, k_rope, v, cu_seqlens, B, max_len, h,
                                          total_rows, scale, out, out_dtype, lse, dev_status,
                                          static_cast<cudaStream_t>(stream)));
}

int mla_cache_fill(const void* c_kv, const void* k_rope, int src_dtype,
                   const int32_t* cu_seqlens, int B, int max_len, const int32_t* block_table,
                   int max_blocks_per_seq, const mla_kv_cache* kv, double rope_theta,
                   int32_t* dev_status, void* stream) {
  if (!c_kv || !k_rope || !cu_seqlens || !block_table) return MLA_ERR_ARG;
  if (B <= 0 || max_len < 0 || max_blocks_per_seq <= 0 || !(rope_theta > 0.0)) return MLA_ERR_ARG;
  int st = check_cache(kv);
  if (st != MLA_OK) return st;
  if (!is_float_dtype(src_dtype)) return MLA_ERR_DTYPE;
  if (kv->latent_dtype == MLA_FP8E4M3 ? src_dtype != MLA_BF16 : src_dtype != kv->latent_dtype)
    return MLA_ERR_DTYPE;
  return from_cuda(mla::launch_cache_fill(c_kv, k_rope, src_dtype, cu_seqlens, B, max_len,
                                          block_table, max_blocks_per_seq, *kv, rope_theta,
                                          dev_status, static_cast<cudaStream_t>(stream)));
}

int mla_cache_append(const void* c_new, const void* k_rope, int src_dtype, const int32_t* pos,
                     int B, const int32_t* block_table, int max_blocks_per_seq,
                     const mla_kv_cache* kv, double rope_theta, int32_t* dev_status,
                     void* stream) {
  if (!c_new || !k_rope || !pos || !block_table) return MLA_ERR_ARG;
  if (B <= 0 || max_blocks_per_seq <= 0 || !(rope_theta > 0.0)) return MLA_ERR_ARG;
  int st = check_cache(kv);
  if (st != MLA_OK) return st;
  if (!is_float_dtype(src_dtype)) return MLA_ERR_DTYPE;
  if (kv->latent_dtype == MLA_FP8E4M3 ? src_dtype != MLA_BF16 : src_dtype != kv->latent_dtype)
    return MLA_ERR_DTYPE;
  if (!aligned16(c_new) || !aligned16(k_rope)) return MLA_ERR_ALIGN;
  return from_cuda(mla::launch_cache_append(c_new, k_rope, src_dtype, pos, B, block_table,
                                            max_blocks_per_seq, *kv, rope_theta, dev_status,
                                            static_cast<cudaStream_t>(stream)));
}

int mla_paged_gather(const mla_kv_cache* kv, const int32_t* block_table, int max_blocks_per_seq,
                     const int32_t* cu_seqlens, int B, int max_len, void* latent_out,
                     void* rope_out, int32_t* dev_status, void* stream) {
  if (!block_table || !cu_seqlens) return MLA_ERR_ARG;
  if (B <= 0 || max_len < 0 || max_blocks_per_seq <= 0) return MLA_ERR_ARG;
  int st = check_cache(kv);
  if (st != MLA_OK) return st;
  return from_cuda(mla::launch_paged_gather(*kv, block_table, max_blocks_per_seq, cu_seqlens, B,
                                            max_len, latent_out, rope_out, dev_status,
                                            static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
