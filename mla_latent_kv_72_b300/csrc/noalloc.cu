// mla_decode_attend_noalloc: attention of the decode step (mla_decode_fwd
// followed by mla_combine) for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside another
// framework's memory pool or allocator hooks, a runtime that forbids
// allocation on its hot path, or a host that holds a fixed device budget.
// The split-KV partials that mla_decode_fwd writes and mla_combine reads are
// pure scratch for such a caller, so this entry point keeps them in a
// file-scope device array instead of caller-provided buffers.  The caller
// still passes every input and output.
//
// The array is fixed at kScratchPartFloats + kScratchLseFloats floats
// (64 MiB + 4 MiB); every GPU that loads the library holds it until the process
// exits.  All calls share it: calls that overlap on the GPU (on different
// streams, or from different host threads) race on it.  Nothing in it has to
// start at zero: every partial slot that the combine reads is written by the
// decode of the same call first.  Host code cannot use the array's name as a
// device address, so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current; make that first call
// before any stream capture.  The address is kept per device together with
// the unique id of the CUDA context it was looked up in: after a device reset
// (a new primary context, where the module and the array may sit elsewhere)
// the next call looks it up again.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "device_registry.h"

namespace mla {
namespace {

constexpr size_t kScratchPartFloats = size_t(16) << 20;  // o_part: slots * h * d_c
constexpr size_t kScratchLseFloats = size_t(1) << 20;    // lse_part: slots * h
static __device__ __align__(256) float g_scratch[kScratchPartFloats + kScratchLseFloats];

std::mutex g_mu;
float* g_addr[kMaxDevices] = {nullptr};
unsigned long long g_ctx_id[kMaxDevices] = {0};

// Unique id of the calling thread's current CUDA context (0 if none can be had).
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag flag;
  std::call_once(flag, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    cudaGetLastError();
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
      get_id(ctx, &id) == CUDA_SUCCESS)
    return id;
  return 0;
}

// Device address of g_scratch on the current device, looked up once per
// (device, context).
cudaError_t scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr || ctx == 0 || g_ctx_id[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = static_cast<float*>(p);
    // the look-up makes the runtime's primary context current if this thread
    // had none, so the id is read again after it
    g_ctx_id[dev] = current_context_id();
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace mla

namespace {
inline bool aligned16_na(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

extern "C" int mla_decode_attend_noalloc(const void* q_cat, int q_dtype, const mla_kv_cache* kv,
                                         const int32_t* block_table, int max_blocks_per_seq,
                                         const int32_t* seq_lens, int B, int h, int num_parts,
                                         float softmax_scale, void* o_lat, int o_dtype, float* lse,
                                         int32_t* dev_status, void* stream) {
  if (!q_cat || !kv || !block_table || !seq_lens || !o_lat) return MLA_ERR_ARG;
  if (B <= 0 || h <= 0 || num_parts <= 0 || max_blocks_per_seq <= 0) return MLA_ERR_ARG;
  if (num_parts > MLA_MAX_PARTS) return MLA_ERR_SHAPE;
  if (!(o_dtype == MLA_F32 || o_dtype == MLA_BF16)) return MLA_ERR_DTYPE;
  if (kv->d_c <= 0 || kv->d_c % 4 != 0) return MLA_ERR_SHAPE;
  // sizes beyond the fixed scratch array are rejected before anything runs
  const size_t slots = (size_t)B + (size_t)num_parts - 1;
  if (slots * (size_t)h * (size_t)kv->d_c > mla::kScratchPartFloats ||
      slots * (size_t)h > mla::kScratchLseFloats)
    return MLA_ERR_SHAPE;
  if (!aligned16_na(o_lat)) return MLA_ERR_ALIGN;
  float* scratch = nullptr;
  if (mla::scratch_address(&scratch) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_DEVICE;
  }
  float* o_part = scratch;
  float* lse_part = scratch + mla::kScratchPartFloats;
  // the decode and the combine through their own entry points (argument
  // checks included); neither allocates
  int st = mla_decode_fwd(q_cat, q_dtype, kv, block_table, max_blocks_per_seq, seq_lens, B, h,
                          num_parts, softmax_scale, o_part, lse_part, dev_status,
                          MLA_DECODE_AUTO, stream);
  if (st != MLA_OK) return st;
  return mla_combine(o_part, lse_part, seq_lens, kv->block_size, max_blocks_per_seq, B, h,
                     kv->d_c, num_parts, o_lat, o_dtype, lse, stream);
}
