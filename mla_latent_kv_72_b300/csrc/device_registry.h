// Per-device, thread-safe one-time set-up records of the library.
//
// Some launch settings live per device in CUDA: a kernel's dynamic
// shared-memory limit (cudaFuncSetAttribute applies to the current device
// only) and the device's compute capability.  A process that drives several
// GPUs must therefore set each device up once, and host threads that make
// their first calls at the same time must not race on the records.  This
// header is plain C++ (no CUDA types), so that the bookkeeping can be
// compiled and tested on a machine without a GPU.
#pragma once

#include <stdint.h>

#include <mutex>

namespace mla {

constexpr int kMaxDevices = 64;   // device ordinals 0 .. 63
constexpr int kMaxSetupKeys = 64; // distinct one-time settings per device

class DeviceRegistry {
 public:
  // Runs setup() for (device, key) until one run returns 0, then never again;
  // returns 0 once the setting is in place, setup()'s non-zero result if it
  // failed (a later call retries), or -1 for an ordinal or key out of range.
  template <class F>
  int once(int device, int key, F&& setup) {
    if (device < 0 || device >= kMaxDevices || key < 0 || key >= kMaxSetupKeys) return -1;
    const uint64_t bit = uint64_t(1) << key;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[device] & bit) return 0;
    const int r = setup();
    if (r == 0) done_[device] |= bit;
    return r;
  }

  // A per-device integer computed once by compute() (e.g. the compute
  // capability); fallback for an ordinal out of range.
  template <class F>
  int value(int device, F&& compute, int fallback) {
    if (device < 0 || device >= kMaxDevices) return fallback;
    std::lock_guard<std::mutex> lock(mu_);
    if (!have_[device]) {
      val_[device] = compute();
      have_[device] = true;
    }
    return val_[device];
  }

 private:
  std::mutex mu_;
  uint64_t done_[kMaxDevices] = {};
  int val_[kMaxDevices] = {};
  bool have_[kMaxDevices] = {};
};

// The library's one registry (defined in decode_tc.cu).
DeviceRegistry& device_registry();

// Keys of the one-time settings.
enum SetupKey : int {
  kSetupDecodeBf16 = 0,   // dynamic shared memory of the bf16-cache decode kernel
  kSetupDecodeFp8 = 1,    // ... of the FP8-latent decode kernel
  kSetupGemmMN = 2,       // ... of the per-head GEMM, MN-major A (absorb)
  kSetupGemmK = 3,        // ... of the per-head GEMM, K-major A (out_proj)
  kSetupAppend = 4,       // ... of the cache-append kernel
  kSetupPrefill = 5,      // ... of the prefill attention kernel
  kSetupCombineProj = 6,  // ... of the merged combine + output projection kernel
  kSetupKeyCount
};

}  // namespace mla
