// kvq_context_cache.h -- a value computed once per (device, CUDA context).
//
// Kernel attributes (the dynamic shared-memory limit), occupancy and the
// device address of a module symbol belong to the context they were taken
// in.  A process may drive several devices, and cudaDeviceReset replaces a
// device's context, so such values are cached per device together with the
// identity of the context they came from, and recomputed when the current
// context is a different one.  Plain C++ (no CUDA headers), so the logic is
// testable on a host without a GPU.
#pragma once

#include <mutex>

namespace kvq {

constexpr int kMaxDevices = 64;

template <class T>
class ContextCache {
 public:
  // The value for device `dev` under context `ctx` (0 = unknown).  When the
  // slot holds a value taken under the same known context it is returned;
  // otherwise setup(T*) -> bool computes it, and on success it is stored
  // with the context ctx_after() reports (the setup may be what made a
  // context current).  False when dev is out of range or setup fails.
  template <class Setup, class CtxAfter>
  bool get(int dev, unsigned long long ctx, T* out, Setup setup, CtxAfter ctx_after) {
    if (dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(mu_);
    if (ctx != 0 && ctx_[dev] == ctx) {
      *out = value_[dev];
      return true;
    }
    T v{};
    if (!setup(&v)) return false;
    value_[dev] = v;
    ctx_[dev] = ctx_after();
    *out = v;
    return true;
  }

 private:
  unsigned long long ctx_[kMaxDevices] = {};
  T value_[kMaxDevices] = {};
  std::mutex mu_;
};

}  // namespace kvq
