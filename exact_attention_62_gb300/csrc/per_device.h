// per_device.h -- a value computed once per device and cached, for the
// library's launch set-up (kernel attributes, register counts, SM counts,
// occupancy).  Plain C++ without CUDA types, so that the host tests compile
// and check it on its own.
#pragma once

#include <mutex>

namespace attn_host {

// Devices a process may drive; every per-device cache is this large.
constexpr int kMaxDevices = 64;

// The value of device `dev`: made by `make(&value)` (which returns true on
// success) on the first call for that device, then returned from the cache.
// Devices never share an entry: a process that drives several GPUs sets each
// one up.  A failed `make` is not cached, so the next call retries; a device
// outside [0, kMaxDevices) gets no value.  get returns false in both cases.
// Thread-safe: `make` runs under the cache's lock.
template <typename T>
class PerDevice {
  public:
    template <typename Make>
    bool get(int dev, T* out, Make&& make) {
        if (dev < 0 || dev >= kMaxDevices) return false;
        std::lock_guard<std::mutex> lock(mu_);
        if (!done_[dev]) {
            T v{};
            if (!make(&v)) return false;
            val_[dev] = v;
            done_[dev] = true;
        }
        *out = val_[dev];
        return true;
    }

  private:
    std::mutex mu_;
    bool done_[kMaxDevices] = {};
    T val_[kMaxDevices] = {};
};

}  // namespace attn_host
