// cpa_host.h -- host-side bookkeeping of the library that needs no GPU:
// a set-up step run once per device index (kernel attributes, the address of
// the static scratch), remembered per device so that one process can drive
// several GPUs through the same library instance.
#pragma once
#include <mutex>

namespace cpa {

constexpr int kMaxDevices = 64;

// Per-device result of a set-up step.  `run(dev, f)` calls `f(value&)` the
// first time it is asked for device `dev` (and again after a failure), under a
// lock; `f` returns 0 on success, and the value it filled in is kept for every
// later call on that device.  Returns `f`'s error, or `bad_device` for an
// index outside [0, kMaxDevices).
template <class T>
class PerDevice {
   public:
    template <class F>
    int run(int dev, int bad_device, F&& f, T* out = nullptr) {
        if (dev < 0 || dev >= kMaxDevices) return bad_device;
        std::lock_guard<std::mutex> lock(mu_);
        if (!done_[dev]) {
            T v{};
            const int e = f(v);
            if (e != 0) return e;
            value_[dev] = v;
            done_[dev] = true;
        }
        if (out) *out = value_[dev];
        return 0;
    }

   private:
    std::mutex mu_;
    bool done_[kMaxDevices] = {};
    T value_[kMaxDevices] = {};
};

}  // namespace cpa
