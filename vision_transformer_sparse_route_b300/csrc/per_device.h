// per_device.h -- a set of (device, key) pairs for which a one-time set-up
// step (a kernel attribute raised with cudaFuncSetAttribute, which holds per
// device context) has been done. Plain C++, no CUDA: the host code asks
// `done(dev, key)` before the step and calls `mark(dev, key)` after it
// succeeded, so that every device gets its own set-up.
#pragma once

#include <algorithm>
#include <mutex>
#include <utility>
#include <vector>

namespace bra {

class PerDeviceOnce {
 public:
  bool done(int dev, const void *key) const {
    std::lock_guard<std::mutex> lock(mu_);
    return std::find(seen_.begin(), seen_.end(), std::make_pair(dev, key)) != seen_.end();
  }
  void mark(int dev, const void *key) {
    std::lock_guard<std::mutex> lock(mu_);
    if (std::find(seen_.begin(), seen_.end(), std::make_pair(dev, key)) == seen_.end())
      seen_.emplace_back(dev, key);
  }

 private:
  mutable std::mutex mu_;
  std::vector<std::pair<int, const void *>> seen_;
};

}  // namespace bra
