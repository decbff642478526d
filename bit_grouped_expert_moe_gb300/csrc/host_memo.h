// Host-side memos of one-time launch set-up, kept per device and per CUDA
// context: the dynamic shared-memory limit raised for a kernel, and a device
// array's address. Both belong to one context on one device, so a memo
// recorded on device 0 says nothing about device 1, and one recorded before
// a cudaDeviceReset (after which the runtime makes a new primary context,
// reloads the module and may place a __device__ array elsewhere) says nothing
// about the context that follows. Every entry is keyed by the device index
// and the context's identifier; a different identifier makes the set-up run
// again. Access is serialised by a mutex, so host threads may launch
// concurrently.
//
// This header has no CUDA dependency: the set-up step is passed in as a
// callable returning 0 on success, which lets a plain C++ test drive it.
#pragma once

#include <mutex>

namespace bgmoe {

constexpr int kMaxDevices = 64;

// Whether a grid whose blocks wait for one another (each polls data that
// other blocks write, with no grid barrier the runtime would check) can have
// every block resident at once: `blocks_per_sm` is the occupancy the runtime
// reports for the kernel's block size and shared memory. A launch that fails
// this is refused, not attempted: its resident blocks would wait until their
// deadline for blocks that never start.
inline bool all_blocks_resident(int blocks_per_sm, int sm_count, int grid) {
  return blocks_per_sm >= 1 && sm_count >= 1 && grid >= 1 && (long long)grid <= (long long)blocks_per_sm * sm_count;
}

// The largest dynamic shared-memory size allowed so far for one kernel.
class SmemLimitMemo {
 public:
  // Makes `bytes` allowed on (dev, ctx): calls set(bytes) unless a size at
  // least as large was set under the same device and context. ctx == 0 (no
  // context known) is never memoised. Returns set's result, or 0.
  template <typename Set>
  int ensure(int dev, unsigned long long ctx, int bytes, Set set) {
    if (bytes <= 0) return 0;
    if (dev < 0 || dev >= kMaxDevices || ctx == 0) return set(bytes);
    std::lock_guard<std::mutex> lock(mu_);
    Slot& s = slot_[dev];
    if (s.ctx == ctx && bytes <= s.bytes) return 0;
    const int e = set(bytes);
    if (e == 0) {
      if (s.ctx != ctx) s.bytes = 0;
      s.ctx = ctx;
      if (bytes > s.bytes) s.bytes = bytes;
    }
    return e;
  }

 private:
  struct Slot {
    unsigned long long ctx = 0;
    int bytes = 0;
  };
  std::mutex mu_;
  Slot slot_[kMaxDevices];
};

// One pointer per (device, context), looked up once by find(&ptr).
class PointerMemo {
 public:
  template <typename Find>
  int get(int dev, unsigned long long ctx, void** out, Find find) {
    if (dev < 0 || dev >= kMaxDevices || ctx == 0) return find(out);
    std::lock_guard<std::mutex> lock(mu_);
    Slot& s = slot_[dev];
    if (s.ctx == ctx && s.ptr != nullptr) {
      *out = s.ptr;
      return 0;
    }
    void* p = nullptr;
    const int e = find(&p);
    if (e != 0) return e;
    s.ctx = ctx;
    s.ptr = p;
    *out = p;
    return 0;
  }

 private:
  struct Slot {
    unsigned long long ctx = 0;
    void* ptr = nullptr;
  };
  std::mutex mu_;
  Slot slot_[kMaxDevices];
};

}  // namespace bgmoe
