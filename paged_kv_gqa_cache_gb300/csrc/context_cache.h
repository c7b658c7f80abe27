// Per-device cache of a value that belongs to one CUDA context.
//
// The device address of a __device__ variable (the error word, the fixed
// scratch array of the allocation-free decode) and a kernel's raised
// shared-memory limit exist once per context: a host application that makes
// its own driver-API context current, or a cudaDeviceReset() that recreates
// the primary context, leaves the module loaded anew at other addresses.  An
// entry is therefore tagged with the unique id of the context it was taken in
// (cuCtxGetId: ids are never reused within a process, unlike context
// handles), and a lookup under another id takes the value again.
//
// Host code only, no CUDA types: the cache logic is tested on the CPU.
#pragma once

#include <mutex>

namespace pa {

template <typename V, int kMaxDevices = 64>
class ContextCache {
 public:
  // The value for (device, ctx_id): the cached one if it was taken in the
  // context ctx_id, else fetch(&value) is called (under the cache's lock) and
  // its result cached when it returns true.  Returns false for a device
  // outside [0, kMaxDevices), a context id of 0 (no context), or a failed fetch.
  template <typename Fetch>
  bool get(int device, unsigned long long ctx_id, Fetch fetch, V *out) {
    if (device < 0 || device >= kMaxDevices || ctx_id == 0) return false;
    std::lock_guard<std::mutex> lock(mutex_);
    Entry &e = entries_[device];
    if (e.ctx_id != ctx_id) {
      V v{};
      if (!fetch(&v)) return false;
      e.value = v;
      e.ctx_id = ctx_id;
    }
    *out = e.value;
    return true;
  }

 private:
  struct Entry {
    unsigned long long ctx_id = 0;  // 0: nothing cached
    V value{};
  };
  std::mutex mutex_;
  Entry entries_[kMaxDevices];
};

}  // namespace pa
