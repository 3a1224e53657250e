// fa_fwd_decode_noalloc: the split-KV decode call for callers that cannot
// allocate device memory at call time. Such callers include code running
// under a memory manager that owns the whole device heap (for example a
// serving process whose memory plan is fixed when it starts), and code that
// must not allocate on its hot path because an allocation can block on the
// device or fail once memory is fragmented. The split workspace of
// fa_fwd_decode lives here in a fixed-size array in the library's own
// device memory instead of in a caller-provided buffer.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fa.h"

namespace {

// Scratch for the per-split partial states (fp32 O and LSE). Every device
// that loads this library holds these bytes until the process exits.
constexpr unsigned long long kScratchBytes = 16ull << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device. In host code the
// array's name only stands for the symbol; the address a kernel may use has
// to come from the runtime, once per device, with that device current.
// The library is built without relocatable device code, so the array sits in
// a module of its own; CUDA loads modules lazily by default, and the first
// lookup on a device is what loads it (and reserves the array's bytes). Only
// a successful lookup is kept: a failed one (for example out of memory while
// the module loads) is tried again on the next call.
void* scratch_address(int dev) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) == cudaSuccess) g_scratch_addr[dev] = ptr;
    else (void)cudaGetLastError();   // reset the runtime's last-error state for later calls
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int fa_fwd_decode_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq,
                                     int Sk, int Hq, int Hkv, int D, float scale, int causal, int dtype,
                                     int num_splits, fa_stream_t stream) {
  // Same sizes and checks as fa_fwd_decode; the workspace the call needs must
  // fit the fixed scratch array.
  unsigned long long need = 0;
  int rc = fa_decode_workspace_size(B, Sq, Sk, Hq, Hkv, D, num_splits, &need);
  if (rc != FA_OK) return rc;
  if (need > kScratchBytes) return FA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (need > 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    scratch = scratch_address(dev);
    if (!scratch) return FA_ERR_CUDA;
  }
  // Every split writes all of its partial rows before the merge reads them,
  // so nothing in the scratch has to start at zero.
  return fa_fwd_decode(q, k, v, o, lse, B, Sq, Sk, Hq, Hkv, D, scale, causal, dtype, num_splits, scratch,
                       need > 0 ? kScratchBytes : 0, stream);
}
