// moda_bwd_noalloc: the backward for callers that cannot allocate device memory.
//
// moda_bwd needs a caller-provided device workspace (float32 row statistics and
// the float32 dq accumulator).  Some callers have no way to obtain one: code that
// runs inside a framework's custom-allocator hook or an allocator-free runtime,
// code that is not allowed to touch the device heap after start-up (memory
// budgets fixed at initialisation, real-time or safety-critical loops), and
// plain-C callers with no allocator of their own.  This entry point gives them
// the same backward with its scratch taken from a fixed array that lives in this
// library's device image, so it performs no allocation at all.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes: every GPU
// that loads the library holds it for the life of the process.  Host code cannot
// use the array's name as a device address (on the host it names a stand-in), so
// the first call on each device looks the device address up with
// cudaGetSymbolAddress while that device is current and caches it; that first call
// should therefore be made before any stream capture begins.  The cache lives as long
// as the process: after cudaDeviceReset on a device the library's device image is
// loaded again and may sit elsewhere, so a process that resets a device must not call
// this entry point on it afterwards.  All calls share the
// one array and it keeps whatever the previous call left in it; the backward
// overwrites every word it reads, so nothing needs clearing.  Calls that overlap on
// the GPU (different streams, or different host threads) race on the array.
#include <mutex>

#include "moda.h"

namespace {

// 32 MiB: enough for problems with B*H*T*(d+2)*4 bytes of workspace up to this size
// (for example B*H*T = 127,000 rows at d = 64, or 64,000 rows at d = 128).
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_lock;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per device).
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> guard(g_setup_lock);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

size_t moda_bwd_noalloc_max_workspace_bytes(void) { return kNoAllocScratchBytes; }

moda_status moda_bwd_noalloc(const moda_desc* desc, const void* q, const void* k, const void* v, const void* kd,
                             const void* vd, const void* o, const float* lse, const void* dout, void* dq, void* dk,
                             void* dv, void* dkd, void* dvd, void* stream) {
  const size_t need = moda_bwd_workspace_bytes(desc);
  // an invalid description: let moda_bwd report why, before anything is launched
  if (need == 0) return moda_bwd(desc, q, k, v, kd, vd, o, lse, dout, dq, dk, dv, dkd, dvd, nullptr, 0, stream);
  if (need > kNoAllocScratchBytes) return MODA_ERR_WORKSPACE;
  void* scratch = scratch_for_current_device();
  if (scratch == nullptr) return MODA_ERR_CUDA;
  return moda_bwd(desc, q, k, v, kd, vd, o, lse, dout, dq, dk, dv, dkd, dvd, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
