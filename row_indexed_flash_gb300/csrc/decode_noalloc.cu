// fa_rows_decode_static: the decode entry point for callers that cannot
// allocate device memory.
//
// Some hosts of this library may not call cudaMalloc (or any allocating
// routine) at the point where they run attention: code that runs inside a
// custom device-memory allocator or its callbacks, plugins whose host
// framework owns every device allocation and forbids others, and real-time
// paths where an allocation's latency or possible failure is not acceptable.
// They cannot provide the split-merge scratch that fa_rows_decode needs, so
// this variant takes its scratch from one statically sized device array that
// lives in this library.
//
// The array holds kStaticScratchBytes on every GPU that loads the library,
// until the process exits.  All calls share it and it keeps the previous
// call's contents, so each call first zero-fills the part it uses; calls whose
// work overlaps on the GPU (different streams, or different host threads)
// race on it and must be serialised by the caller.
#include <stdio.h>

#include <atomic>

#include "fa_internal.cuh"

namespace far {
void set_last_error(const char* msg);  // the message fa_last_error() returns
}

namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// Device address of the scratch array for the current device, looked up once
// per device.  In host code the array's name is only a host-side stand-in, so
// the address must come from the runtime.  The cache is atomic: two host
// threads making their first call at once both look the address up and store
// the same value.
void* scratch_address(int* err) {
  static std::atomic<void*> addr[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    *err = e == cudaSuccess ? (int)cudaErrorInvalidDevice : (int)e;
    return nullptr;
  }
  void* cached = addr[dev].load(std::memory_order_relaxed);
  if (cached) return cached;
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (e != cudaSuccess || !p) {
    *err = e == cudaSuccess ? (int)cudaErrorInvalidSymbol : (int)e;
    return nullptr;
  }
  addr[dev].store(p, std::memory_order_relaxed);
  return p;
}

}  // namespace

extern "C" {

fa_status fa_rows_decode_static(const fa_rows_args* a, fa_stream_t stream) {
  if (!a) return fa_rows_decode(a, nullptr, 0, stream);  // reports the NULL argument
  const size_t need = fa_rows_workspace_size(a, 0);
  if (need == 0 && fa_last_error()[0] != 0) return fa_rows_decode(a, nullptr, 0, stream);  // invalid arguments
  if (need > kStaticScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "fa_rows_decode_static: these arguments need %zu bytes of scratch; the static array holds %zu", need,
             kStaticScratchBytes);
    far::set_last_error(msg);
    return FA_ERR_WORKSPACE;
  }
  int err = 0;
  void* ws = scratch_address(&err);
  if (!ws) {
    char msg[256];
    snprintf(msg, sizeof(msg), "fa_rows_decode_static: scratch address lookup failed: %s",
             cudaGetErrorString((cudaError_t)err));
    far::set_last_error(msg);
    return FA_ERR_CUDA;
  }
  if (need > 0) {   // the status word, the split counters and the partials start from zero
    const fa_status st = fa_rows_workspace_init(ws, need, stream);
    if (st != FA_OK) return st;
  }
  return fa_rows_decode(a, ws, kStaticScratchBytes, stream);
}

}  // extern "C"
