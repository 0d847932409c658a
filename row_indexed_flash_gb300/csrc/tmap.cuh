// Host side: encoding of TMA tensor maps through the CUDA driver API entry point, with
// a small cache so that repeated calls on the same tensors (a decode step per
// token) skip the encode.  Shared by the kernels' launch code.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

namespace far {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// A 3-D tiled map (unit element strides, no interleave, 256-byte L2
// promotion, zero fill).  The last encodings are kept keyed by every argument
// and the device; a hit copies the stored map.
inline bool tmap_encode_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, const cuuint64_t (&dims)[3],
                           const cuuint64_t (&strides)[2], const cuuint32_t (&box)[3], CUtensorMapSwizzle sw) {
  struct Key {
    const void* base;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    int dt, sw, dev;
  };
  struct Entry {
    Key key;
    CUtensorMap map;
    bool used;
  };
  constexpr int N = 32;
  static Entry cache[N];
  static int next = 0;
  static std::mutex mu;
  Key key;
  memset(&key, 0, sizeof(key));   // padding bytes take part in the comparison
  key.base = base;
  for (int i = 0; i < 3; ++i) key.dims[i] = dims[i], key.box[i] = box[i];
  for (int i = 0; i < 2; ++i) key.strides[i] = strides[i];
  key.dt = (int)dt;
  key.sw = (int)sw;
  if (cudaGetDevice(&key.dev) != cudaSuccess) key.dev = -1;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < N; ++i)
      if (cache[i].used && memcmp(&cache[i].key, &key, sizeof(Key)) == 0) {
        *m = cache[i].map;
        return true;
      }
  }
  auto enc = tmap_encode_fn();
  if (!enc) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  if (enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(mu);
  cache[next].key = key;
  cache[next].map = *m;
  cache[next].used = true;
  next = (next + 1) % N;
  return true;
}

}  // namespace far
