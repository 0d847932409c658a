// KV-pool kernels: page-table expansion, INT8 / INT4 / FP8 quantise / dequantise, 16-bit
// row appends and the row-list range check.
//
// Paged KV with 64-token pages and INT8 storage: v100llm article, sections
// 1-2.  Negative row = padding: "llama.cpp 0.9.0 inference boundaries",
// section 1.
#include <cuda_fp8.h>
#include <limits.h>

#include "fa_internal.cuh"

namespace far {

// Scale of one (row, head) for a codec whose largest code is `top`:
// fp16_rne(min(amax/top, 65504)) with one fp32 division (amax = +Inf gives
// 65504).  A row holding a NaN keeps it: the fp16 quiet NaN 0x7E00, and the
// caller writes NaN codes (0 for the integer codecs, 0x7f for E4M3).
__device__ __forceinline__ unsigned short row_scale_bits(float amax, bool has_nan, float top) {
  if (has_nan) return 0x7E00u;
  return __half_as_ushort(__float2half_rn(fminf(__fdiv_rn(amax, top), 65504.0f)));
}

// kv_rows[s, j] = page_table[s, j/page]*page + j%page for j < seq_len[s], else -1.
// One thread writes four consecutive positions.
__global__ void page_table_to_rows_kernel(const int32_t* __restrict__ pt, int max_pages,
                                          const int32_t* __restrict__ seq_len, int n_seq, int page,
                                          int32_t* __restrict__ rows, int list_len) {
  const long long quads = (long long)n_seq * ((list_len + 3) / 4);
  const int qpr = (list_len + 3) / 4;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < quads;
       t += (long long)gridDim.x * blockDim.x) {
    const int s = (int)(t / qpr);
    const int j0 = (int)(t % qpr) * 4;
    int len = seq_len[s];
    len = min(max(len, 0), max_pages * page);
    int out[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u;
      int r = -1;
      if (j < len) {
        const int pid = __ldg(pt + (size_t)s * max_pages + j / page);
        r = pid >= 0 ? pid * page + j % page : -1;
      }
      out[u] = r;
    }
    int32_t* dst = rows + (size_t)s * list_len + j0;
    if ((list_len & 3) == 0) {
      *reinterpret_cast<int4*>(dst) = make_int4(out[0], out[1], out[2], out[3]);
    } else {
      for (int u = 0; u < 4 && j0 + u < list_len; ++u) dst[u] = out[u];
    }
  }
}

cudaError_t launch_page_table_to_rows(const int32_t* pt, int max_pages, const int32_t* seq_len, int n_seq, int page,
                                      int32_t* rows, int list_len, cudaStream_t st) {
  const long long quads = (long long)n_seq * ((list_len + 3) / 4);
  if (quads == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (quads + threads - 1) / threads;
  page_table_to_rows_kernel<<<(unsigned)(blocks < 65535 * 16 ? blocks : 65535 * 16), threads, 0, st>>>(
      pt, max_pages, seq_len, n_seq, page, rows, list_len);
  return cudaGetLastError();
}

// One warp per (source row, head): amax over D, fp16 scale, int8 codes (a row
// holding a NaN: scale 0x7E00, codes 0).
__global__ void quantize_int8_kernel(const uint16_t* __restrict__ x, int x_bf16, long long n_rows, int Hkv, int D,
                                     const int32_t* __restrict__ dst_rows, int8_t* __restrict__ q,
                                     uint16_t* __restrict__ scale, long long R) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x / 32);
  for (long long w = blockIdx.x * (long long)(blockDim.x / 32) + (threadIdx.x >> 5); w < n_rows * Hkv; w += warps) {
    const long long i = w / Hkv;
    const int g = (int)(w % Hkv);
    const long long dst = dst_rows ? (long long)dst_rows[i] : i;
    if (dst < 0 || dst >= R) continue;
    const uint16_t* src = x + (size_t)w * D;
    float vals[8];   // D <= 256
    float amax = 0.f;
    bool nan = false;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int d = lane + 32 * u;
      float f = 0.f;
      if (d < D) {
        const uint32_t b = src[d];
        f = x_bf16 ? __uint_as_float(b << 16) : __half2float(__ushort_as_half((unsigned short)b));
      }
      vals[u] = f;
      amax = fmaxf(amax, fabsf(f));   // fmaxf skips NaN: tracked separately
      nan |= f != f;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const bool has_nan = __any_sync(0xffffffffu, nan);
    const unsigned short sb = row_scale_bits(amax, has_nan, 127.0f);
    const float sf = __half2float(__ushort_as_half(sb));
    int8_t* qd = q + ((size_t)dst * Hkv + g) * D;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int d = lane + 32 * u;
      if (d < D) {
        int c = 0;
        if (sf != 0.f && !has_nan) c = min(max(__float2int_rn(__fdiv_rn(vals[u], sf)), -127), 127);
        qd[d] = (int8_t)c;
      }
    }
    if (lane == 0) scale[((size_t)(dst / kPage) * Hkv + g) * kPage + (dst % kPage)] = sb;
  }
}

// The same rule for D = 32 * EPL (64, 128, 256) with 16-byte aligned x and q:
// lane l holds elements EPL*l .. EPL*l + EPL - 1, loaded and stored with one
// vector access each, and the row's values are loaded together with its
// destination index rather than after it.
template <int EPL>
__global__ void quantize_int8_vec_kernel(const uint16_t* __restrict__ x, int x_bf16, long long n_rows, int Hkv,
                                         const int32_t* __restrict__ dst_rows, int8_t* __restrict__ q,
                                         uint16_t* __restrict__ scale, long long R) {
  constexpr int D = 32 * EPL;
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x / 32);
  for (long long w = blockIdx.x * (long long)(blockDim.x / 32) + (threadIdx.x >> 5); w < n_rows * Hkv; w += warps) {
    const long long i = w / Hkv;
    const int g = (int)(w % Hkv);
    const uint16_t* src = x + (size_t)w * D + lane * EPL;
    uint32_t raw[EPL / 2];
    if constexpr (EPL == 2) {
      raw[0] = __ldg(reinterpret_cast<const unsigned int*>(src));
    } else if constexpr (EPL == 4) {
      const uint2 t = __ldg(reinterpret_cast<const uint2*>(src));
      raw[0] = t.x;
      raw[1] = t.y;
    } else {
      const uint4 t = __ldg(reinterpret_cast<const uint4*>(src));
      raw[0] = t.x;
      raw[1] = t.y;
      raw[2] = t.z;
      raw[3] = t.w;
    }
    const long long dst = dst_rows ? (long long)__ldg(dst_rows + i) : i;
    float vals[EPL];
    float amax = 0.f;
    bool nan = false;
#pragma unroll
    for (int k = 0; k < EPL / 2; ++k) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t b = e ? (raw[k] >> 16) : (raw[k] & 0xffffu);
        const float f = x_bf16 ? __uint_as_float(b << 16) : __half2float(__ushort_as_half((unsigned short)b));
        vals[2 * k + e] = f;
        amax = fmaxf(amax, fabsf(f));   // fmaxf skips NaN: tracked separately
        nan |= f != f;
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const bool has_nan = __any_sync(0xffffffffu, nan);
    if (dst < 0 || dst >= R) continue;   // the same for every lane of the warp
    const unsigned short sb = row_scale_bits(amax, has_nan, 127.0f);
    const float sf = __half2float(__ushort_as_half(sb));
    uint32_t packed[(EPL + 3) / 4] = {};
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      int c = 0;
      if (sf != 0.f && !has_nan) c = min(max(__float2int_rn(__fdiv_rn(vals[e], sf)), -127), 127);
      packed[e / 4] |= ((uint32_t)c & 0xffu) << (8 * (e % 4));
    }
    int8_t* qd = q + ((size_t)dst * Hkv + g) * D + lane * EPL;
    if constexpr (EPL == 2) {
      *reinterpret_cast<uint16_t*>(qd) = (uint16_t)packed[0];
    } else if constexpr (EPL == 4) {
      *reinterpret_cast<uint32_t*>(qd) = packed[0];
    } else {
      *reinterpret_cast<uint2*>(qd) = make_uint2(packed[0], packed[1]);
    }
    if (lane == 0) scale[((size_t)(dst / kPage) * Hkv + g) * kPage + (dst % kPage)] = sb;
  }
}

cudaError_t launch_quantize_int8(const void* x, int x_bf16, long long n_rows, int Hkv, int D, const int32_t* dst,
                                 int8_t* q, uint16_t* scale, long long R, cudaStream_t st) {
  const long long warps = n_rows * Hkv;
  if (warps == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (warps + 7) / 8;
  if (blocks > 152 * 64) blocks = 152 * 64;
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  const bool aligned16 = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (reinterpret_cast<uintptr_t>(q) % 16 == 0);
  if (aligned16 && D == 64)
    quantize_int8_vec_kernel<2><<<(unsigned)blocks, threads, 0, st>>>(xs, x_bf16, n_rows, Hkv, dst, q, scale, R);
  else if (aligned16 && D == 128)
    quantize_int8_vec_kernel<4><<<(unsigned)blocks, threads, 0, st>>>(xs, x_bf16, n_rows, Hkv, dst, q, scale, R);
  else if (aligned16 && D == 256)
    quantize_int8_vec_kernel<8><<<(unsigned)blocks, threads, 0, st>>>(xs, x_bf16, n_rows, Hkv, dst, q, scale, R);
  else
    quantize_int8_kernel<<<(unsigned)blocks, threads, 0, st>>>(xs, x_bf16, n_rows, Hkv, D, dst, q, scale, R);
  return cudaGetLastError();
}

// One warp per (source row, head), INT4: the INT8 rule with 7 in place of
// 127; two's-complement nibbles, element 2t in the low nibble of byte t.
// Lane l handles the element pairs l, l + 32, ... (D <= 256).
__global__ void quantize_int4_kernel(const uint16_t* __restrict__ x, int x_bf16, long long n_rows, int Hkv, int D,
                                     const int32_t* __restrict__ dst_rows, uint8_t* __restrict__ q,
                                     uint16_t* __restrict__ scale, long long R) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x / 32);
  for (long long w = blockIdx.x * (long long)(blockDim.x / 32) + (threadIdx.x >> 5); w < n_rows * Hkv; w += warps) {
    const long long i = w / Hkv;
    const int g = (int)(w % Hkv);
    const long long dst = dst_rows ? (long long)dst_rows[i] : i;
    if (dst < 0 || dst >= R) continue;
    const uint16_t* src = x + (size_t)w * D;
    float vals[8];
    float amax = 0.f;
    bool nan = false;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int d = 2 * (lane + 32 * u);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float f = 0.f;
        if (d + e < D) {
          const uint32_t b = src[d + e];
          f = x_bf16 ? __uint_as_float(b << 16) : __half2float(__ushort_as_half((unsigned short)b));
        }
        vals[2 * u + e] = f;
        amax = fmaxf(amax, fabsf(f));   // fmaxf skips NaN: tracked separately
        nan |= f != f;
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const bool has_nan = __any_sync(0xffffffffu, nan);
    const unsigned short sb = row_scale_bits(amax, has_nan, 7.0f);
    const float sf = __half2float(__ushort_as_half(sb));
    uint8_t* qd = q + ((size_t)dst * Hkv + g) * (D / 2);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = lane + 32 * u;   // byte t holds elements 2t, 2t+1
      if (2 * t < D) {
        int c0 = 0, c1 = 0;
        if (sf != 0.f && !has_nan) {
          c0 = min(max(__float2int_rn(__fdiv_rn(vals[2 * u], sf)), -7), 7);
          c1 = min(max(__float2int_rn(__fdiv_rn(vals[2 * u + 1], sf)), -7), 7);
        }
        qd[t] = (uint8_t)((c0 & 0xF) | ((c1 & 0xF) << 4));
      }
    }
    if (lane == 0) scale[((size_t)(dst / kPage) * Hkv + g) * kPage + (dst % kPage)] = sb;
  }
}

cudaError_t launch_quantize_int4(const void* x, int x_bf16, long long n_rows, int Hkv, int D, const int32_t* dst,
                                 uint8_t* q, uint16_t* scale, long long R, cudaStream_t st) {
  const long long warps = n_rows * Hkv;
  if (warps == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (warps + 7) / 8;
  if (blocks > 152 * 64) blocks = 152 * 64;
  quantize_int4_kernel<<<(unsigned)blocks, threads, 0, st>>>(static_cast<const uint16_t*>(x), x_bf16, n_rows, Hkv, D,
                                                             dst, q, scale, R);
  return cudaGetLastError();
}

// out = float(nibble code) * float(scale), exact in fp32.
__global__ void dequantize_int4_kernel(const uint8_t* __restrict__ q, const uint16_t* __restrict__ scale,
                                       long long n_rows, int Hkv, int D, float* __restrict__ out) {
  const long long n = n_rows * Hkv * D;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n; t += (long long)gridDim.x * blockDim.x) {
    const long long rh = t / D;
    const long long r = rh / Hkv;
    const int g = (int)(rh % Hkv);
    const int d = (int)(t % D);
    const int byte = q[rh * (D / 2) + d / 2];
    int c = (d & 1) ? (byte >> 4) : (byte & 0xF);
    c = c >= 8 ? c - 16 : c;
    const float sf = __half2float(__ushort_as_half(scale[((size_t)(r / kPage) * Hkv + g) * kPage + (r % kPage)]));
    out[t] = __fmul_rn((float)c, sf);
  }
}

cudaError_t launch_dequantize_int4(const uint8_t* q, const uint16_t* scale, long long n_rows, int Hkv, int D,
                                   float* out, cudaStream_t st) {
  const long long n = n_rows * Hkv * D;
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (n + threads - 1) / threads;
  if (blocks > 152 * 64) blocks = 152 * 64;
  dequantize_int4_kernel<<<(unsigned)blocks, threads, 0, st>>>(q, scale, n_rows, Hkv, D, out);
  return cudaGetLastError();
}

// One warp per (source row, head), FP8 E4M3: s = fp16(min(amax/448, 65504)),
// code = the saturating round-to-nearest-even E4M3 of x/s (one fp32 division);
// s = 0 gives code 0; a row holding a NaN gets scale 0x7E00 and code 0x7f.
__global__ void quantize_fp8_kernel(const uint16_t* __restrict__ x, int x_bf16, long long n_rows, int Hkv, int D,
                                    const int32_t* __restrict__ dst_rows, uint8_t* __restrict__ q,
                                    uint16_t* __restrict__ scale, long long R) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x / 32);
  for (long long w = blockIdx.x * (long long)(blockDim.x / 32) + (threadIdx.x >> 5); w < n_rows * Hkv; w += warps) {
    const long long i = w / Hkv;
    const int g = (int)(w % Hkv);
    const long long dst = dst_rows ? (long long)dst_rows[i] : i;
    if (dst < 0 || dst >= R) continue;
    const uint16_t* src = x + (size_t)w * D;
    float vals[8];
    float amax = 0.f;
    bool nan = false;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int d = lane + 32 * u;
      float f = 0.f;
      if (d < D) {
        const uint32_t b = src[d];
        f = x_bf16 ? __uint_as_float(b << 16) : __half2float(__ushort_as_half((unsigned short)b));
      }
      vals[u] = f;
      amax = fmaxf(amax, fabsf(f));   // fmaxf skips NaN: tracked separately
      nan |= f != f;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const bool has_nan = __any_sync(0xffffffffu, nan);
    const unsigned short sb = row_scale_bits(amax, has_nan, 448.0f);
    const float sf = __half2float(__ushort_as_half(sb));
    uint8_t* qd = q + ((size_t)dst * Hkv + g) * D;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int d = lane + 32 * u;
      if (d < D)
        qd[d] = has_nan ? (uint8_t)0x7f
                        : sf != 0.f ? (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(vals[u], sf), __NV_SATFINITE, __NV_E4M3)
                                    : (uint8_t)0;
    }
    if (lane == 0) scale[((size_t)(dst / kPage) * Hkv + g) * kPage + (dst % kPage)] = sb;
  }
}

cudaError_t launch_quantize_fp8(const void* x, int x_bf16, long long n_rows, int Hkv, int D, const int32_t* dst,
                                uint8_t* q, uint16_t* scale, long long R, cudaStream_t st) {
  const long long warps = n_rows * Hkv;
  if (warps == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (warps + 7) / 8;
  if (blocks > 152 * 64) blocks = 152 * 64;
  quantize_fp8_kernel<<<(unsigned)blocks, threads, 0, st>>>(static_cast<const uint16_t*>(x), x_bf16, n_rows, Hkv, D,
                                                            dst, q, scale, R);
  return cudaGetLastError();
}

// out = float(E4M3 value) * float(scale), exact in fp32.
__global__ void dequantize_fp8_kernel(const uint8_t* __restrict__ q, const uint16_t* __restrict__ scale,
                                      long long n_rows, int Hkv, int D, float* __restrict__ out) {
  const long long n = n_rows * Hkv * D;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n; t += (long long)gridDim.x * blockDim.x) {
    const long long rh = t / D;
    const long long r = rh / Hkv;
    const int g = (int)(rh % Hkv);
    const __half_raw hv = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)q[t], __NV_E4M3);
    const float v = __half2float(__half(hv));
    const float sf = __half2float(__ushort_as_half(scale[((size_t)(r / kPage) * Hkv + g) * kPage + (r % kPage)]));
    out[t] = __fmul_rn(v, sf);
  }
}

cudaError_t launch_dequantize_fp8(const uint8_t* q, const uint16_t* scale, long long n_rows, int Hkv, int D,
                                  float* out, cudaStream_t st) {
  const long long n = n_rows * Hkv * D;
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (n + threads - 1) / threads;
  if (blocks > 152 * 64) blocks = 152 * 64;
  dequantize_fp8_kernel<<<(unsigned)blocks, threads, 0, st>>>(q, scale, n_rows, Hkv, D, out);
  return cudaGetLastError();
}

// out = float(code) * float(scale): both factors are exact in fp32 and the
// product of an 8-bit and an 11-bit significand is exact too.
__global__ void dequantize_int8_kernel(const int8_t* __restrict__ q, const uint16_t* __restrict__ scale,
                                       long long n_rows, int Hkv, int D, float* __restrict__ out) {
  const long long n = n_rows * Hkv * D;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n; t += (long long)gridDim.x * blockDim.x) {
    const long long rh = t / D;
    const long long r = rh / Hkv;
    const int g = (int)(rh % Hkv);
    const float s = __half2float(__ushort_as_half(scale[((size_t)(r / kPage) * Hkv + g) * kPage + (r % kPage)]));
    out[t] = __fmul_rn((float)q[t], s);
  }
}

cudaError_t launch_dequantize_int8(const int8_t* q, const uint16_t* scale, long long n_rows, int Hkv, int D,
                                   float* out, cudaStream_t st) {
  const long long n = n_rows * Hkv * D;
  if (n == 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  dequantize_int8_kernel<<<(unsigned)blocks, 256, 0, st>>>(q, scale, n_rows, Hkv, D, out);
  return cudaGetLastError();
}

// pool[dst_rows[i]] = x[i]; one CTA per source row, 16-byte copies.
__global__ void kv_append_kernel(const uint4* __restrict__ x, long long n_rows, int row_vec,
                                 const int32_t* __restrict__ dst_rows, uint4* __restrict__ pool, long long R) {
  for (long long i = blockIdx.x; i < n_rows; i += gridDim.x) {
    const long long dst = dst_rows[i];
    if (dst < 0 || dst >= R) continue;
    for (int c = threadIdx.x; c < row_vec; c += blockDim.x) pool[(size_t)dst * row_vec + c] = x[(size_t)i * row_vec + c];
  }
}

cudaError_t launch_kv_append(const void* x, long long n_rows, int row_bytes, const int32_t* dst, void* pool,
                             long long R, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  const long long blocks = n_rows < 152 * 32 ? n_rows : 152 * 32;
  kv_append_kernel<<<(unsigned)blocks, 128, 0, st>>>(static_cast<const uint4*>(x), n_rows, row_bytes / 16, dst,
                                                     static_cast<uint4*>(pool), R);
  return cudaGetLastError();
}

// status[0] += number of entries >= R (within kv_len); status[1] = min flat index
// of such an entry, kept as unsigned so that the initial all-ones reads as -1.
__global__ void validate_kernel(const int32_t* __restrict__ rows, const int32_t* __restrict__ kv_len, int S, int L,
                                long long R, unsigned long long* status) {
  const long long n = (long long)S * L;
  unsigned long long bad = 0, first = ~0ull;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n; t += (long long)gridDim.x * blockDim.x) {
    const int s = (int)(t / L), j = (int)(t % L);
    const int len = kv_len ? min(max(kv_len[s], 0), L) : L;
    if (j < len && (long long)rows[t] >= R) {
      ++bad;
      if ((unsigned long long)t < first) first = (unsigned long long)t;
    }
  }
  for (int o = 16; o >= 1; o >>= 1) {
    bad += __shfl_xor_sync(0xffffffffu, bad, o);
    const unsigned long long f2 = __shfl_xor_sync(0xffffffffu, first, o);
    first = f2 < first ? f2 : first;
  }
  if ((threadIdx.x & 31) == 0 && bad) {
    atomicAdd(status, bad);
    atomicMin(status + 1, first);
  }
}

cudaError_t launch_validate(const int32_t* rows, const int32_t* kv_len, int S, int L, long long R, long long* status,
                            cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(long long), st);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(status + 1, 0xff, sizeof(long long), st);
  if (e != cudaSuccess) return e;
  const long long n = (long long)S * L;
  if (n == 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  validate_kernel<<<(unsigned)blocks, 256, 0, st>>>(rows, kv_len, S, L, R,
                                                    reinterpret_cast<unsigned long long*>(status));
  return cudaGetLastError();
}

}  // namespace far
