// Packing and exact widening of quantised KV codes to the 16-bit type of Q,
// shared by the tensor-core decode kernels.
#pragma once

#include <cuda_fp8.h>

#include "fa_internal.cuh"

namespace far {

__device__ __forceinline__ uint32_t pack2h(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Integer value u (0 <= u < 256) in byte b of x -> fp32 (2^23 + u), exact.
__device__ __forceinline__ float magic_byte(uint32_t x, uint32_t sel) {
  return __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7650u | sel));
}

// Four INT8 codes (one word) -> four 16-bit values of Q's type, exact.
// bf16: (code + 128) is placed in the low mantissa bits of 2^23 and 2^23 + 128
// subtracted, which leaves the code as an fp32 whose low 16 bits are zero, so
// its upper half is the bf16 value.  f16: (code + 128) is placed in the low
// mantissa bits of 1024 (0x6400) and 1152 subtracted.
__device__ __forceinline__ uint2 widen_i8x4(uint32_t w, bool bf16) {
  const uint32_t x = w ^ 0x80808080u;
  if (bf16) {
    const float2 bias = make_float2(-8388736.0f, -8388736.0f);
    const float2 lo = __fadd2_rn(make_float2(magic_byte(x, 0), magic_byte(x, 1)), bias);
    const float2 hi = __fadd2_rn(make_float2(magic_byte(x, 2), magic_byte(x, 3)), bias);
    return make_uint2(__byte_perm(__float_as_uint(lo.x), __float_as_uint(lo.y), 0x7632u),
                      __byte_perm(__float_as_uint(hi.x), __float_as_uint(hi.y), 0x7632u));
  }
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));   // 1152
  uint32_t a = __byte_perm(x, 0x64646464u, 0x4140u), b = __byte_perm(x, 0x64646464u, 0x4342u);
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  return make_uint2(*reinterpret_cast<uint32_t*>(&ha), *reinterpret_cast<uint32_t*>(&hb));
}

// Four bytes u0..u3 (each < 16 after the bias) -> four 16-bit values u - 8.
__device__ __forceinline__ uint2 widen_u4x4(uint32_t p, bool bf16) {
  if (bf16) {
    const float2 bias = make_float2(-8388616.0f, -8388616.0f);   // 2^23 + 8
    const float2 lo = __fadd2_rn(make_float2(magic_byte(p, 0), magic_byte(p, 1)), bias);
    const float2 hi = __fadd2_rn(make_float2(magic_byte(p, 2), magic_byte(p, 3)), bias);
    return make_uint2(__byte_perm(__float_as_uint(lo.x), __float_as_uint(lo.y), 0x7632u),
                      __byte_perm(__float_as_uint(hi.x), __float_as_uint(hi.y), 0x7632u));
  }
  const __half2 bias = __halves2half2(__ushort_as_half(0x6408u), __ushort_as_half(0x6408u));   // 1032
  uint32_t a = __byte_perm(p, 0x64646464u, 0x4140u), b = __byte_perm(p, 0x64646464u, 0x4342u);
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  return make_uint2(*reinterpret_cast<uint32_t*>(&ha), *reinterpret_cast<uint32_t*>(&hb));
}

// Eight INT4 codes (one word; element 2t in the low nibble of byte t, two's
// complement) -> eight 16-bit values of Q's type, exact.  The bias 8 makes
// every nibble an unsigned u = code + 8; the low and high nibbles are spread
// into bytes in element order and widened as u - 8.
__device__ __forceinline__ uint4 widen_i4x8(uint32_t w, bool bf16) {
  const uint32_t x = w ^ 0x88888888u;
  const uint32_t even = x & 0x0F0F0F0Fu, odd = (x >> 4) & 0x0F0F0F0Fu;   // elements 0,2,4,6 / 1,3,5,7
  const uint2 a = widen_u4x4(__byte_perm(even, odd, 0x5140u), bf16);     // elements 0..3
  const uint2 b = widen_u4x4(__byte_perm(even, odd, 0x7362u), bf16);     // elements 4..7
  return make_uint4(a.x, a.y, b.x, b.y);
}

// Four FP8 E4M3 codes (one word, element t in byte t) -> four f16 values,
// exact (every E4M3 value is an f16 value).
__device__ __forceinline__ uint2 widen_e4m3x4(uint32_t w) {
  const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
  const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  return make_uint2((uint32_t)lo.x | ((uint32_t)lo.y << 16), (uint32_t)hi.x | ((uint32_t)hi.y << 16));
}

}  // namespace far
