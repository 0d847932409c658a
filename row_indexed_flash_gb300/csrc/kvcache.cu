// KV-pool kernels: page-table expansion, INT8 / INT4 / FP8 quantise / dequantise, 16-bit
// row appends and the row-list range check.
//
// Paged KV with 64-token pages and INT8 storage: v100llm article, sections
// 1-2.  Negative row = padding: "llama.cpp 0.9.0 inference boundaries",
// section 1.
#include <cuda_fp8.h>
#include <atomic>
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

// x / s rounded to nearest (even) in fp32, for x a bf16 or fp16 value widened
// to fp32, s a positive finite fp16 scale (or one of the codec tops) and r an
// approximation of 1/s within a relative 2^-20: one multiply and two fused
// multiply-adds in place of a division, after the quotient correction of
// P. Markstein ("IA-64 and Elementary Functions", 2000).  q0 = RN(x*r) lies
// within 5 ulp of x/s, so the residual x - q0*s is exact in one fma, and the
// exact q0 + (x - q0*s)*r equals x/s + (x/s - q0)*(s*r - 1): within
// 5 * 2^-20 ulp of x/s.  Rounding it gives RN(x/s) unless a midpoint of the
// fp32 grid lies that close.  It cannot: writing x = mx*2^a, s = ms*2^b with
// mx, ms < 2^11 integers and x/s in [2^e, 2^(e+1)), a - b >= e - 24, so
// |x/s - M| for a midpoint M = odd * 2^(e-24) is a multiple of 2^(e-24)
// divided by ms: zero or at least 2^-12 ulp; and zero would make x/s a dyadic
// number of at most 11 bits equal to a 25-bit one.  The caller handles an
// infinite x (the residual is NaN; x/s is that infinity).  A zero x gives +0
// (the sum drops the sign of -0).  A quotient small enough for the residual to
// underflow is below 2^-76 and codes as a zero either way.
__device__ __forceinline__ float div_by_scale(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  return __fmaf_rn(__fmaf_rn(-q0, s, x), r, q0);
}

__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));   // within 1 ulp; s is a normal fp32 here
  return r;
}

// The per-row codecs for D = 64, 128, 256 with 16-byte aligned x and q, one
// kernel for all three.  A (row, head) item spans D / 16 lanes, each coding
// 16 elements: the 8 at 8 * part and the 8 at D/2 + 8 * part, so that every
// load and every code store is contiguous across the item's lanes.  Each warp
// streams its own tiles (32 / (D / 16) consecutive items, 1 KB) through
// shared memory with cp.async, kQuantStages tiles ahead, and each lane copies
// exactly the pieces and the destination index that it later reads: no
// barrier, no register held by a load in flight, and a small ubatch is
// requested whole at the start.  Same results as the one-warp-per-item
// kernels, with cheaper steps:
// * amax and the NaN test from the 16-bit patterns: with the sign bit
//   cleared, bf16 and fp16 values order as their magnitudes do, +Inf above
//   every finite value, and the NaN-propagating packed max gives the canonical
//   NaN (above +Inf) when any element is NaN;
// * the divisions by div_by_scale (the scale's with RN(1/top), the codes'
//   with an approximate reciprocal of s);
// * the integer codes by adding 1.5 * 2^23 to the quotient: in [2^23, 2^24)
//   the fp32 grid step is 1, so the sum's rounding is the round half to even
//   of the quotient and its low byte is the two's-complement code.  The clamp
//   to +-top is needed only for a subnormal or saturated scale: otherwise
//   s >= (amax / top)(1 - 2^-11)(1 - 2^-24), so |x / s| < top + 1/2;
// * item -> (row, head) by stepping both, since a warp's tiles are a fixed
//   stride apart.
enum { kCodecInt8 = 0, kCodecInt4 = 1, kCodecFp8 = 2 };

// Lane-wise max of two bf16x2 (or f16x2) words of non-negative values, any NaN
// giving the canonical NaN (0x7fff, above +Inf in either format).
template <bool BF16>
__device__ __forceinline__ uint32_t hmax2_nan_bits(uint32_t a, uint32_t b) {
  if constexpr (BF16) {
    const __nv_bfloat162 r = __hmax2_nan(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                         *reinterpret_cast<const __nv_bfloat162*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
  } else {
    const __half2 r = __hmax2_nan(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
  }
}

// Codes of 16 quotients (8 of the first half row, 8 of the second) packed for
// the two stores: integer codes from the low bits of q + 1.5 * 2^23 (q already
// within +-top), E4M3 codes by the saturating conversion with the zero's sign
// taken from the element.
template <int CODEC>
__device__ __forceinline__ void encode_codes(const float (&qv)[16], const float (&vals)[16], uint32_t (&packed)[4]) {
  constexpr float ROUNDER = 12582912.0f;   // 1.5 * 2^23
  if constexpr (CODEC == kCodecFp8) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = __nv_cvt_float2_to_fp8x2(
          make_float2(copysignf(qv[4 * j], vals[4 * j]), copysignf(qv[4 * j + 1], vals[4 * j + 1])), __NV_SATFINITE,
          __NV_E4M3);
      const uint32_t hi = __nv_cvt_float2_to_fp8x2(
          make_float2(copysignf(qv[4 * j + 2], vals[4 * j + 2]), copysignf(qv[4 * j + 3], vals[4 * j + 3])),
          __NV_SATFINITE, __NV_E4M3);
      packed[j] = __byte_perm(lo, hi, 0x5410);
    }
  } else {
    uint32_t c[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) c[e] = __float_as_uint(qv[e] + ROUNDER);
    if constexpr (CODEC == kCodecInt4) {
      uint32_t b[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) b[j] = (c[2 * j] & 0xfu) | ((c[2 * j + 1] << 4) & 0xf0u);
      packed[0] = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
      packed[1] = __byte_perm(__byte_perm(b[4], b[5], 0x0040), __byte_perm(b[6], b[7], 0x0040), 0x5410);
      packed[2] = packed[3] = 0u;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        packed[j] = __byte_perm(__byte_perm(c[4 * j], c[4 * j + 1], 0x0040),
                                __byte_perm(c[4 * j + 2], c[4 * j + 3], 0x0040), 0x5410);
    }
  }
}
constexpr int kQuantStages = 4;   // tiles in flight per warp

template <int CODEC, int D, bool BF16>
__global__ void __launch_bounds__(256, 4) quantize_rows_staged_kernel(const uint4* __restrict__ x, int n_items,
                                                                      int Hkv, int rows_step, int heads_step,
                                                                      const int32_t* __restrict__ dst_rows,
                                                                      uint8_t* __restrict__ q,
                                                                      uint16_t* __restrict__ scale, int R) {
  constexpr int LPI = D / 16;                      // lanes per item
  constexpr int IPW = 32 / LPI;                    // items per tile
  constexpr int IC = 2 * D / 16;                   // 16-byte pieces per item
  constexpr int S = kQuantStages;
  constexpr int QROW = CODEC == kCodecInt4 ? D / 2 : D;
  constexpr float TOP = CODEC == kCodecInt8 ? 127.0f : CODEC == kCodecInt4 ? 7.0f : 448.0f;
  constexpr float RTOP = 1.0f / TOP;              // RN(1/top), folded by the compiler
  constexpr uint32_t INF_BITS = BF16 ? 0x7f80u : 0x7c00u;
  extern __shared__ uint4 smem[];                 // per warp: S tiles of 64 pieces, then S x 32 indices
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane / LPI, part = lane % LPI;
  uint4* wtiles = smem + (size_t)warp * S * 64;
  int32_t* widx = reinterpret_cast<int32_t*>(smem + (size_t)(blockDim.x / 32) * S * 64) + warp * S * 32;
  const int gw = blockIdx.x * (blockDim.x / 32) + warp;
  const int item_step = gridDim.x * (blockDim.x / 32) * IPW;   // = rows_step * Hkv + heads_step

  // the lane's item in the tile being issued and in the tile being coded, with
  // its row and head, stepped by item_step each tile
  int it_i = gw * IPW + sub, row_i = (int)((unsigned)it_i / (unsigned)Hkv), head_i = it_i - row_i * Hkv;
  int it_c = it_i, row_c = row_i, head_c = head_i;
  auto advance = [&](int& it, int& row, int& head) {
    it += item_step;
    row += rows_step;
    head += heads_step;
    if (head >= Hkv) {
      head -= Hkv;
      ++row;
    }
  };
  auto issue = [&](int slot) {
    const bool ok = it_i < n_items;
    const uint4* src = ok ? x + (size_t)it_i * IC + part : x;
    cp_async16(wtiles + slot * 64 + lane, src, ok);
    cp_async16(wtiles + slot * 64 + 32 + lane, ok ? src + LPI : x, ok);
    if (dst_rows) cp_async4(widx + slot * 32 + lane, ok ? dst_rows + row_i : dst_rows, ok);
    cp_async_commit();   // one group per tile, empty or not, so the wait count below holds
    advance(it_i, row_i, head_i);
  };
#pragma unroll
  for (int st = 0; st < S; ++st) issue(st);

  for (int k = 0; it_c - sub < n_items; ++k) {   // warp-uniform: the tile's first item
    const int slot = k % S;
    cp_async_wait<S - 1>();                        // this lane's pieces of tile k have landed
    const uint4 h0 = wtiles[slot * 64 + lane];
    const uint4 h1 = wtiles[slot * 64 + 32 + lane];
    const int d = it_c < n_items ? (dst_rows ? widx[slot * 32 + lane] : row_c) : -1;
    const uint32_t w[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    uint32_t m2 = w[0] & 0x7fff7fffu;
#pragma unroll
    for (int j = 1; j < 8; ++j) m2 = hmax2_nan_bits<BF16>(m2, w[j] & 0x7fff7fffu);
    uint32_t mag = max(m2 & 0xffffu, m2 >> 16);
#pragma unroll
    for (int o = LPI / 2; o >= 1; o >>= 1) mag = max(mag, __shfl_xor_sync(0xffffffffu, mag, o));
    const bool live = (unsigned)d < (unsigned)R;   // not padding, out of range or past the end
    const bool has_nan = mag > INF_BITS;
    const bool row_inf = mag == INF_BITS;
    const float amax = BF16 ? __uint_as_float(mag << 16) : __half2float(__ushort_as_half((unsigned short)mag));
    unsigned short sb;
    if (has_nan) {
      sb = 0x7E00u;
    } else {
      const float sq = row_inf ? amax : div_by_scale(amax, TOP, RTOP);
      sb = __half_as_ushort(__float2half_rn(fminf(sq, 65504.0f)));
    }
    const float sf = __half2float(__ushort_as_half(sb));
    // no NaN, no Inf, and a scale that needs no clamp (integer codecs) or is not zero
    const bool plain =
        !has_nan && !row_inf && (CODEC == kCodecFp8 ? sb != 0u : (sb >= 0x0400u && sb < 0x7bffu));
    float vals[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if constexpr (BF16) {
        vals[2 * j] = __uint_as_float(w[j] << 16);
        vals[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
      } else {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
        vals[2 * j] = f.x;
        vals[2 * j + 1] = f.y;
      }
    }
    const float rs = rcp_approx(sf);
    float qv[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) qv[e] = div_by_scale(vals[e], sf, rs);
    uint32_t packed[4];   // codes of the first half row, then of the second
    if (__all_sync(0xffffffffu, plain || !live)) {
      encode_codes<CODEC>(qv, vals, packed);
    } else {   // some item of the warp holds a NaN or an Inf or has a subnormal, saturated or zero scale
      if (row_inf) {
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (isinf(vals[e])) qv[e] = vals[e];
      }
      if constexpr (CODEC != kCodecFp8) {
#pragma unroll
        for (int e = 0; e < 16; ++e) qv[e] = fminf(fmaxf(qv[e], -TOP), TOP);
      }
      encode_codes<CODEC>(qv, vals, packed);
      const uint32_t fill = has_nan && CODEC == kCodecFp8 ? 0x7f7f7f7fu : 0u;
      if (has_nan || sf == 0.f) packed[0] = packed[1] = packed[2] = packed[3] = fill;
    }
    if (live) {
      uint8_t* qrow = q + ((size_t)d * Hkv + head_c) * QROW;
      if constexpr (CODEC == kCodecInt4) {
        *reinterpret_cast<uint32_t*>(qrow + part * 4) = packed[0];
        *reinterpret_cast<uint32_t*>(qrow + QROW / 2 + part * 4) = packed[1];
      } else {
        *reinterpret_cast<uint2*>(qrow + part * 8) = make_uint2(packed[0], packed[1]);
        *reinterpret_cast<uint2*>(qrow + QROW / 2 + part * 8) = make_uint2(packed[2], packed[3]);
      }
      if (part == 0) scale[((size_t)((unsigned)d / kPage) * Hkv + head_c) * kPage + ((unsigned)d % kPage)] = sb;
    }
    issue(slot);   // h0, h1 and d are consumed above, so the slot is free again
    advance(it_c, row_c, head_c);
  }
  cp_async_wait<0>();
}

// Launches the staged kernel when D is 64, 128 or 256, x and q are 16-byte
// aligned and the item count and pool rows fit an int; returns false (nothing
// launched) otherwise.  Four blocks of 8 warps per SM (147 KB of stages, 64
// registers: measured 7.8 us per 25 MB launch against 8.2 us for three blocks
// with eight tiles each and 8.7 us for two with twelve; five or six blocks
// spill), at most one warp per tile.
template <int CODEC, int D, bool BF16>
void launch_quantize_staged(const uint4* x, int items, int Hkv, const int32_t* dst, uint8_t* q, uint16_t* scale,
                            int R, cudaStream_t st) {
  constexpr int smem = 8 * kQuantStages * (64 * 16 + 32 * 4);
  static std::atomic<bool> attr_set{false};
  if (!attr_set.load(std::memory_order_relaxed)) {
    cudaFuncSetAttribute(quantize_rows_staged_kernel<CODEC, D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         smem);
    attr_set.store(true, std::memory_order_relaxed);
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 1;
  constexpr int IPW = 32 / (D / 16);
  const int tiles = (items + IPW - 1) / IPW;
  int blocks = (tiles + 7) / 8;
  if (blocks > 4 * sms) blocks = 4 * sms;
  const int item_step = blocks * 8 * IPW;
  quantize_rows_staged_kernel<CODEC, D, BF16><<<blocks, 256, smem, st>>>(x, items, Hkv, item_step / Hkv,
                                                                         item_step % Hkv, dst, q, scale, R);
}

template <int CODEC, bool BF16>
bool launch_quantize_staged_d(const uint4* x, int items, int Hkv, int D, const int32_t* dst, uint8_t* q,
                              uint16_t* scale, int R, cudaStream_t st) {
  if (D == 64)
    launch_quantize_staged<CODEC, 64, BF16>(x, items, Hkv, dst, q, scale, R, st);
  else if (D == 128)
    launch_quantize_staged<CODEC, 128, BF16>(x, items, Hkv, dst, q, scale, R, st);
  else if (D == 256)
    launch_quantize_staged<CODEC, 256, BF16>(x, items, Hkv, dst, q, scale, R, st);
  else
    return false;
  return true;
}

template <int CODEC>
bool launch_quantize_v8(const void* x, int x_bf16, long long n_rows, int Hkv, int D, const int32_t* dst, void* q,
                        uint16_t* scale, long long R, cudaStream_t st) {
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0 || reinterpret_cast<uintptr_t>(q) % 16 != 0) return false;
  const long long items = n_rows * Hkv;
  if (items >= (1LL << 30) || R >= (1LL << 31)) return false;
  const uint4* xv = static_cast<const uint4*>(x);
  uint8_t* qb = static_cast<uint8_t*>(q);
  return x_bf16 ? launch_quantize_staged_d<CODEC, true>(xv, (int)items, Hkv, D, dst, qb, scale, (int)R, st)
                : launch_quantize_staged_d<CODEC, false>(xv, (int)items, Hkv, D, dst, qb, scale, (int)R, st);
}

cudaError_t launch_quantize_int8(const void* x, int x_bf16, long long n_rows, int Hkv, int D, const int32_t* dst,
                                 int8_t* q, uint16_t* scale, long long R, cudaStream_t st) {
  const long long warps = n_rows * Hkv;
  if (warps == 0) return cudaSuccess;
  if (launch_quantize_v8<kCodecInt8>(x, x_bf16, n_rows, Hkv, D, dst, q, scale, R, st)) return cudaGetLastError();
  const int threads = 256;
  long long blocks = (warps + 7) / 8;
  if (blocks > 152 * 64) blocks = 152 * 64;
  quantize_int8_kernel<<<(unsigned)blocks, threads, 0, st>>>(static_cast<const uint16_t*>(x), x_bf16, n_rows, Hkv, D,
                                                             dst, q, scale, R);
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
  if (launch_quantize_v8<kCodecInt4>(x, x_bf16, n_rows, Hkv, D, dst, q, scale, R, st)) return cudaGetLastError();
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
  if (launch_quantize_v8<kCodecFp8>(x, x_bf16, n_rows, Hkv, D, dst, q, scale, R, st)) return cudaGetLastError();
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
