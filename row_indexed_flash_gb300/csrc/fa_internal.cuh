// Internal declarations of the fa_rows CUDA library (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/fa_rows.h"

namespace far {

// KV storage kinds the kernels are built for.
enum KvKind { KV_BF16 = 0, KV_F16 = 1, KV_I8 = 2, KV_I4 = 3, KV_F8 = 4 };

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kPage = 64;  // rows per page of the INT8 scale layout

// ---------------------------------------------------------------------------
// decode

// Upper bound on list positions handled by one decode CTA (its index stage).
constexpr int kDecodeChunkMax = 2048;
constexpr int kDecodeWarps = 4;
// Splits per (slice, KV head): the in-launch merge stages every split's
// (max, sum) for up to 32 rows in shared memory (64 KB at this cap).
constexpr int kDecodeMaxSplits = 256;

// Every decode and prefill workspace starts with a status block of this many
// bytes; its first word is the status word (FA_WS_WAIT_EXPIRED when a
// bounded pipeline wait ran out).  Decode's split counters follow it.
constexpr size_t kStatusBytes = 256;
// A CTA whose pipeline was aborted still arrives on its (slice, KV head)
// split counter, adding this much more than a normal arrival (the low 16 bits
// count arrivals, splits <= 256): the last arrival then knows that a split's
// partial result is invalid, skips the merge and leaves the counter at zero
// as every call must.
constexpr unsigned int kAbortArrival = 1u << 16;

struct DecodeParams {
  const void* q;
  const void* k;
  const void* v;
  const uint16_t* k_scale;
  const uint16_t* v_scale;
  const int32_t* kv_rows;
  const int32_t* kv_len;
  const float* mask;
  void* out;
  float* lse;
  float* part_o;            // [S, Hkv, nsplit, QVP, D]  un-normalised partial outputs
  float* part_ml;           // [S, Hkv, nsplit, QVP, 2]  (max in log2 units, sum)
  unsigned int* counters;   // [S, Hkv] split arrival counters (zero between calls)
  long long R;
  int S, Nq, Hq, Hkv, L, G, QV, chunk, nsplit;
  int q_bf16;               // Q storage: 1 = bf16, 0 = f16
  int out_dtype;            // fa_dtype of out
  int mask_kind;            // fa_mask_kind
  float qscale;             // scale * log2(e), folded into Q
  unsigned long long wait_ns;   // limit of a pipeline wait (tensor-core kernels)
  int merge_kernel;         // 1: the splits are merged by decode_merge_launch after the decode, not in it
};

struct DecodeConfig {
  int qvp;        // padded query vectors per KV head (power of two)
  int rt;         // rows per warp tile = 32 / qvp
  int nstage;     // cp.async ring depth per warp
  int slot_bytes; // bytes of one ring slot
  size_t smem;    // dynamic shared memory of one CTA
};

// Shape of the kernel instance for (D, qvp, kind); false if not built.
bool decode_config(int D, int qvp, int kind, DecodeConfig* cfg);
// Launch one decode (split kernel with in-launch merge); returns a cudaError_t.
cudaError_t decode_launch(const DecodeParams& p, int D, int qvp, int kind, cudaStream_t st);
// CTAs of the instance that fit on one SM (cached).
int decode_occupancy(int D, int qvp, int kind);

// Tensor-core decode (16-bit or INT8 pools, D 128/256, up to 32 query
// vectors per KV head, no dense mask).  Partials are laid out [unit][split][QV][D].
bool decode_tc_supported(int D, int kind, int qv, int mask_kind);
int decode_tc_occupancy(int D, int kind, int qv);
int decode_tc_tile();
cudaError_t decode_tc_launch(const DecodeParams& p, int D, int kind, unsigned int* err, cudaStream_t st);
// The cross-split merge as a kernel of its own (one thread per query-vector
// row and 4 dimensions of every (slice, KV head)), for decodes launched with
// merge_kernel = 1.  D 128 or 256.
cudaError_t decode_merge_launch(const DecodeParams& p, int D, cudaStream_t st);

// Tensor-core decode for quantised pools (INT8 / INT4 / FP8 codes + fp16 scales),
// D 128: one CTA per SM with a deep code ring.  Same workspace as above.
bool decode_tcq_supported(int D, int kind, int qv, int mask_kind);
int decode_tcq_occupancy(int kind, int qv);
int decode_tcq_tile();
cudaError_t decode_tcq_launch(const DecodeParams& p, int kind, unsigned int* err, cudaStream_t st);

// ---------------------------------------------------------------------------
// prefill

struct PrefillParams {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* kv_rows;
  const int32_t* kv_len;
  const float* mask;
  void* out;
  float* lse;
  long long R;
  int S, Nq, Hq, Hkv, L, G;
  int out_dtype;
  int mask_kind;
  int is_bf16;
  float qscale;         // scale * log2(e)
  unsigned int* err;    // the workspace status word: FA_WS_WAIT_EXPIRED is or-ed in when a wait expires
  unsigned long long wait_ns;   // limit of a pipeline wait
};
cudaError_t prefill_launch(const PrefillParams& p, cudaStream_t st);
bool prefill_supported(int D, int kind);

// ---------------------------------------------------------------------------
// KV pool helpers

cudaError_t launch_page_table_to_rows(const int32_t* pt, int max_pages, const int32_t* seq_len, int n_seq,
                                      int page, int32_t* rows, int list_len, cudaStream_t st);
cudaError_t launch_quantize_int8(const void* x, int x_bf16, long long n_rows, int Hkv, int D, const int32_t* dst,
                                 int8_t* q, uint16_t* scale, long long R, cudaStream_t st);
cudaError_t launch_dequantize_int8(const int8_t* q, const uint16_t* scale, long long n_rows, int Hkv, int D,
                                   float* out, cudaStream_t st);
cudaError_t launch_quantize_int4(const void* x, int x_bf16, long long n_rows, int Hkv, int D, const int32_t* dst,
                                 uint8_t* q, uint16_t* scale, long long R, cudaStream_t st);
cudaError_t launch_dequantize_int4(const uint8_t* q, const uint16_t* scale, long long n_rows, int Hkv, int D,
                                   float* out, cudaStream_t st);
cudaError_t launch_quantize_fp8(const void* x, int x_bf16, long long n_rows, int Hkv, int D, const int32_t* dst,
                                uint8_t* q, uint16_t* scale, long long R, cudaStream_t st);
cudaError_t launch_dequantize_fp8(const uint8_t* q, const uint16_t* scale, long long n_rows, int Hkv, int D,
                                  float* out, cudaStream_t st);
cudaError_t launch_kv_append(const void* x, long long n_rows, int row_bytes, const int32_t* dst, void* pool,
                             long long R, cudaStream_t st);
cudaError_t launch_sparse_rows(const float* score, int n_max, const int32_t* n_len, int S, int sinks, int recent, int k,
                               const int32_t* row_map, int32_t* rows, int list_len, cudaStream_t st);
size_t sparse_rows_workspace(int S, int n_max);
cudaError_t launch_sparse_rows_ws(const float* score, int n_max, const int32_t* n_len, int S, int sinks, int recent,
                                  int k, const int32_t* row_map, int32_t* rows, int list_len, void* ws,
                                  cudaStream_t st);
cudaError_t launch_validate(const int32_t* rows, const int32_t* kv_len, int S, int L, long long R,
                            long long* status, cudaStream_t st);

// ---------------------------------------------------------------------------
// small device helpers shared by the kernels of this library

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy global -> shared; when !valid nothing is read and
// the 16 destination bytes are zero-filled.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Hardware base-2 exponential (MUFU); ex2(-inf) = +0.
__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float2 f16x2_to_f2(uint32_t w) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  return __half22float2(h);
}
// Byte b (0..3) of w, read as a signed int8, converted to float exactly:
// place (code + 128) in the low mantissa bits of 2^23 and subtract 2^23 + 128.
__device__ __forceinline__ float i8_to_f(uint32_t w_xor80, int b) {
  return __uint_as_float(__byte_perm(w_xor80, 0x4B000000u, 0x7650u | b)) - 8388736.0f;
}

__device__ __forceinline__ void store_out(void* out, size_t i, float x, int dt) {
  if (dt == FA_F32) {
    static_cast<float*>(out)[i] = x;
  } else if (dt == FA_BF16) {
    static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(x);
  } else {
    static_cast<__half*>(out)[i] = __float2half_rn(x);
  }
}

}  // namespace far
