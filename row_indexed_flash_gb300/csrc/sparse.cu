// Sparse row-list builder: sinks + recent + the top-k middle positions of a
// caller-provided score, written as a sorted kv_rows list per query slice.
//
// The selection is the v100llm article's anchor + recent + sink (section 5)
// and the llama.cpp-v100 README's QSA subset of a long context; the list is
// what "llama.cpp 0.9.0 inference boundaries" (section 1) feeds to the
// row-indexed attention.  Ties in score go to the smaller position and a NaN
// ranks below every number, so the list is unique.
//
// One CTA per slice.  The k-th largest score key among the middle positions
// is found by radix selection over an order-preserving 32-bit key (digits of
// 11, 11 and 10 bits, shared-memory histograms with one atomic per distinct
// bin of a warp); one more pass in position order takes every key above it
// and, from the keys equal to it, the first ones by position, and writes them
// between the sinks and the recent positions with block-wide prefix sums.
#include "fa_internal.cuh"

namespace far {

namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelBins = 2048;
constexpr int kSelCopies = 16;   // histogram copies: two warps share one
constexpr size_t kSelSmem = (size_t)kSelCopies * kSelBins * sizeof(int);

// Larger float -> larger key; NaN -> 0, below every number (-inf -> 0x007fffff).
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  if (x != x) return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum of v over the block (1024 threads); *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;   // inclusive sums of the warps
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  *total = warp_sums[31];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kSelThreads) sparse_rows_kernel(const float* __restrict__ score, int n_max,
                                                                  const int32_t* __restrict__ n_len, int sinks,
                                                                  int recent, int k, const int32_t* __restrict__ row_map,
                                                                  int32_t* __restrict__ rows, int list_len) {
  extern __shared__ int hist_copies[];   // [kSelCopies][kSelBins]; copy 0 receives the sums
  int* hist = hist_copies;
  int* my_hist = hist_copies + (size_t)((threadIdx.x >> 5) % kSelCopies) * kSelBins;
  __shared__ int warp_sums[32];
  __shared__ int sel_state[4];   // prefix, remaining
  const int s = blockIdx.x, tid = threadIdx.x;
  const float* sc = score + (size_t)s * n_max;
  const int32_t* map = row_map ? row_map + (size_t)s * n_max : nullptr;
  int32_t* out = rows + (size_t)s * list_len;
  const int n = n_len ? min(max(__ldg(n_len + s), 0), n_max) : n_max;
  const int lo = min(sinks, n);
  const int hi = max(lo, n - recent);
  const int m = hi - lo;
  const int kk = min(k, m);
  auto row_of = [&](int pos) { return map ? __ldg(map + pos) : pos; };
  // the scans run over a grid aligned to 8 elements; 16-byte loads when the row allows
  const int start = lo & ~7;
  const bool vec = (reinterpret_cast<uintptr_t>(sc) & 15u) == 0 && (n_max & 3) == 0;

  // sinks
  for (int pos = tid; pos < lo; pos += kSelThreads) out[pos] = row_of(pos);

  // k-th largest key among the middle positions (all of them when kk == m)
  uint32_t T = 0xffffffffu;   // above every key: with need_eq = 0 nothing is taken (k = 0)
  int need_eq = 0;
  const bool take_all = kk == m;
  if (!take_all && kk > 0) {
    uint32_t prefix = 0u, mask = 0u;
    int remaining = kk;   // how many keys at or below the current prefix still to take
    const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = shifts[pass];
      const uint32_t bmask = (1u << widths[pass]) - 1u;
      for (int b = tid; b < kSelCopies * kSelBins; b += kSelThreads) hist_copies[b] = 0;
      __syncthreads();
      // positions [start, hi) on a grid of 4-element groups (16-byte loads when
      // the row is 16-byte aligned); positions before lo are masked off
      for (int base = start; base < hi; base += kSelThreads * 32) {
        float v[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int pos = base + 4 * (u * kSelThreads + tid);
          if (vec) {
            const float4 f = pos < hi ? __ldg(reinterpret_cast<const float4*>(sc + pos)) : make_float4(0.f, 0.f, 0.f, 0.f);
            v[4 * u] = f.x;
            v[4 * u + 1] = f.y;
            v[4 * u + 2] = f.z;
            v[4 * u + 3] = f.w;
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[4 * u + e] = pos + e < hi ? __ldg(sc + pos + e) : 0.f;
          }
        }
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int pos = base + 4 * ((u / 4) * kSelThreads + tid) + (u % 4);
          const uint32_t key = order_key(v[u]);
          const bool live = pos >= lo && pos < hi && (key & mask) == prefix;
          // one shared-memory atomic per distinct bin of the warp (scores
          // crowd a few bins of the top digit)
          const uint32_t bin = live ? (key >> shift) & bmask : 0xffffffffu;
          const unsigned peers = __match_any_sync(0xffffffffu, bin);
          if (live && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&my_hist[bin], __popc(peers));
        }
      }
      __syncthreads();
      for (int b = tid; b < kSelBins; b += kSelThreads) {
        int t = 0;
#pragma unroll
        for (int c = 0; c < kSelCopies; ++c) t += hist_copies[c * kSelBins + b];
        hist[b] = t;
      }
      __syncthreads();
      if (tid < 32) {
        // lane l owns bins [64*(31-l), 64*(31-l)+64): lane 0 the top ones
        const int b0 = 64 * (31 - tid);
        int local = 0;
        for (int b = 0; b < 64; ++b) local += hist[b0 + b];
        int incl = local;   // inclusive count from the top bin down to this lane's bins
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += y;
        }
        const int above = incl - local;   // keys in higher bins than this lane's
        const bool here = above < remaining && incl >= remaining;
        if (here) {
          int cum = above;
          for (int b = 63; b >= 0; --b) {
            const int c = hist[b0 + b];
            if (cum + c >= remaining) {
              sel_state[0] = (int)(prefix | ((uint32_t)(b0 + b) << shift));
              sel_state[1] = remaining - cum;
              break;
            }
            cum += c;
          }
        }
      }
      __syncthreads();
      prefix = (uint32_t)sel_state[0];
      remaining = sel_state[1];
      mask |= bmask << shift;
      __syncthreads();
    }
    T = prefix;
    need_eq = remaining;   // keys equal to T to take, smallest positions first
  }

  // middle positions in order: every key above T, then the first need_eq
  // equal to T.  Each thread takes 8 consecutive positions per step, so one
  // pair of block-wide prefix sums orders 8192 positions.
  constexpr int PER = 8;
  int out_at = lo, eq_seen = 0;
  for (int base = start; base < hi; base += kSelThreads * PER) {
    const int p0 = base + tid * PER;
    uint32_t keys[PER];
    if (vec) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float4 f = p0 + 4 * h < hi ? __ldg(reinterpret_cast<const float4*>(sc + p0 + 4 * h))
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
        keys[4 * h] = order_key(f.x);
        keys[4 * h + 1] = order_key(f.y);
        keys[4 * h + 2] = order_key(f.z);
        keys[4 * h + 3] = order_key(f.w);
      }
    } else {
#pragma unroll
      for (int u = 0; u < PER; ++u) keys[u] = p0 + u < hi ? order_key(__ldg(sc + p0 + u)) : 0u;
    }
    int n_eq = 0;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int pos = p0 + u;
      n_eq += (pos >= lo && pos < hi && !take_all && keys[u] == T) ? 1 : 0;
    }
    int eq_total = 0;
    int eq_before = eq_seen + block_exclusive_scan(n_eq, warp_sums, &eq_total);
    unsigned sel_bits = 0u;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int pos = p0 + u;
      if (pos < lo || pos >= hi) continue;
      bool sel = take_all || keys[u] > T;
      if (!take_all && keys[u] == T) {
        sel = eq_before < need_eq;
        ++eq_before;
      }
      sel_bits |= (sel ? 1u : 0u) << u;
    }
    int sel_total = 0;
    int at = out_at + block_exclusive_scan(__popc(sel_bits), warp_sums, &sel_total);
#pragma unroll
    for (int u = 0; u < PER; ++u)
      if ((sel_bits >> u) & 1u) out[at++] = row_of(p0 + u);
    out_at += sel_total;
    eq_seen += eq_total;
  }

  // recent positions, then padding
  for (int pos = hi + tid; pos < n; pos += kSelThreads) out[out_at + (pos - hi)] = row_of(pos);
  out_at += n - hi;
  for (int j = out_at + tid; j < list_len; j += kSelThreads) out[j] = -1;
}

}  // namespace

cudaError_t launch_sparse_rows(const float* score, int n_max, const int32_t* n_len, int S, int sinks, int recent, int k,
                               const int32_t* row_map, int32_t* rows, int list_len, cudaStream_t st) {
  if (S == 0) return cudaSuccess;
  static int attr_set[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(sparse_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSelSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  sparse_rows_kernel<<<S, kSelThreads, kSelSmem, st>>>(score, n_max, n_len, sinks, recent, k, row_map, rows, list_len);
  return cudaGetLastError();
}

}  // namespace far
