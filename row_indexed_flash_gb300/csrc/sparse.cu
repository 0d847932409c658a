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

// Larger float -> larger key; NaN -> 0, below every number (-inf -> 0x007fffff);
// -0.0 and +0.0 compare equal as numbers, so both take +0.0's key and a tie
// between them goes to the smaller position like any other tie.
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  if (x != x) return 0u;
  if (x == 0.f) return 0x80000000u;
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

// ---------------------------------------------------------------------------
// Multi-CTA form (with a workspace): the same selection, each slice spread
// over blocks of kChunk middle positions.  Three histogram passes add block
// histograms into global ones, each followed by a one-warp pick of the next
// digit; a count pass and an ordered write pass place the chosen positions.

constexpr int kChunk = 8192;        // middle positions per block
constexpr int kMThreads = 1024;     // kChunk / 8 positions per thread

struct SliceGeom {
  int n, lo, hi, m, kk;
  bool take_all;
};

__device__ __forceinline__ SliceGeom slice_geom(int s, int n_max, const int32_t* n_len, int sinks, int recent, int k) {
  SliceGeom q;
  q.n = n_len ? min(max(__ldg(n_len + s), 0), n_max) : n_max;
  q.lo = min(sinks, q.n);
  q.hi = max(q.lo, q.n - recent);
  q.m = q.hi - q.lo;
  q.kk = min(k, q.m);
  q.take_all = q.kk == q.m;
  return q;
}

// workspace of one slice: hist[3][kSelBins], state[4] (prefix, remaining), counts[nblk][2] (above, equal)
__device__ __forceinline__ int* ws_hist(int* ws, int s, int nblk, int pass) {
  return ws + (size_t)s * (3 * kSelBins + 4 + 2 * nblk) + pass * kSelBins;
}
__device__ __forceinline__ int* ws_state(int* ws, int s, int nblk) {
  return ws + (size_t)s * (3 * kSelBins + 4 + 2 * nblk) + 3 * kSelBins;
}
__device__ __forceinline__ int* ws_counts(int* ws, int s, int nblk) { return ws_state(ws, s, nblk) + 4; }

__device__ __forceinline__ float load_score(const float* sc, int pos) { return __ldg(sc + pos); }

template <int PASS>
__global__ void __launch_bounds__(kMThreads) sparse_hist_kernel(const float* __restrict__ score, int n_max,
                                                                const int32_t* __restrict__ n_len, int sinks,
                                                                int recent, int k, int* __restrict__ ws, int nblk) {
  __shared__ int hist[4][kSelBins];
  const int s = blockIdx.y, b = blockIdx.x, tid = threadIdx.x;
  const SliceGeom q = slice_geom(s, n_max, n_len, sinks, recent, k);
  if (q.take_all || q.kk == 0) return;
  const int c0 = q.lo + b * kChunk;
  if (c0 >= q.hi) return;
  const int c1 = min(q.hi, c0 + kChunk);
  constexpr int shift = PASS == 0 ? 21 : (PASS == 1 ? 10 : 0);
  constexpr uint32_t bmask = PASS == 2 ? 0x3ffu : 0x7ffu;
  constexpr uint32_t mask = PASS == 0 ? 0u : (PASS == 1 ? 0xffe00000u : 0xfffffc00u);
  const uint32_t prefix = PASS == 0 ? 0u : (uint32_t)ws_state(ws, s, nblk)[0];
  for (int t = tid; t < 4 * kSelBins; t += kMThreads) (&hist[0][0])[t] = 0;
  __syncthreads();
  int* my = hist[(tid >> 5) & 3];
  const float* sc = score + (size_t)s * n_max;
#pragma unroll
  for (int u = 0; u < kChunk / kMThreads; ++u) {
    const int pos = c0 + u * kMThreads + tid;
    const bool in = pos < c1;
    const uint32_t key = in ? order_key(load_score(sc, pos)) : 0u;
    const bool live = in && (key & mask) == prefix;
    const uint32_t bin = live ? (key >> shift) & bmask : 0xffffffffu;
    const unsigned peers = __match_any_sync(0xffffffffu, bin);
    if (live && (tid & 31) == __ffs(peers) - 1) atomicAdd(&my[bin], __popc(peers));
  }
  __syncthreads();
  int* gh = ws_hist(ws, s, nblk, PASS);
  for (int t = tid; t < kSelBins; t += kMThreads) {
    const int v = hist[0][t] + hist[1][t] + hist[2][t] + hist[3][t];
    if (v) atomicAdd(gh + t, v);
  }
}

// One warp per slice: the digit of PASS where the count from the top reaches
// the number still to take; state <- (prefix with that digit, remaining).
template <int PASS>
__global__ void sparse_pick_kernel(int n_max, const int32_t* __restrict__ n_len, int sinks, int recent, int k,
                                   int* __restrict__ ws, int nblk) {
  const int s = blockIdx.x, lane = threadIdx.x;
  const SliceGeom q = slice_geom(s, n_max, n_len, sinks, recent, k);
  if (q.take_all || q.kk == 0) return;
  constexpr int shift = PASS == 0 ? 21 : (PASS == 1 ? 10 : 0);
  int* st = ws_state(ws, s, nblk);
  const int* gh = ws_hist(ws, s, nblk, PASS);
  const uint32_t prefix = PASS == 0 ? 0u : (uint32_t)st[0];
  const int remaining = PASS == 0 ? q.kk : st[1];
  const int b0 = 64 * (31 - lane);
  int local = 0;
  for (int t = 0; t < 64; ++t) local += gh[b0 + t];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int above = incl - local;
  if (above < remaining && incl >= remaining) {
    int cum = above;
    for (int t = 63; t >= 0; --t) {
      const int c = gh[b0 + t];
      if (cum + c >= remaining) {
        st[0] = (int)(prefix | ((uint32_t)(b0 + t) << shift));
        st[1] = remaining - cum;
        break;
      }
      cum += c;
    }
  }
}

// Per block: keys above the threshold and keys equal to it.
__global__ void __launch_bounds__(kMThreads) sparse_count_kernel(const float* __restrict__ score, int n_max,
                                                                 const int32_t* __restrict__ n_len, int sinks,
                                                                 int recent, int k, int* __restrict__ ws, int nblk) {
  __shared__ int red[2];
  const int s = blockIdx.y, b = blockIdx.x, tid = threadIdx.x;
  const SliceGeom q = slice_geom(s, n_max, n_len, sinks, recent, k);
  const int c0 = q.lo + b * kChunk;
  const int c1 = min(q.hi, c0 + kChunk);
  if (tid < 2) red[tid] = 0;
  __syncthreads();
  const uint32_t T = q.kk == 0 ? 0xffffffffu : (uint32_t)ws_state(ws, s, nblk)[0];
  int above = 0, equal = 0;
  if (c0 < q.hi) {
    const float* sc = score + (size_t)s * n_max;
    for (int pos = c0 + tid; pos < c1; pos += kMThreads) {
      const uint32_t key = order_key(load_score(sc, pos));
      above += q.take_all || key > T;
      equal += !q.take_all && key == T;
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    above += __shfl_xor_sync(0xffffffffu, above, o);
    equal += __shfl_xor_sync(0xffffffffu, equal, o);
  }
  if ((tid & 31) == 0) {
    atomicAdd(&red[0], above);
    atomicAdd(&red[1], equal);
  }
  __syncthreads();
  if (tid == 0) {
    int* cnt = ws_counts(ws, s, nblk);
    cnt[2 * b] = red[0];
    cnt[2 * b + 1] = red[1];
  }
}

// Per block: its chosen positions at their place in the list (after the
// sinks and the earlier blocks' choices); block 0 also writes the sinks, the
// recent positions and the padding.
__global__ void __launch_bounds__(kMThreads) sparse_write_kernel(const float* __restrict__ score, int n_max,
                                                                 const int32_t* __restrict__ n_len, int sinks,
                                                                 int recent, int k,
                                                                 const int32_t* __restrict__ row_map,
                                                                 int32_t* __restrict__ rows, int list_len,
                                                                 const int* __restrict__ ws, int nblk) {
  __shared__ int warp_sums[32];
  __shared__ int base[2];
  const int s = blockIdx.y, b = blockIdx.x, tid = threadIdx.x;
  const SliceGeom q = slice_geom(s, n_max, n_len, sinks, recent, k);
  const int32_t* map = row_map ? row_map + (size_t)s * n_max : nullptr;
  int32_t* out = rows + (size_t)s * list_len;
  auto row_of = [&](int pos) { return map ? __ldg(map + pos) : pos; };
  const int* st = ws_state(const_cast<int*>(ws), s, nblk);
  const uint32_t T = (q.take_all || q.kk == 0) ? 0xffffffffu : (uint32_t)st[0];
  const int need_eq = (q.take_all || q.kk == 0) ? 0 : st[1];
  if (b == 0) {
    for (int pos = tid; pos < q.lo; pos += kMThreads) out[pos] = row_of(pos);
    const int r0 = q.lo + q.kk;
    for (int pos = q.hi + tid; pos < q.n; pos += kMThreads) out[r0 + (pos - q.hi)] = row_of(pos);
    for (int jj = r0 + (q.n - q.hi) + tid; jj < list_len; jj += kMThreads) out[jj] = -1;
  }
  const int c0 = q.lo + b * kChunk;
  if (c0 >= q.hi) return;
  const int c1 = min(q.hi, c0 + kChunk);
  if (tid == 0) {
    // output position and equal keys before this block
    const int* cnt = ws_counts(const_cast<int*>(ws), s, nblk);
    int at = q.lo, eq_seen = 0;
    for (int bb = 0; bb < b; ++bb) {
      const int a = cnt[2 * bb], e = cnt[2 * bb + 1];
      at += a + min(e, max(need_eq - eq_seen, 0));
      eq_seen += e;
    }
    base[0] = at;
    base[1] = eq_seen;
  }
  __syncthreads();
  const float* sc = score + (size_t)s * n_max;
  constexpr int PER = kChunk / kMThreads;
  const int p0 = c0 + tid * PER;
  uint32_t keys[PER];
  int n_eq = 0;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int pos = p0 + u;
    keys[u] = pos < c1 ? order_key(load_score(sc, pos)) : 0u;
    n_eq += (pos < c1 && !q.take_all && keys[u] == T) ? 1 : 0;
  }
  int eq_total = 0;
  int eq_before = base[1] + block_exclusive_scan(n_eq, warp_sums, &eq_total);
  unsigned sel_bits = 0u;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int pos = p0 + u;
    if (pos >= c1) continue;
    bool sel = q.take_all || keys[u] > T;
    if (!q.take_all && keys[u] == T) {
      sel = eq_before < need_eq;
      ++eq_before;
    }
    sel_bits |= (sel ? 1u : 0u) << u;
  }
  int sel_total = 0;
  int at = base[0] + block_exclusive_scan(__popc(sel_bits), warp_sums, &sel_total);
#pragma unroll
  for (int u = 0; u < PER; ++u)
    if ((sel_bits >> u) & 1u) out[at++] = row_of(p0 + u);
}

}  // namespace

size_t sparse_rows_workspace(int S, int n_max) {
  const int nblk = n_max > 0 ? (n_max + kChunk - 1) / kChunk : 1;
  return (size_t)S * (3 * kSelBins + 4 + 2 * nblk) * sizeof(int);
}

cudaError_t launch_sparse_rows_ws(const float* score, int n_max, const int32_t* n_len, int S, int sinks, int recent,
                                  int k, const int32_t* row_map, int32_t* rows, int list_len, void* ws,
                                  cudaStream_t st) {
  if (S == 0) return cudaSuccess;
  const int nblk = n_max > 0 ? (n_max + kChunk - 1) / kChunk : 1;
  cudaError_t e = cudaMemsetAsync(ws, 0, sparse_rows_workspace(S, n_max), st);
  if (e != cudaSuccess) return e;
  int* w = static_cast<int*>(ws);
  const dim3 grid(nblk, S);
  sparse_hist_kernel<0><<<grid, kMThreads, 0, st>>>(score, n_max, n_len, sinks, recent, k, w, nblk);
  sparse_pick_kernel<0><<<S, 32, 0, st>>>(n_max, n_len, sinks, recent, k, w, nblk);
  sparse_hist_kernel<1><<<grid, kMThreads, 0, st>>>(score, n_max, n_len, sinks, recent, k, w, nblk);
  sparse_pick_kernel<1><<<S, 32, 0, st>>>(n_max, n_len, sinks, recent, k, w, nblk);
  sparse_hist_kernel<2><<<grid, kMThreads, 0, st>>>(score, n_max, n_len, sinks, recent, k, w, nblk);
  sparse_pick_kernel<2><<<S, 32, 0, st>>>(n_max, n_len, sinks, recent, k, w, nblk);
  sparse_count_kernel<<<grid, kMThreads, 0, st>>>(score, n_max, n_len, sinks, recent, k, w, nblk);
  sparse_write_kernel<<<grid, kMThreads, 0, st>>>(score, n_max, n_len, sinks, recent, k, row_map, rows, list_len, w,
                                                  nblk);
  return cudaGetLastError();
}

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
