// Cross-split merge of decode partials, run by every thread of the last CTA
// to finish a (slice, KV head).
//
// Split k left, for each of the unit's query-vector rows, its reference max
// m_k (log2 units, -inf if it saw nothing), its sum l_k and its un-normalised
// output O_k (not written when m_k = -inf).  With M = max m_k and weights
// w_k = 2^(m_k - M):  O = sum w_k O_k / sum w_k l_k,  LSE = (M + log2 sum w_k l_k) ln 2.
//
// All (m_k, l_k) are first staged in shared memory with independent loads, the
// weights computed once per (row, split), and the O sums issue 16 float4
// loads at a time (a zero weight skips its value, so an unwritten partial
// never contributes).
#pragma once

#include "fa_internal.cuh"

namespace far {

// Arrival of a finished split CTA (thread 0) on its (slice, KV head) counter.
// True for the last arrival when no split of the unit was aborted: that CTA
// merges, then resets the counter.  An aborted split arrives with
// kAbortArrival added; when the unit's last arrival sees one (or is one), it
// resets the counter itself and nothing is merged, so the counter is zero
// again for the next call whatever happened in this one.
__device__ __forceinline__ bool split_arrive_last(unsigned int* counter, int nsplit, bool aborted) {
  const unsigned int old = atomicAdd(counter, aborted ? kAbortArrival + 1u : 1u);
  if ((old & (kAbortArrival - 1u)) != (unsigned int)(nsplit - 1)) return false;
  if (aborted || old >= kAbortArrival) {
    *counter = 0u;
    return false;
  }
  return true;
}

// part_ml / part_o rows are indexed (unit * nsplit + k) * rows + r; the
// first ns_used splits of the unit are merged (0: all nsplit).
// scratch: at least 2 * nsplit * QV + 2 * QV floats of shared memory.
template <int D>
__device__ __forceinline__ void merge_splits(const DecodeParams& p, size_t unit, int rows, int QV, int s, int g,
                                             float* scratch, int ns_used = 0) {
  const float NEG_INF = __int_as_float(0xff800000);
  const int nthreads = blockDim.x, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
  const int ns = ns_used > 0 ? ns_used : p.nsplit;
  float* sw = scratch;                 // [ns][QV] weights (after step 2; m before)
  float* sl = scratch + ns * QV;       // [ns][QV] sums
  float* fin = sl + ns * QV;           // [QV] merged max, [QV] merged sum
  const size_t base = unit * p.nsplit;
  for (int t = tid; t < ns * QV; t += nthreads) {
    const int k = t / QV, r = t % QV;
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + (base + k) * rows + r);
    sw[t] = ml.x;
    sl[t] = ml.y;
  }
  __syncthreads();
  for (int r = warp; r < QV; r += nwarps) {
    float M = NEG_INF;
    for (int k = lane; k < ns; k += 32) M = fmaxf(M, sw[k * QV + r]);
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, w));
    const float Mu = (M == NEG_INF) ? 0.f : M;
    float L = 0.f;
    for (int k = lane; k < ns; k += 32) {
      const float mk = sw[k * QV + r];
      const float wk = (mk == NEG_INF) ? 0.f : fast_ex2(mk - Mu);
      L = fmaf(sl[k * QV + r], wk, L);
      sw[k * QV + r] = wk;
    }
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) L += __shfl_xor_sync(0xffffffffu, L, w);
    if (lane == 0) {
      fin[r] = M;
      fin[QV + r] = L;
    }
  }
  __syncthreads();
  const int G = p.G;
  // one thread per (row, 4 consecutive dimensions); 16 splits' loads in flight
  constexpr int D4 = D / 4;
  for (int t = tid; t < QV * D4; t += nthreads) {
    const int r = t / D4, d4 = t % D4;
    const float4* po = reinterpret_cast<const float4*>(p.part_o + (base * rows + r) * (size_t)D) + d4;
    const size_t kstride = (size_t)rows * D4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int k = 0;
    for (; k + 16 <= ns; k += 16) {
      float4 v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) v[u] = __ldcg(po + (size_t)(k + u) * kstride);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float wk = sw[(k + u) * QV + r];
        if (wk != 0.f) {
          acc.x = fmaf(wk, v[u].x, acc.x);
          acc.y = fmaf(wk, v[u].y, acc.y);
          acc.z = fmaf(wk, v[u].z, acc.z);
          acc.w = fmaf(wk, v[u].w, acc.w);
        }
      }
    }
    for (; k < ns; ++k) {
      const float wk = sw[k * QV + r];
      const float4 vk = __ldcg(po + (size_t)k * kstride);
      if (wk != 0.f) {
        acc.x = fmaf(wk, vk.x, acc.x);
        acc.y = fmaf(wk, vk.y, acc.y);
        acc.z = fmaf(wk, vk.z, acc.z);
        acc.w = fmaf(wk, vk.w, acc.w);
      }
    }
    const float M = fin[r], Ls = fin[QV + r];
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    const int i = r / G, h = g * G + r % G;
    const size_t oi = ((size_t)s * p.Nq + i) * p.Hq + h;
    store_out(p.out, oi * D + 4 * d4 + 0, acc.x * inv, p.out_dtype);
    store_out(p.out, oi * D + 4 * d4 + 1, acc.y * inv, p.out_dtype);
    store_out(p.out, oi * D + 4 * d4 + 2, acc.z * inv, p.out_dtype);
    store_out(p.out, oi * D + 4 * d4 + 3, acc.w * inv, p.out_dtype);
    if (p.lse && d4 == 0) p.lse[oi] = Ls > 0.f ? (M + __log2f(Ls)) * kLn2 : NEG_INF;
  }
}

// The same merge as a kernel of its own, for small decodes whose last CTA per
// (slice, KV head) would otherwise merge on the critical path with a few
// hundred threads: here every (query-vector row, 4 dimensions) of every unit
// has a thread, whose (m_k, l_k) and O_k loads for 16 splits at a time go out
// together, with a running maximum across groups of 16.  Units that one split
// covers (their output was written by the decode) are skipped.
template <int D>
__global__ void __launch_bounds__(64) merge_splits_kernel(const DecodeParams p) {
  // launched as a programmatic dependent of the decode: wait for that grid to
  // complete and its partials to be visible (a no-op for a plain launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int D4 = D / 4;
  const float NEG_INF = __int_as_float(0xff800000);
  const int unit = blockIdx.y;
  const int s = unit / p.Hkv, g = unit % p.Hkv;
  int n_s = p.L;
  if (p.kv_len) n_s = min(max(__ldg(p.kv_len + s), 0), p.L);
  const int ns = n_s > 0 && p.chunk > 0 ? (n_s + p.chunk - 1) / p.chunk : 1;
  const int QV = p.QV;
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (ns <= 1 || t >= QV * D4) return;
  const int r = t / D4, d4 = t % D4;
  const size_t base = (size_t)unit * p.nsplit;
  const float2* pml = reinterpret_cast<const float2*>(p.part_ml) + base * QV + r;
  const float4* po = reinterpret_cast<const float4*>(p.part_o + (base * QV + r) * (size_t)D) + d4;
  const size_t kstride = (size_t)QV * D4;
  float M = NEG_INF, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < ns; k0 += 16) {
    float2 ml[16];
    float4 v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      ml[u] = k0 + u < ns ? __ldcg(pml + (size_t)(k0 + u) * QV) : make_float2(NEG_INF, 0.f);
      v[u] = k0 + u < ns ? __ldcg(po + (size_t)(k0 + u) * kstride) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float Mg = M;
#pragma unroll
    for (int u = 0; u < 16; ++u) Mg = fmaxf(Mg, ml[u].x);
    if (Mg == NEG_INF) continue;   // nothing seen yet
    const float c = M == NEG_INF ? 0.f : fast_ex2(M - Mg);   // rescale of the groups before
    L *= c;
    acc.x *= c;
    acc.y *= c;
    acc.z *= c;
    acc.w *= c;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const float wk = ml[u].x == NEG_INF ? 0.f : fast_ex2(ml[u].x - Mg);
      if (wk != 0.f) {   // a zero weight skips its value: an unwritten partial never contributes
        L = fmaf(ml[u].y, wk, L);
        acc.x = fmaf(wk, v[u].x, acc.x);
        acc.y = fmaf(wk, v[u].y, acc.y);
        acc.z = fmaf(wk, v[u].z, acc.z);
        acc.w = fmaf(wk, v[u].w, acc.w);
      }
    }
    M = Mg;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int i = r / p.G, h = g * p.G + r % p.G;
  const size_t oi = ((size_t)s * p.Nq + i) * p.Hq + h;
  store_out(p.out, oi * D + 4 * d4 + 0, acc.x * inv, p.out_dtype);
  store_out(p.out, oi * D + 4 * d4 + 1, acc.y * inv, p.out_dtype);
  store_out(p.out, oi * D + 4 * d4 + 2, acc.z * inv, p.out_dtype);
  store_out(p.out, oi * D + 4 * d4 + 3, acc.w * inv, p.out_dtype);
  if (p.lse && d4 == 0) p.lse[oi] = L > 0.f ? (M + __log2f(L)) * kLn2 : NEG_INF;
}

}  // namespace far
