// Split-KV decode over row-indexed lists ("llama.cpp 0.9.0 inference
// boundaries", section 1: shared K/V pool, per-slice kv_rows, negative =
// padding with mask -inf; exact attention over the listed rows).
//
// One CTA handles one (slice s, KV head g, split) item: a contiguous range of
// list positions.  Its warps stream the listed rows' K and V through private
// cp.async rings in shared memory (each row of one head is D contiguous
// elements, so a row is a fully coalesced 16-byte-per-lane gather).  All
// Nq*G query vectors that share KV head g are packed into the warp:
//
//   * QK: each lane owns D/32 consecutive dimensions and forms partial dot
//     products for RT rows x QVP query vectors (RT*QVP = 32), then a
//     transposing butterfly leaves lane l with the full dot product of
//     (row l/QVP, query vector l%QVP): 31 shuffles per 32 dot products.
//   * online softmax in base 2 (scale*log2e folded into Q), per query vector
//     across the RT lanes that hold it.
//   * PV: p is broadcast through shared memory and each lane accumulates its
//     D/32 output dimensions for all query vectors.
//
// Warps merge in shared memory; splits write (max, sum, unnormalised O) to the
// workspace and the last CTA to arrive for (s, g) merges them and writes the
// output (an arrival counter, reset by that CTA; nothing waits).
#pragma once

#include "fa_internal.cuh"

namespace far {

template <int D, int QVP, int KIND>
struct DecodeShape {
  static constexpr int RT = 32 / QVP;                      // rows per warp tile
  static constexpr int E = D / 32;                         // dimensions per lane
  static constexpr int ES = (KIND == KV_I8) ? 1 : 2;       // bytes per element
  static constexpr int KB = D * ES;                        // bytes of one (row, head)
  static constexpr int CPR = KB / 16;                      // 16-byte chunks per (row, head)
  static constexpr int TILE_CH = RT * CPR;                 // chunks per tile for K (and for V)
  static constexpr int SC_BYTES = (KIND == KV_I8) ? 2 * RT * 4 : 0;
  static constexpr int SLOT = 2 * RT * KB + SC_BYTES;      // one ring slot: K tile, V tile, scales
  static constexpr int NSTAGE_RAW = (16384 / SLOT) < 2 ? 2 : (16384 / SLOT);
  static constexpr int NSTAGE = NSTAGE_RAW > 8 ? 8 : NSTAGE_RAW;
  static constexpr int NW = kDecodeWarps;
  static constexpr int IDX_BYTES = kDecodeChunkMax * 4;
  static constexpr int RING = NW * NSTAGE * SLOT;
  static constexpr int MERGE = NW * QVP * (D + 2) * 4;
  static constexpr int BODY = RING > MERGE ? RING : MERGE;
  static constexpr int PBUF = NW * 64 * 4;
  static constexpr int SMEM = IDX_BYTES + BODY + PBUF + 2 * QVP * 4;
};

// Loads this lane's E consecutive elements of one (row, head) from shared
// memory and widens them to fp32 (INT8: the raw code, scaled later).
template <int E, int KIND>
__device__ __forceinline__ void load_lane(const unsigned char* p, float (&x)[E]) {
  if constexpr (KIND == KV_I8) {
    if constexpr (E == 2) {
      uint32_t w = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) ^ 0x8080u;
      x[0] = i8_to_f(w, 0);
      x[1] = i8_to_f(w, 1);
    } else {
#pragma unroll
      for (int c = 0; c < E / 4; ++c) {
        uint32_t w = reinterpret_cast<const uint32_t*>(p)[c] ^ 0x80808080u;
#pragma unroll
        for (int b = 0; b < 4; ++b) x[4 * c + b] = i8_to_f(w, b);
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < E / 2; ++c) {
      uint32_t w = reinterpret_cast<const uint32_t*>(p)[c];
      if constexpr (KIND == KV_BF16) {
        x[2 * c] = bf16_lo(w);
        x[2 * c + 1] = bf16_hi(w);
      } else {
        float2 f = f16x2_to_f2(w);
        x[2 * c] = f.x;
        x[2 * c + 1] = f.y;
      }
    }
  }
}

// Sum of 32 per-lane values across the warp, transposed: on return lane l
// holds the warp-wide sum of value index l.
__device__ __forceinline__ float transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? v[i] : v[i + w];
      const float keep = up ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

template <int D, int QVP, int KIND>
__global__ void __launch_bounds__(kDecodeWarps * 32) fa_rows_decode_kernel(const DecodeParams p) {
  using Sh = DecodeShape<D, QVP, KIND>;
  constexpr int RT = Sh::RT, E = Sh::E, KB = Sh::KB, CPR = Sh::CPR, NW = Sh::NW, NSTAGE = Sh::NSTAGE;
  const float NEG_INF = __int_as_float(0xff800000);

  extern __shared__ __align__(128) unsigned char smem[];
  int32_t* idx_s = reinterpret_cast<int32_t*>(smem);
  unsigned char* body = smem + Sh::IDX_BYTES;
  float* pbuf = reinterpret_cast<float*>(body + Sh::BODY);   // [NW][32] p, [NW][32] alpha
  float* fin = pbuf + NW * 64;                                // [QVP] merged max, [QVP] merged sum

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int split = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int G = p.G;
  int n_s = p.L;
  if (p.kv_len) n_s = min(max(__ldg(p.kv_len + s), 0), p.L);
  const int j0 = split * p.chunk;
  const int cnt = max(min(j0 + p.chunk, n_s) - j0, 0);

  // ---- stage this item's row indices (out-of-range rows count as padding)
  const int32_t* rows_g = p.kv_rows + (size_t)s * p.L + j0;
  for (int t = threadIdx.x; t < cnt; t += NW * 32) {
    const int r = __ldg(rows_g + t);
    idx_s[t] = (r >= 0 && (long long)r < p.R) ? r : -1;
  }

  // ---- this lane's slice of every query vector, pre-scaled by scale*log2(e)
  float qr[QVP][E];
#pragma unroll
  for (int qv = 0; qv < QVP; ++qv) {
    if (qv < p.QV && cnt > 0) {
      const int i = qv / G, h = g * G + qv % G;
      const size_t base = (((size_t)s * p.Nq + i) * p.Hq + h) * D + lane * E;
      const uint16_t* qp = static_cast<const uint16_t*>(p.q) + base;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const uint32_t b = qp[e];
        const float f = p.q_bf16 ? __uint_as_float(b << 16) : __half2float(__ushort_as_half((unsigned short)b));
        qr[qv][e] = f * p.qscale;
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) qr[qv][e] = 0.f;
    }
  }
  __syncthreads();

  float m = NEG_INF, l = 0.f;
  float o[QVP][E];
#pragma unroll
  for (int qv = 0; qv < QVP; ++qv)
#pragma unroll
    for (int e = 0; e < E; ++e) o[qv][e] = 0.f;

  const int ntiles = (cnt + RT - 1) / RT;
  const int nk = ntiles > warp ? (ntiles - warp + NW - 1) / NW : 0;
  unsigned char* wring = body + warp * NSTAGE * Sh::SLOT;
  const char* kbase = static_cast<const char*>(p.k);
  const char* vbase = static_cast<const char*>(p.v);

  auto issue = [&](int kk) {
    if (kk < nk) {
      const int t = warp + kk * NW;
      unsigned char* slot = wring + (kk % NSTAGE) * Sh::SLOT;
#pragma unroll
      for (int c = lane; c < Sh::TILE_CH; c += 32) {
        const int r = c / CPR, off = (c % CPR) * 16;
        const int pos = t * RT + r;
        const int row = pos < cnt ? idx_s[pos] : -1;
        const bool ok = row >= 0;
        const size_t go = ((size_t)(ok ? row : 0) * p.Hkv + g) * KB + off;
        cp_async16(slot + r * KB + off, kbase + go, ok);
        cp_async16(slot + RT * KB + r * KB + off, vbase + go, ok);
      }
      if constexpr (KIND == KV_I8) {
        for (int c = lane; c < 2 * RT; c += 32) {
          const int r = c % RT;
          const int pos = t * RT + r;
          const int row = pos < cnt ? idx_s[pos] : -1;
          const bool ok = row >= 0;
          const size_t si = ok ? ((((size_t)row >> 6) * p.Hkv + g) * kPage + (row & (kPage - 1))) & ~(size_t)1 : 0;
          const uint16_t* src = (c < RT ? p.k_scale : p.v_scale) + si;
          cp_async4(slot + 2 * RT * KB + c * 4, src, ok);
        }
      }
    }
    cp_async_commit();
  };

#pragma unroll
  for (int kk = 0; kk < NSTAGE - 1; ++kk) issue(kk);

  for (int kk = 0; kk < nk; ++kk) {
    issue(kk + NSTAGE - 1);
    cp_async_wait<NSTAGE - 1>();
    __syncwarp();
    const unsigned char* slot = wring + (kk % NSTAGE) * Sh::SLOT;
    const int t = warp + kk * NW;

    // QK^T partial sums: value index r*QVP + qv
    float part[32];
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      float kf[E];
      load_lane<E, KIND>(slot + r * KB + lane * E * Sh::ES, kf);
#pragma unroll
      for (int qv = 0; qv < QVP; ++qv) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc = fmaf(qr[qv][e], kf[e], acc);
        part[r * QVP + qv] = acc;
      }
    }
    float logit = transpose_reduce32(part, lane);
    const int my_r = lane / QVP, my_qv = lane % QVP;
    const int pos = t * RT + my_r;
    const int row = pos < cnt ? idx_s[pos] : -1;
    bool ok = row >= 0 && my_qv < p.QV;
    float vsc = 1.f;
    if constexpr (KIND == KV_I8) {
      const uint32_t kw = reinterpret_cast<const uint32_t*>(slot + 2 * RT * KB)[my_r];
      const uint32_t vw = reinterpret_cast<const uint32_t*>(slot + 2 * RT * KB)[RT + my_r];
      const int hi = row & 1;
      logit *= __half2float(__ushort_as_half((unsigned short)(hi ? (kw >> 16) : (kw & 0xffffu))));
      vsc = __half2float(__ushort_as_half((unsigned short)(hi ? (vw >> 16) : (vw & 0xffffu))));
    }
    const int qi = my_qv / G;
    const int jpos = j0 + pos;
    if (p.mask_kind == FA_MASK_CAUSAL) ok = ok && (jpos <= n_s - p.Nq + qi);
    if (ok && p.mask_kind == FA_MASK_DENSE)
      logit += __ldg(p.mask + ((size_t)s * p.Nq + qi) * p.L + jpos) * kLog2e;
    if (!ok) logit = NEG_INF;

    // online softmax over the RT lanes holding the same query vector
    float tmax = logit;
#pragma unroll
    for (int w = QVP; w < 32; w <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, w));
    const float mnew = fmaxf(m, tmax);
    const float muse = (mnew == NEG_INF) ? 0.f : mnew;
    const float pr = fast_ex2(logit - muse);
    const float alpha = fast_ex2(m - muse);
    float ps = pr;
#pragma unroll
    for (int w = QVP; w < 32; w <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, w);
    l = l * alpha + ps;
    m = mnew;

    float* wp = pbuf + warp * 64;
    wp[lane] = pr * vsc;
    if (lane < QVP) wp[32 + lane] = alpha;
    __syncwarp();
#pragma unroll
    for (int qv = 0; qv < QVP; ++qv) {
      const float a = wp[32 + qv];
#pragma unroll
      for (int e = 0; e < E; ++e) o[qv][e] *= a;
    }
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      float vf[E];
      load_lane<E, KIND>(slot + RT * KB + r * KB + lane * E * Sh::ES, vf);
#pragma unroll
      for (int qv = 0; qv < QVP; ++qv) {
        const float pp = wp[r * QVP + qv];
#pragma unroll
        for (int e = 0; e < E; ++e) o[qv][e] = fmaf(pp, vf[e], o[qv][e]);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- merge the warps of this CTA (the ring is free now)
  float* wo = reinterpret_cast<float*>(body);   // [NW][QVP][D]
  float* wm = wo + NW * QVP * D;                // [NW][QVP]
  float* wl = wm + NW * QVP;                    // [NW][QVP]
#pragma unroll
  for (int qv = 0; qv < QVP; ++qv)
#pragma unroll
    for (int e = 0; e < E; ++e) wo[(warp * QVP + qv) * D + lane * E + e] = o[qv][e];
  if (lane < QVP) {
    wm[warp * QVP + lane] = m;
    wl[warp * QVP + lane] = l;
  }
  __syncthreads();

  const size_t unit = (size_t)s * p.Hkv + g;
  for (int t = threadIdx.x; t < QVP * D; t += NW * 32) {
    const int qv = t / D, d = t % D;
    float M = NEG_INF;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w * QVP + qv]);
    const float Mu = (M == NEG_INF) ? 0.f : M;
    float Ls = 0.f, Os = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = fast_ex2(wm[w * QVP + qv] - Mu);
      Ls = fmaf(wl[w * QVP + qv], f, Ls);
      Os = fmaf(wo[(w * QVP + qv) * D + d], f, Os);
    }
    if (p.nsplit == 1) {
      if (qv < p.QV) {
        const int i = qv / G, h = g * G + qv % G;
        const size_t oi = ((size_t)s * p.Nq + i) * p.Hq + h;
        store_out(p.out, oi * D + d, Ls > 0.f ? Os / Ls : 0.f, p.out_dtype);
        if (p.lse && d == 0) p.lse[oi] = Ls > 0.f ? (M + __log2f(Ls)) * kLn2 : NEG_INF;
      }
    } else {
      const size_t pi = (unit * p.nsplit + split) * QVP + qv;
      if (M != NEG_INF) p.part_o[pi * D + d] = Os;
      if (d == 0) {
        p.part_ml[pi * 2] = M;
        p.part_ml[pi * 2 + 1] = Ls;
      }
    }
  }
  if (p.nsplit == 1) return;

  // ---- cross-split merge by the last CTA of this (s, g)
  __shared__ int am_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) am_last = (atomicAdd(p.counters + unit, 1u) == (unsigned)(p.nsplit - 1));
  __syncthreads();
  if (!am_last) return;
  __threadfence();

  const size_t pbase = unit * p.nsplit;
  for (int qv = warp; qv < QVP; qv += NW) {
    float M = NEG_INF;
    for (int k = lane; k < p.nsplit; k += 32) M = fmaxf(M, __ldcg(p.part_ml + ((pbase + k) * QVP + qv) * 2));
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, w));
    const float Mu = (M == NEG_INF) ? 0.f : M;
    float Ls = 0.f;
    for (int k = lane; k < p.nsplit; k += 32) {
      const float mk = __ldcg(p.part_ml + ((pbase + k) * QVP + qv) * 2);
      if (mk != NEG_INF) Ls = fmaf(__ldcg(p.part_ml + ((pbase + k) * QVP + qv) * 2 + 1), fast_ex2(mk - Mu), Ls);
    }
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, w);
    if (lane == 0) {
      fin[qv] = M;
      fin[QVP + qv] = Ls;
    }
  }
  __syncthreads();
  for (int t = threadIdx.x; t < QVP * D; t += NW * 32) {
    const int qv = t / D, d = t % D;
    if (qv >= p.QV) continue;
    const float M = fin[qv], Ls = fin[QVP + qv];
    const float Mu = (M == NEG_INF) ? 0.f : M;
    float Os = 0.f;
    for (int k = 0; k < p.nsplit; ++k) {
      const float mk = __ldcg(p.part_ml + ((pbase + k) * QVP + qv) * 2);
      if (mk != NEG_INF) Os = fmaf(__ldcg(p.part_o + ((pbase + k) * QVP + qv) * D + d), fast_ex2(mk - Mu), Os);
    }
    const int i = qv / G, h = g * G + qv % G;
    const size_t oi = ((size_t)s * p.Nq + i) * p.Hq + h;
    store_out(p.out, oi * D + d, Ls > 0.f ? Os / Ls : 0.f, p.out_dtype);
    if (p.lse && d == 0) p.lse[oi] = Ls > 0.f ? (M + __log2f(Ls)) * kLn2 : NEG_INF;
  }
  if (threadIdx.x == 0) p.counters[unit] = 0u;
}

}  // namespace far

namespace far {

// (D, QVP) pairs built: QVP * D <= 2048 keeps Q and O of a lane in registers.
#define FAR_DECODE_SHAPES(X) \
  X(64, 1) X(64, 2) X(64, 4) X(64, 8) X(64, 16) X(64, 32) \
  X(128, 1) X(128, 2) X(128, 4) X(128, 8) X(128, 16) \
  X(256, 1) X(256, 2) X(256, 4) X(256, 8)

template <int D, int QVP, int KIND>
int decode_occupancy_inst() {
  using Sh = DecodeShape<D, QVP, KIND>;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] > 0) return cached[dev];
  auto kern = fa_rows_decode_kernel<D, QVP, KIND>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Sh::NW * 32, Sh::SMEM) != cudaSuccess) return 0;
  cached[dev] = n;
  return n;
}

template <int D, int QVP, int KIND>
cudaError_t decode_launch_inst(const DecodeParams& p, cudaStream_t st) {
  using Sh = DecodeShape<D, QVP, KIND>;
  if (decode_occupancy_inst<D, QVP, KIND>() <= 0) return cudaErrorInvalidConfiguration;
  dim3 grid(p.nsplit, p.Hkv, p.S);
  fa_rows_decode_kernel<D, QVP, KIND><<<grid, Sh::NW * 32, Sh::SMEM, st>>>(p);
  return cudaGetLastError();
}

template <int KIND>
bool decode_config_kind(int D, int qvp, DecodeConfig* c) {
#define FAR_X(DD, QQ)                                 \
  if (D == DD && qvp == QQ) {                         \
    using Sh = DecodeShape<DD, QQ, KIND>;             \
    c->qvp = QQ;                                      \
    c->rt = Sh::RT;                                   \
    c->nstage = Sh::NSTAGE;                           \
    c->slot_bytes = Sh::SLOT;                         \
    c->smem = Sh::SMEM;                               \
    return true;                                      \
  }
  FAR_DECODE_SHAPES(FAR_X)
#undef FAR_X
  return false;
}

template <int KIND>
int decode_occupancy_kind(int D, int qvp) {
#define FAR_X(DD, QQ) \
  if (D == DD && qvp == QQ) return decode_occupancy_inst<DD, QQ, KIND>();
  FAR_DECODE_SHAPES(FAR_X)
#undef FAR_X
  return 0;
}

template <int KIND>
cudaError_t decode_launch_kind(const DecodeParams& p, int D, int qvp, cudaStream_t st) {
#define FAR_X(DD, QQ) \
  if (D == DD && qvp == QQ) return decode_launch_inst<DD, QQ, KIND>(p, st);
  FAR_DECODE_SHAPES(FAR_X)
#undef FAR_X
  return cudaErrorInvalidValue;
}

// per-kind entry points, each defined in its own translation unit
bool decode_config_bf16(int D, int qvp, DecodeConfig* c);
bool decode_config_f16(int D, int qvp, DecodeConfig* c);
bool decode_config_i8(int D, int qvp, DecodeConfig* c);
int decode_occupancy_bf16(int D, int qvp);
int decode_occupancy_f16(int D, int qvp);
int decode_occupancy_i8(int D, int qvp);
cudaError_t decode_launch_bf16(const DecodeParams& p, int D, int qvp, cudaStream_t st);
cudaError_t decode_launch_f16(const DecodeParams& p, int D, int qvp, cudaStream_t st);
cudaError_t decode_launch_i8(const DecodeParams& p, int D, int qvp, cudaStream_t st);

}  // namespace far
