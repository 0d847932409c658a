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
#include "merge.cuh"

namespace far {

template <int D, int QVP, int KIND>
struct DecodeShape {
  static constexpr int ES = (KIND == KV_I8) ? 1 : 2;       // bytes per element
  // dimensions per lane of one row: at least D/32, and 16 (or 64/QVP) so that
  // a row spans few lanes and the cross-lane reduction stays short
  static constexpr int EPL_A = D / 32;
  static constexpr int EPL_B = (64 / QVP) > 16 ? 16 : (64 / QVP);
  static constexpr int EPL = EPL_A > EPL_B ? EPL_A : EPL_B;
  static constexpr int LG = D / EPL;                       // lanes per row
  static constexpr int NG = 32 / LG;                       // rows per warp step
  static constexpr int RT = 8;                             // rows per warp tile
  static constexpr int STEPS = RT / NG;
  static constexpr int LB = EPL * ES;                      // bytes of one row held by a lane
  static constexpr int CH = LB >= 16 ? LB / 16 : 1;        // 16-byte pieces per lane and row
  static constexpr int PB = LB >= 16 ? 16 : LB;            // bytes per piece
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
  static constexpr int MERGE = NW * QVP * (D + 2) * 4;                      // warp merge
  static constexpr int SPLITS = (2 * kDecodeMaxSplits + 2) * QVP * 4;        // split merge
  static constexpr int BODY_A = RING > MERGE ? RING : MERGE;
  static constexpr int BODY = BODY_A > SPLITS ? BODY_A : SPLITS;
  static constexpr int PBUF = NW * (RT * QVP + QVP) * 4;   // per warp: p[RT][QVP], alpha[QVP]
  static constexpr int SMEM = IDX_BYTES + BODY + PBUF + 2 * QVP * 4;
  static_assert(LG >= 1 && LG <= 32 && NG * LG == 32 && STEPS * NG == RT, "bad decode shape");
  static_assert(QVP <= LG, "query vectors must fit in one row group");
};

// Element e (0..EPL-1) of a lane with in-row index k covers dimension:
template <int D, int QVP, int KIND>
__device__ __forceinline__ int lane_dim(int k, int e) {
  using Sh = DecodeShape<D, QVP, KIND>;
  constexpr int PE = Sh::PB / Sh::ES;  // elements per piece
  if constexpr (Sh::LB >= 16) {
    return (k + Sh::LG * (e / PE)) * PE + (e % PE);
  } else {
    return k * Sh::EPL + e;
  }
}

// Loads this lane's EPL elements of one (row, head) from shared memory as
// fp32 pairs (INT8: the raw codes, scaled later).  Pieces are interleaved
// across the lanes of a row so that each quarter warp reads contiguous bytes.
template <int D, int QVP, int KIND>
__device__ __forceinline__ void load_row(const unsigned char* row, int k,
                                         float2 (&x)[DecodeShape<D, QVP, KIND>::EPL / 2]) {
  using Sh = DecodeShape<D, QVP, KIND>;
  constexpr int PE = Sh::PB / Sh::ES;
#pragma unroll
  for (int u = 0; u < Sh::CH; ++u) {
    const unsigned char* src = row + (Sh::LB >= 16 ? (k + Sh::LG * u) * 16 : k * Sh::LB);
    uint32_t w[4];
    if constexpr (Sh::PB == 16) {
      const uint4 v = *reinterpret_cast<const uint4*>(src);
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (Sh::PB == 8) {
      const uint2 v = *reinterpret_cast<const uint2*>(src);
      w[0] = v.x; w[1] = v.y;
    } else if constexpr (Sh::PB == 4) {
      w[0] = *reinterpret_cast<const uint32_t*>(src);
    } else {
      w[0] = *reinterpret_cast<const uint16_t*>(src);
    }
    if constexpr (KIND == KV_I8) {
#pragma unroll
      for (int c = 0; c < (PE + 3) / 4; ++c) {
        const uint32_t xw = w[c] ^ 0x80808080u;
        const float2 bias = make_float2(8388736.0f, 8388736.0f);
        if (4 * c + 1 < PE)
          x[(u * PE + 4 * c) / 2] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(xw, 0x4B000000u, 0x7650u)),
                                                           __uint_as_float(__byte_perm(xw, 0x4B000000u, 0x7651u))),
                                               make_float2(-bias.x, -bias.y));
        if (4 * c + 3 < PE)
          x[(u * PE + 4 * c) / 2 + 1] =
              __fadd2_rn(make_float2(__uint_as_float(__byte_perm(xw, 0x4B000000u, 0x7652u)),
                                     __uint_as_float(__byte_perm(xw, 0x4B000000u, 0x7653u))),
                         make_float2(-bias.x, -bias.y));
      }
    } else {
#pragma unroll
      for (int c = 0; c < PE / 2; ++c) {
        if constexpr (KIND == KV_BF16) {
          x[(u * PE) / 2 + c] = make_float2(bf16_lo(w[c]), bf16_hi(w[c]));
        } else {
          x[(u * PE) / 2 + c] = f16x2_to_f2(w[c]);
        }
      }
    }
  }
}

// Sum across the LG lanes of a row group of QVP per-lane values, transposed:
// afterwards lane k of the group holds the group sum of value k / (LG / QVP).
template <int QVP, int LG>
__device__ __forceinline__ float group_reduce(float (&v)[QVP], int lane) {
  int w = LG / 2;
#pragma unroll
  for (int n = QVP; n > 1; n >>= 1, w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = up ? v[i] : v[i + n / 2];
      const float keep = up ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
#pragma unroll
  for (; w >= 1; w >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], w);
  return v[0];
}

template <int D, int QVP, int KIND>
__global__ void __launch_bounds__(kDecodeWarps * 32) fa_rows_decode_kernel(const DecodeParams p) {
  using Sh = DecodeShape<D, QVP, KIND>;
  constexpr int RT = Sh::RT, EPL = Sh::EPL, LG = Sh::LG, NG = Sh::NG, STEPS = Sh::STEPS;
  constexpr int KB = Sh::KB, CPR = Sh::CPR, NW = Sh::NW, NSTAGE = Sh::NSTAGE;
  constexpr int QSTRIDE = LG / QVP;   // lanes of a group holding the same query vector
  const float NEG_INF = __int_as_float(0xff800000);

  extern __shared__ __align__(128) unsigned char smem[];
  int32_t* idx_s = reinterpret_cast<int32_t*>(smem);
  unsigned char* body = smem + Sh::IDX_BYTES;
  float* pbuf_all = reinterpret_cast<float*>(body + Sh::BODY);
  float* fin = pbuf_all + NW * (RT * QVP + QVP);              // [QVP] merged max, [QVP] merged sum

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = lane / LG, k = lane % LG;
  const int my_qv = k / QSTRIDE;
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

  // ---- this lane's dimensions of every query vector, pre-scaled by scale*log2(e)
  float2 qr[QVP][EPL / 2];
#pragma unroll
  for (int qv = 0; qv < QVP; ++qv) {
    const bool live = qv < p.QV && cnt > 0;
    const int i = qv / G, h = g * G + qv % G;
    const uint16_t* qp = static_cast<const uint16_t*>(p.q) + (((size_t)s * p.Nq + i) * p.Hq + h) * D;
#pragma unroll
    for (int e2 = 0; e2 < EPL / 2; ++e2) {
      float f[2] = {0.f, 0.f};
      if (live) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint32_t b = qp[lane_dim<D, QVP, KIND>(k, 2 * e2 + t)];
          f[t] = (p.q_bf16 ? __uint_as_float(b << 16) : __half2float(__ushort_as_half((unsigned short)b))) * p.qscale;
        }
      }
      qr[qv][e2] = make_float2(f[0], f[1]);
    }
  }
  __syncthreads();

  float m_used = NEG_INF, l_part = 0.f;   // per query vector my_qv; l over this lane's rows
  float2 o[QVP][EPL / 2];
#pragma unroll
  for (int qv = 0; qv < QVP; ++qv)
#pragma unroll
    for (int e2 = 0; e2 < EPL / 2; ++e2) o[qv][e2] = make_float2(0.f, 0.f);

  const int ntiles = (cnt + RT - 1) / RT;
  const int nk = ntiles > warp ? (ntiles - warp + NW - 1) / NW : 0;
  unsigned char* wring = body + warp * NSTAGE * Sh::SLOT;
  float* pbuf = pbuf_all + warp * (RT * QVP + QVP);
  const char* kbase = static_cast<const char*>(p.k);
  const char* vbase = static_cast<const char*>(p.v);
  const int qi = my_qv / G;

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

    // ---- logits of this lane's rows (one per step) for query vector my_qv
    float lg[STEPS];
    float vsc[STEPS];
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
      const int r = st * NG + grp;
      float2 kf[EPL / 2];
      load_row<D, QVP, KIND>(slot + r * KB, k, kf);
      float part[QVP];
#pragma unroll
      for (int qv = 0; qv < QVP; ++qv) {
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int e2 = 0; e2 < EPL / 2; ++e2) acc = __ffma2_rn(qr[qv][e2], kf[e2], acc);
        part[qv] = acc.x + acc.y;
      }
      float x = group_reduce<QVP, LG>(part, lane);
      const int pos = t * RT + r;
      const int row = pos < cnt ? idx_s[pos] : -1;
      bool ok = row >= 0 && my_qv < p.QV;
      vsc[st] = 1.f;
      if constexpr (KIND == KV_I8) {
        const uint32_t kw = reinterpret_cast<const uint32_t*>(slot + 2 * RT * KB)[r];
        const uint32_t vw = reinterpret_cast<const uint32_t*>(slot + 2 * RT * KB)[RT + r];
        const int hi = row & 1;
        x *= __half2float(__ushort_as_half((unsigned short)(hi ? (kw >> 16) : (kw & 0xffffu))));
        vsc[st] = __half2float(__ushort_as_half((unsigned short)(hi ? (vw >> 16) : (vw & 0xffffu))));
      }
      const int jpos = j0 + pos;
      if (p.mask_kind == FA_MASK_CAUSAL) ok = ok && (jpos <= n_s - p.Nq + qi);
      if (ok && p.mask_kind == FA_MASK_DENSE) x += __ldg(p.mask + ((size_t)s * p.Nq + qi) * p.L + jpos) * kLog2e;
      lg[st] = ok ? x : NEG_INF;
    }

    // ---- online softmax; the reference max only moves when it grows by > 2^8
    float tmax = lg[0];
#pragma unroll
    for (int st = 1; st < STEPS; ++st) tmax = fmaxf(tmax, lg[st]);
#pragma unroll
    for (int w = LG; w < 32; w <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, w));
    const float m_new = fmaxf(m_used, tmax);
    const bool need = m_new > m_used + 8.f;
    if (__any_sync(0xffffffffu, need)) {
      const float alpha = need ? fast_ex2(m_used - m_new) : 1.f;
      if (need) {
        l_part *= alpha;
        m_used = m_new;
      }
      if (lane < LG && (lane % QSTRIDE) == 0) pbuf[RT * QVP + my_qv] = alpha;
      __syncwarp();
#pragma unroll
      for (int qv = 0; qv < QVP; ++qv) {
        const float a = pbuf[RT * QVP + qv];
        const float2 a2 = make_float2(a, a);
#pragma unroll
        for (int e2 = 0; e2 < EPL / 2; ++e2) o[qv][e2] = __fmul2_rn(o[qv][e2], a2);
      }
    }
    const float mu = (m_used == NEG_INF) ? 0.f : m_used;
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
      const float pr = fast_ex2(lg[st] - mu);
      l_part += pr;
      if ((k % QSTRIDE) == 0) pbuf[(st * NG + grp) * QVP + my_qv] = pr * vsc[st];
    }
    __syncwarp();

    // ---- PV for this lane's rows
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
      const int r = st * NG + grp;
      float2 vf[EPL / 2];
      load_row<D, QVP, KIND>(slot + RT * KB + r * KB, k, vf);
      float pp[QVP];
      if constexpr (QVP % 4 == 0) {
#pragma unroll
        for (int q4 = 0; q4 < QVP / 4; ++q4) {
          const float4 v4 = reinterpret_cast<const float4*>(pbuf + r * QVP)[q4];
          pp[4 * q4] = v4.x; pp[4 * q4 + 1] = v4.y; pp[4 * q4 + 2] = v4.z; pp[4 * q4 + 3] = v4.w;
        }
      } else {
#pragma unroll
        for (int qv = 0; qv < QVP; ++qv) pp[qv] = pbuf[r * QVP + qv];
      }
#pragma unroll
      for (int qv = 0; qv < QVP; ++qv) {
        const float2 p2 = make_float2(pp[qv], pp[qv]);
#pragma unroll
        for (int e2 = 0; e2 < EPL / 2; ++e2) o[qv][e2] = __ffma2_rn(p2, vf[e2], o[qv][e2]);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();

  // ---- fold the row groups of the warp: O and l over groups (m is shared)
#pragma unroll
  for (int w = LG; w < 32; w <<= 1) {
    l_part += __shfl_xor_sync(0xffffffffu, l_part, w);
#pragma unroll
    for (int qv = 0; qv < QVP; ++qv)
#pragma unroll
      for (int e2 = 0; e2 < EPL / 2; ++e2) {
        o[qv][e2].x += __shfl_xor_sync(0xffffffffu, o[qv][e2].x, w);
        o[qv][e2].y += __shfl_xor_sync(0xffffffffu, o[qv][e2].y, w);
      }
  }
  __syncthreads();

  // ---- merge the warps of this CTA (the ring is free now)
  float* wo = reinterpret_cast<float*>(body);   // [NW][QVP][D]
  float* wm = wo + NW * QVP * D;                // [NW][QVP]
  float* wl = wm + NW * QVP;                    // [NW][QVP]
  if (grp == 0) {
#pragma unroll
    for (int qv = 0; qv < QVP; ++qv)
#pragma unroll
      for (int e2 = 0; e2 < EPL / 2; ++e2) {
        wo[(warp * QVP + qv) * D + lane_dim<D, QVP, KIND>(k, 2 * e2)] = o[qv][e2].x;
        wo[(warp * QVP + qv) * D + lane_dim<D, QVP, KIND>(k, 2 * e2 + 1)] = o[qv][e2].y;
      }
    if ((k % QSTRIDE) == 0) {
      wm[warp * QVP + my_qv] = m_used;
      wl[warp * QVP + my_qv] = l_part;
    }
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
  if (threadIdx.x == 0) am_last = split_arrive_last(p.counters + unit, p.nsplit, false);
  __syncthreads();
  if (!am_last) return;
  __threadfence();

  merge_splits<D>(p, unit, QVP, p.QV, s, g, reinterpret_cast<float*>(body));
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
