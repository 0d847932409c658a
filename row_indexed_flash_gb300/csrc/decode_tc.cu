// Split-KV decode over row-indexed lists on the 5th-generation tensor cores.
//
// The operation ("llama.cpp 0.9.0 inference boundaries", section 1): each
// query slice attends exactly to the pool rows its kv_rows list names;
// negative entries are padding (mask -inf).
//
// Decode is bound by the HBM bytes of the gathered K/V rows.  On GB300 the
// CUDA cores cannot form the dot products at that rate without becoming the
// bottleneck (a widening conversion and a fused multiply-add per element for
// every query vector), while the tensor pipe is idle.  So the Nq*G query
// vectors that share a KV head (at most 32) are placed in the rows of an
// MMA tile; the other rows carry whatever lies in shared memory after
// the query rows and only ever produce rows of S, P and O that are never read
// (an MMA row depends on its own A row only).
//
// One CTA handles one (slice, KV head, split) item, 64 list entries per tile:
//   producers      2 warps gather K and 2 gather V (cp.async of the listed
//                  rows into the 128-byte-swizzled layout, padding rows
//                  zero-filled), or one TMA tile load per 64-column atom when
//                  the 64 listed rows are one contiguous pool run.  K and V
//                  have separate rings of 3 stages; the copies arrive on the
//                  stage's barrier by themselves, a K stage is freed by its
//                  QK and a V stage by its PV.
//   MMA warp       S_b = Q K^T (M=64 for at most 16 query vectors, else 128;
//                  N=64; both operands in shared memory), then O += P_b V
//                  (M=128, P from tensor memory, V MN-major), S double-
//                  buffered so the next QK overlaps the softmax.
//   softmax warp   the query vectors' S rows are spread over the warp (32/QVP
//                  lanes per row): masks, a reference max that only moves
//                  when it grows by more than 2^8 (then O is rescaled in
//                  place), P written over S as a 16-bit hi/lo pair, and at the
//                  end the split's (max, sum, O) or the final output.
// INT8 pools (codes with one fp16 scale per (row, KV head)) take the same
// pipeline with all four producer warps on both matrices: they gather the
// codes into the upper half of the stage's tiles, widen them in place to Q's
// 16-bit type (exact: |code| <= 127), and store the rows' scales beside the
// tile; the softmax folds the K scale into the logit and the V scale into P,
// so the MMAs see plain 16-bit operands.
// The last CTA to finish a (slice, KV head) merges the splits (an arrival
// counter in the workspace, reset by that CTA; nothing waits on it).
// Every pipeline wait is bounded in time and reported through an error word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

#include "merge.cuh"
#include "tc.cuh"
#include "tmap.cuh"
#include "widen.cuh"

namespace far {

namespace dk {
constexpr int BN = 64;       // list entries per tile
constexpr int QROWS = 32;    // query-vector rows kept in shared memory
constexpr int NST = 3;       // K/V stages of the 16-bit kernel (2 CTAs per SM)
constexpr int NPROD = 4;     // producer warps (16-bit pools: two gather K, two V)
constexpr int NWARP = 2 + NPROD;   // softmax, producers, MMA
constexpr int MMA_WARP = 1 + NPROD;
}  // namespace dk

// KQ: 0 = 16-bit pool, 1 = INT8 codes + fp16 scales.  NS: K/V stages.
template <int D, int QVP, int KQ, int NS_>
struct DkShape {
  static constexpr int NS = NS_;
  static constexpr int KT = D / 64;                  // 128-byte K atoms per row
  static constexpr int QATOM = dk::QROWS * 128;      // bytes of one atom column of the Q tile
  static constexpr int Q_BYTES = KT * QATOM;
  static constexpr int KV_ATOM = dk::BN * 128;       // bytes of one atom column of a K or V tile
  static constexpr int TILE = KT * KV_ATOM;          // one K (or V) tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = ((Q_BYTES + 1023) / 1024) * 1024;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  static constexpr int OFF_BAR = OFF_V + NS * TILE;
  // q_full, k_full[NS], v_full[NS], k_empty[NS], v_empty[NS], s_full[2], p_full[2], o_ready, drain
  static constexpr int NBAR = 1 + 4 * NS + 2 + 2 + 1 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // S rows of the real query vectors (fp32), then in the same place their P
  // rows (packed 16-bit pairs: BN/2 words of P_hi, BN/2 of P_lo).  The softmax
  // spreads each row over LPR lanes that take interleaved column pairs, so the
  // row strides are padded to put the rows of one access on distinct banks:
  // SSTR = 2*LPR (mod 32) for the 8-byte S reads, SPP = LPR (mod 32) for the
  // 4-byte P writes.
  static constexpr int LPR = 32 / QVP;
  static constexpr int SSTR = dk::BN + (2 * LPR) % 32;
  static constexpr int SPP = dk::BN + LPR % 32;
  static constexpr int SROW = SSTR > SPP ? SSTR : SPP;
  static constexpr int OFF_SS = ((OFF_MISC + 16 + 127) / 128) * 128;
  static constexpr int OFF_SC = OFF_SS + ((QVP * SROW * 4 + 15) / 16) * 16;   // [K, V][BN] fp32 scales (KQ)
  static constexpr int SMEM_USED = OFF_SC + (KQ ? 2 * dk::BN * 4 : 0);
  // code bytes of one (row, head), 16-byte chunks of them, first tile atom holding them (KQ)
  static constexpr int CB = KQ ? D : 2 * D;
  static constexpr int CPRQ = CB / 16;
  static constexpr int A0 = KT - (CB + 127) / 128;
  static constexpr int SMEM = SMEM_USED + 1024;
  static constexpr uint32_t TMEM_COLS = (2 * dk::BN + D) <= 256 ? 256 : 512;
  static constexpr uint32_t COL_S = 0;               // S0, S1: 64 columns each
  static constexpr uint32_t COL_O = 2 * dk::BN;      // O: D columns
  // vector (16-byte) accesses: Q/K/V tiles (1024-byte swizzle atoms), S and P rows
  static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && TILE % 1024 == 0, "tiles must be 1024-byte aligned");
  static_assert(OFF_SS % 16 == 0 && (dk::BN * 4) % 16 == 0, "S/P rows must be 16-byte aligned");
  static_assert(OFF_BAR % 8 == 0, "mbarriers must be 8-byte aligned");
  static_assert(OFF_SC % 16 == 0, "scales must be 16-byte aligned");
  static_assert(!KQ || (A0 >= KT / 2 && CPRQ % 2 == 0), "codes must sit in the tile's upper half");
};

struct DecodeTcParams {
  DecodeParams a;   // QV query vectors per KV head; partials laid out [unit][split][QV][D]
  unsigned int* err;
  int tma_kv;
};

namespace {

__device__ __forceinline__ void wait_drain(uint64_t* b, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(b, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

}  // namespace

// The softmax role (warp 0) of fa_rows_decode_tc_kernel for QVP = the query
// vector count rounded up to a power of two.
template <int D, int QVP, int KQ, int NS>
__device__ __forceinline__ void dk_softmax(const DecodeParams& p, unsigned char* sm, uint64_t* s_full, uint64_t* p_full,
                                           uint64_t* o_ready, uint64_t* o_done, volatile int* abort_flag,
                                           uint32_t tbase, int T, int cnt, int j0, int n_s, const int32_t* rows_g,
                                           size_t unit, int split, int s, int g, bool single) {
  using Sh = DkShape<D, QVP, KQ, NS>;
  using namespace dk;
  const float NEG_INF = __int_as_float(0xff800000);
  const unsigned long long wait_ns = p.wait_ns;
  const int lane = threadIdx.x & 31;
  const int G = p.G, QV = p.QV;
  const bool bf16 = p.q_bf16 != 0;
    // Only rows 0..QV-1 of S are real.  After the tensor-memory load (one row
    // per lane), the real rows are spread over all 32 lanes through shared
    // memory: LPR = 32/QVP lanes per row, CPL = BN/LPR columns per lane, so
    // the exponentials and reductions use the whole warp.  P goes back the
    // same way and is stored over S by the lanes that own its rows.
    float* sS = reinterpret_cast<float*>(sm + Sh::OFF_SS);
    uint32_t* sP = reinterpret_cast<uint32_t*>(sm + Sh::OFF_SS);   // replaces S once every lane has read it
    constexpr int qvp = QVP;
    constexpr int LPR = Sh::LPR, CPL = BN / LPR;   // lanes per row, columns per lane
    const int row = lane / LPR, part = lane % LPR;
    const bool row_ok = row < QV;               // this lane's share is of a real row
    const int lim = (p.mask_kind == FA_MASK_CAUSAL) ? n_s - p.Nq + row / G : n_s - 1;
    const float c = p.qscale;
    const uint32_t tO = tbase + Sh::COL_O;
    float m_used = NEG_INF, l = 0.f;            // state of row `row`, held by its LPR lanes
    // INT8 with f16 queries: P * s_v reaches 256 * 65504 / 127, beyond f16, so
    // it is carried as P * s_v * 2^-8 and O multiplied back by 2^8 at the end
    const float pv_scale = (KQ != 0 && !bf16) ? 0.00390625f : 1.f;
    bool ok = true;
    // List entries lane and lane + 32 of tile j (cur) and j + 1 (nx), loaded
    // ahead so no wait lands on their latency; INT8 scales of those entries
    // one tile ahead (their addresses need the entries).
    auto entry = [&](int pos) { return pos < cnt ? __ldg(rows_g + pos) : -1; };
    auto valid = [&](int r) { return r >= 0 && (long long)r < p.R; };
    auto scale_of = [&](const uint16_t* sc, int r) {
      return valid(r) ? __ldg(sc + ((size_t)(r >> 6) * p.Hkv + g) * kPage + (r & 63)) : (unsigned short)0;
    };
    int cur0 = entry(lane), cur1 = entry(lane + 32);
    int nx0 = entry(BN + lane), nx1 = entry(BN + lane + 32);
    unsigned short sk0 = 0, sk1 = 0, sv0 = 0, sv1 = 0;   // scales of tile j's entries
    if constexpr (KQ != 0) {
      sk0 = scale_of(p.k_scale, cur0);
      sk1 = scale_of(p.k_scale, cur1);
      sv0 = scale_of(p.v_scale, cur0);
      sv1 = scale_of(p.v_scale, cur1);
    }
    float* scK = reinterpret_cast<float*>(sm + Sh::OFF_SC);   // [K, V][BN] scales of the current tile
    for (int j = 0; j < T; ++j) {
      const int b = j & 1;
      unsigned vb[2];
      vb[0] = __ballot_sync(0xffffffffu, valid(cur0));
      vb[1] = __ballot_sync(0xffffffffu, valid(cur1));
      if constexpr (KQ != 0) {
        scK[lane] = __half2float(__ushort_as_half(sk0));
        scK[lane + 32] = __half2float(__ushort_as_half(sk1));
        scK[BN + lane] = __half2float(__ushort_as_half(sv0));
        scK[BN + lane + 32] = __half2float(__ushort_as_half(sv1));
        sk0 = scale_of(p.k_scale, nx0);
        sk1 = scale_of(p.k_scale, nx1);
        sv0 = scale_of(p.v_scale, nx0);
        sv1 = scale_of(p.v_scale, nx1);
      }
      cur0 = nx0;
      cur1 = nx1;
      nx0 = entry((j + 2) * BN + lane);
      nx1 = entry((j + 2) * BN + lane + 32);
      const int jb = j0 + j * BN;   // list position of column 0
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(s_full + b, (j >> 1) & 1, abort_flag, wait_ns)))) break;
      tc_fence_after();
      {
        uint32_t sr[2][32];
        tmem_ld32_nowait(tbase + Sh::COL_S + b * BN, sr[0]);
        tmem_ld32_nowait(tbase + Sh::COL_S + b * BN + 32, sr[1]);
        tmem_wait_ld_tied(sr[0]);
        tmem_wait_ld_tied(sr[1]);
        if (lane < QV) {
          float2* dst = reinterpret_cast<float2*>(sS + lane * Sh::SSTR);
#pragma unroll
          for (int k = 0; k < 16; ++k) dst[k] = make_float2(__uint_as_float(sr[0][2 * k]), __uint_as_float(sr[0][2 * k + 1]));
#pragma unroll
          for (int k = 0; k < 16; ++k)
            dst[16 + k] = make_float2(__uint_as_float(sr[1][2 * k]), __uint_as_float(sr[1][2 * k + 1]));
        }
      }
      __syncwarp();
      // this lane's column pairs 2*(part + LPR*kk) of row `row`, scaled into
      // log2 units, masked
      const unsigned long long vbits = ((unsigned long long)vb[1] << 32) | vb[0];
      float x[CPL];
      float mx = NEG_INF;
#pragma unroll
      for (int kk = 0; kk < CPL / 2; ++kk) {
        const int col = 2 * (part + LPR * kk);
        const float2 sv = *reinterpret_cast<const float2*>(sS + row * Sh::SSTR + col);
        float c0s = c, c1s = c;
        if constexpr (KQ != 0) {
          const float2 sk = *reinterpret_cast<const float2*>(scK + col);
          c0s = c * sk.x;
          c1s = c * sk.y;
        }
        float v0 = sv.x * c0s, v1 = sv.y * c1s;
        if (!(row_ok && ((vbits >> col) & 1ull) && (jb + col <= lim))) v0 = NEG_INF;
        if (!(row_ok && ((vbits >> (col + 1)) & 1ull) && (jb + col + 1 <= lim))) v1 = NEG_INF;
        x[2 * kk] = v0;
        x[2 * kk + 1] = v1;
        mx = fmaxf(mx, fmaxf(v0, v1));
      }
#pragma unroll
      for (int w = 1; w < LPR; w <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, w));
      const float m_new = fmaxf(m_used, mx);
      const bool need = row_ok && m_new > m_used + 8.f;
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? fast_ex2(m_used - m_new) : 1.f;
        if (need) {
          l *= alpha;
          m_used = m_new;
        }
        if (j > 0) {
          // O row r (tensor-memory lane r) is rescaled by the lane that owns it
          const float a_r = __shfl_sync(0xffffffffu, alpha, (lane % qvp) * LPR);
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(o_ready, (j - 1) & 1, abort_flag, wait_ns)))) break;
          tc_fence_after();
#pragma unroll
          for (int c4 = 0; c4 < D / 32; ++c4) {
            uint32_t o[32];
            tmem_ld32(tO + c4 * 32, o);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * a_r);
            tmem_st32(tO + c4 * 32, o);
          }
        }
      }
      const float mu = (m_used == NEG_INF) ? 0.f : m_used;
      float sum = 0.f;
      __syncwarp();   // every lane's S reads are done before P overwrites them
      // P (times the V scale for INT8) goes to the tensor core as two 16-bit
      // terms, P_hi = rn(P) and P_lo = rn(P - P_hi), so the PV product keeps
      // about 16 significant bits of P instead of 8 (bf16)
#pragma unroll
      for (int kk = 0; kk < CPL / 2; ++kk) {
        const int pp = part + LPR * kk;   // column pair
        const float p0 = fast_ex2(x[2 * kk] - mu), p1 = fast_ex2(x[2 * kk + 1] - mu);
        sum += p0 + p1;
        float a0 = p0, a1 = p1;
        if constexpr (KQ != 0) {   // the V scale of each column rides on P (times 2^-8 in f16)
          const float2 sv = *reinterpret_cast<const float2*>(scK + BN + 2 * pp);
          a0 *= sv.x * pv_scale;
          a1 *= sv.y * pv_scale;
        }
        const uint32_t hi = pack2h(a0, a1, bf16);
        float h0, h1;
        if (bf16) {
          h0 = __uint_as_float(hi << 16);
          h1 = __uint_as_float(hi & 0xffff0000u);
        } else {
          const float2 hf = f16x2_to_f2(hi);
          h0 = hf.x;
          h1 = hf.y;
        }
        const uint32_t lo = pack2h(a0 - h0, a1 - h1, bf16);
        if (row_ok) {
          sP[row * Sh::SPP + pp] = hi;
          sP[row * Sh::SPP + BN / 2 + pp] = lo;
        }
      }
#pragma unroll
      for (int w = 1; w < LPR; w <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, w);
      l += sum;
      __syncwarp();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
        if (lane < QV) {
          const uint32_t* src = sP + lane * Sh::SPP + half * (BN / 2);
          if constexpr (Sh::SPP % 4 == 0) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint4 w4 = reinterpret_cast<const uint4*>(src)[k];
              pk[4 * k] = w4.x; pk[4 * k + 1] = w4.y; pk[4 * k + 2] = w4.z; pk[4 * k + 3] = w4.w;
            }
          } else if constexpr (Sh::SPP % 2 == 0) {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const uint2 w2 = reinterpret_cast<const uint2*>(src)[k];
              pk[2 * k] = w2.x; pk[2 * k + 1] = w2.y;
            }
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) pk[k] = src[k];
          }
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) pk[k] = 0u;
        }
        tmem_st32_nowait(tbase + Sh::COL_S + b * BN + half * (BN / 2), pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full + b);
    }
    // ---- this split's result: lane r < QV owns O row r; its (m, l) come from lane r*LPR
    const float m_r = __shfl_sync(0xffffffffu, m_used, (lane % qvp) * LPR);
    const float l_r = __shfl_sync(0xffffffffu, l, (lane % qvp) * LPR);
    // O is final once every PV is done: the MMA warp commits `o_done` (its
    // drain barrier, one phase) after issuing the last one.  o_ready cannot
    // serve here: the last S only implies PV of tile T-3, so that barrier may
    // be two phases behind, where a parity wait cannot tell the phases apart.
    if (ok && T > 0) ok = __all_sync(0xffffffffu, mbar_wait(o_done, 0, abort_flag, wait_ns));
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok) {
      const int r = lane;
      const bool own = r < QV;
      const int i = r / G, h = g * G + r % G;
      const size_t oi = ((size_t)s * p.Nq + i) * p.Hq + h;
      const size_t pi = (unit * p.nsplit + split) * QV + r;
      const float inv = l_r > 0.f ? 1.f / l_r / pv_scale : 0.f;
#pragma unroll
      for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t o[32];
        if (T > 0) {
          tmem_ld32(tO + c4 * 32, o);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = 0u;
        }
        if (!own) continue;
        if (single) {
#pragma unroll
          for (int k = 0; k < 32; ++k) store_out(p.out, oi * D + c4 * 32 + k, __uint_as_float(o[k]) * inv, p.out_dtype);
        } else if (m_r != NEG_INF) {
          float4* dst = reinterpret_cast<float4*>(p.part_o + pi * D + c4 * 32);
          const float os = 1.f / pv_scale;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(__uint_as_float(o[4 * k]) * os, __uint_as_float(o[4 * k + 1]) * os,
                                 __uint_as_float(o[4 * k + 2]) * os, __uint_as_float(o[4 * k + 3]) * os);
        }
      }
      if (own) {
        if (single) {
          if (p.lse) p.lse[oi] = l_r > 0.f ? (m_r + __log2f(l_r)) * kLn2 : NEG_INF;
        } else {
          p.part_ml[pi * 2] = m_r;
          p.part_ml[pi * 2 + 1] = l_r;
        }
      }
    }
}

template <int D, int QVP, int KQ, int NS>
__global__ void __launch_bounds__(dk::NWARP * 32, 2)
    fa_rows_decode_tc_kernel(const DecodeTcParams kp, const __grid_constant__ CUtensorMap tk,
                             const __grid_constant__ CUtensorMap tv) {
  using Sh = DkShape<D, QVP, KQ, NS>;
  using namespace dk;
  constexpr int NST = NS;   // stages of this instance
  const DecodeParams& p = kp.a;
  const unsigned long long wait_ns = p.wait_ns;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Sh::OFF_BAR);
  uint64_t* q_full = bars;
  // K and V stages fill and drain separately: a K stage is free once the QK
  // has read it, a V stage once the PV has
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + NST;
  uint64_t* k_empty = v_full + NST;
  uint64_t* v_empty = k_empty + NST;
  uint64_t* s_full = v_empty + NST;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_ready = p_full + 2;
  uint64_t* drain = o_ready + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + Sh::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Sh::OFF_MISC + 4);
  int* am_last = reinterpret_cast<int*>(sm + Sh::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int G = p.G, QV = p.QV;
  const bool bf16 = p.q_bf16 != 0;
  int n_s = p.L;
  if (p.kv_len) n_s = min(max(__ldg(p.kv_len + s), 0), p.L);
  // splits past the sequence's last entry do nothing and are not merged; a
  // sequence that fits one split writes its result directly
  const int ns_unit = n_s > 0 && p.chunk > 0 ? (n_s + p.chunk - 1) / p.chunk : 1;
  if (split >= ns_unit) return;
  const int j0 = split * p.chunk;
  const int cnt = max(min(j0 + p.chunk, n_s) - j0, 0);
  const int T = (cnt + BN - 1) / BN;
  const int32_t* rows_g = p.kv_rows + (size_t)s * p.L + j0;
  const size_t unit = (size_t)s * p.Hkv + g;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NST; ++i) {
      // 16-bit pools: one arrival per lane of the two warps gathering the
      // matrix (asynchronous, when its copies land; a TMA tile's bytes ride
      // on the first lane's).  INT8: one per producer warp on both, after it
      // has widened its rows of K and V in place.
      mbar_init(k_full + i, KQ == 0 ? 64 : NPROD);
      mbar_init(v_full + i, KQ == 0 ? 64 : NPROD);
      mbar_init(k_empty + i, 1);
      mbar_init(v_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 1);
    }
    mbar_init(o_ready, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_holder, Sh::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;
  // a merge kernel launched after this one (programmatic dependent launch)
  // may be scheduled from here on; it waits for this grid's completion
  if (p.merge_kernel) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp >= 1 && warp <= NPROD) {
    // ------------------------------------------------------------ producers
    // Gathered rows are fetched with cp.async by NPROD warps (the load/store
    // path sustains far more independent row requests than one warp or the
    // TMA gather unit).  A tile whose 64 listed rows form one contiguous pool
    // run is loaded by TMA tile loads instead.
    const int pw = warp - 1;
    constexpr int CPR = D / 8;                  // 16-byte chunks per (row, head)
    constexpr int ROWS = BN / NPROD;            // rows per producer warp (INT8)
    const char* kb = static_cast<const char*>(p.k);
    const char* vb = static_cast<const char*>(p.v);
    if (pw == 0 && T > 0) {
      // query vectors -> rows 0..QV-1 of the swizzled Q tile
      const uint16_t* qg = static_cast<const uint16_t*>(p.q);
      for (int f = lane; f < QV * CPR; f += 32) {
        const int r = f / CPR, c = f % CPR;
        const int i = r / G, h = g * G + r % G;
        const char* src = reinterpret_cast<const char*>(qg + (((size_t)s * p.Nq + i) * p.Hq + h) * D) + c * 16;
        cp_async16(sm + Sh::OFF_Q + (c >> 3) * Sh::QATOM + r * 128 + (((c & 7) ^ (r & 7)) << 4), src, true);
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    }
    if constexpr (KQ == 0) {
      // Warps 1-2 gather K, warps 3-4 gather V, 32 rows of each tile per
      // warp.  Each lane's copies arrive on the stage's barrier by
      // themselves when they land (the MMA thread orders them for the tensor
      // core with a proxy fence), so a warp never waits for its loads: it
      // issues tile j as soon as the QK (K) or PV (V) of tile j - NST has
      // freed the stage.
      const bool isv = pw >= 2;
      const int gw = pw & 1;
      constexpr int GROWS = BN / 2;   // rows per warp of a group
      uint64_t* full = isv ? v_full : k_full;
      uint64_t* empty = isv ? v_empty : k_empty;
      unsigned char* const mat = sm + (isv ? Sh::OFF_V : Sh::OFF_K);
      const char* const src = isv ? vb : kb;
      const void* const tmap = isv ? static_cast<const void*>(&tv) : static_cast<const void*>(&tk);
      unsigned tma_pend = 0, tma_par = 0;   // stages with a TMA load issued, and its phase parity (gw 0, lane 0)
      int nrow0 = lane < cnt ? __ldg(rows_g + lane) : -1;   // next tile's rows, one tile ahead
      int nrow1 = lane + 32 < cnt ? __ldg(rows_g + lane + 32) : -1;
      for (int j = 0; j < T; ++j) {
        const int st = j % NST, u = j / NST;
        if (!__all_sync(0xffffffffu, mbar_wait(empty + st, (u & 1) ^ 1, abort_flag, wait_ns))) break;
        int rows[2] = {nrow0, nrow1};
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (rows[t] < 0 || (long long)rows[t] >= p.R) rows[t] = -1;
        {
          const int pos = (j + 1) * BN + lane;
          nrow0 = pos < cnt ? __ldg(rows_g + pos) : -1;
          nrow1 = pos + 32 < cnt ? __ldg(rows_g + pos + 32) : -1;
        }
        unsigned char* dst = mat + st * Sh::TILE;
        const int r0 = __shfl_sync(0xffffffffu, rows[0], 0);
        bool contig = rows[0] >= 0 && rows[0] == r0 + lane && rows[1] >= 0 && rows[1] == r0 + lane + 32;
        contig = __all_sync(0xffffffffu, contig) && kp.tma_kv;
        if (contig) {
          if (gw == 0 && lane == 0) {
            mbar_arrive_expect_tx(full + st, Sh::TILE);
#pragma unroll
            for (int a = 0; a < Sh::KT; ++a) tma_load_3d(dst + a * Sh::KV_ATOM, tmap, a * 64, g, r0, full + st);
          } else {
            mbar_arrive(full + st);
          }
          tma_pend |= 1u << st;
          tma_par = (tma_par & ~(1u << st)) | ((unsigned)(u & 1) << st);
          continue;
        }
        // this warp's rows gw*GROWS .. gw*GROWS+GROWS-1: 16 (D/8) lanes cover one row
#pragma unroll 4
        for (int it = 0; it < GROWS * CPR / 32; ++it) {
          const int f = it * 32 + lane;
          const int e = gw * GROWS + f / CPR, c = f % CPR;
          const int ra = __shfl_sync(0xffffffffu, rows[0], e & 31);
          const int rb = __shfl_sync(0xffffffffu, rows[1], e & 31);
          const int r = e < 32 ? ra : rb;
          const bool okr = r >= 0;
          const size_t go = ((size_t)(okr ? r : 0) * p.Hkv + g) * (D * 2) + c * 16;
          cp_async16(dst + (c >> 3) * Sh::KV_ATOM + e * 128 + (((c & 7) ^ (e & 7)) << 4), src + go, okr);
        }
        cp_async_mbar_arrive_noinc(full + st);
      }
      cp_async_wait_all();
      if (gw == 0 && lane == 0 && *abort_flag) {   // no TMA load may still be writing when the CTA exits
        for (int c = 0; c < NST; ++c)
          if ((tma_pend >> c) & 1u) wait_drain(full + c, (tma_par >> c) & 1u);
      }
    } else {
      // INT8 codes: each warp widens its rows of a stage in place once they
      // have landed, then publishes it, NST - 1 tiles after issuing it.
      int nrow0 = lane < cnt ? __ldg(rows_g + lane) : -1;   // next tile's rows, one tile ahead
      int nrow1 = lane + 32 < cnt ? __ldg(rows_g + lane + 32) : -1;
      int published = 0;
      auto publish = [&](int t) {
        // every lane reads the code chunks it copied itself, then writes
        // their 16-bit values
        constexpr int NIT = ROWS * Sh::CPRQ / 32;
#pragma unroll
        for (int mat = 0; mat < 2; ++mat) {
          unsigned char* tile = sm + (mat ? Sh::OFF_V : Sh::OFF_K) + (t % NST) * Sh::TILE;
          uint4 cw[NIT];
#pragma unroll
          for (int it = 0; it < NIT; ++it) {
            const int f = it * 32 + lane;
            const int e = pw * ROWS + f / Sh::CPRQ, c = f % Sh::CPRQ;
            cw[it] = *reinterpret_cast<const uint4*>(tile + (Sh::A0 + c / 8) * Sh::KV_ATOM + e * 128 +
                                                     (((c & 7) ^ (e & 7)) << 4));
          }
          __syncwarp();
#pragma unroll
          for (int it = 0; it < NIT; ++it) {
            const int f = it * 32 + lane;
            const int e = pw * ROWS + f / Sh::CPRQ, c = f % Sh::CPRQ;
            // 16 codes = columns 16c .. 16c+15: two 16-byte chunks of atom c / 4
            const uint2 a = widen_i8x4(cw[it].x, bf16), b = widen_i8x4(cw[it].y, bf16);
            const uint2 cc = widen_i8x4(cw[it].z, bf16), d = widen_i8x4(cw[it].w, bf16);
            unsigned char* row = tile + (c / 4) * Sh::KV_ATOM + e * 128;
            const int k0 = 2 * (c % 4);
            *reinterpret_cast<uint4*>(row + ((k0 ^ (e & 7)) << 4)) = make_uint4(a.x, a.y, b.x, b.y);
            *reinterpret_cast<uint4*>(row + (((k0 + 1) ^ (e & 7)) << 4)) = make_uint4(cc.x, cc.y, d.x, d.y);
          }
          __syncwarp();
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(k_full + t % NST);
          mbar_arrive(v_full + t % NST);
        }
      };
      for (int j = 0; j < T; ++j) {
        const int st = j % NST, u = j / NST;
        // publish tile j - (NST - 1) before waiting for stage st: the MMA
        // needs it before it can free that stage (its V half, freed by the
        // PV, is the later of the two)
        if (j >= NST - 1) {
          cp_async_wait<NST - 2>();
          publish(j - (NST - 1));
          published = j - (NST - 1) + 1;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(v_empty + st, (u & 1) ^ 1, abort_flag, wait_ns))) break;
        int rows[2] = {nrow0, nrow1};
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (rows[t] < 0 || (long long)rows[t] >= p.R) rows[t] = -1;
        {
          const int pos = (j + 1) * BN + lane;
          nrow0 = pos < cnt ? __ldg(rows_g + pos) : -1;
          nrow1 = pos + 32 < cnt ? __ldg(rows_g + pos + 32) : -1;
        }
        unsigned char* Ks = sm + Sh::OFF_K + st * Sh::TILE;
        unsigned char* Vs = sm + Sh::OFF_V + st * Sh::TILE;
        // codes of this warp's rows -> the upper atoms of row e, chunk c swizzled as the tile
#pragma unroll
        for (int it = 0; it < ROWS * Sh::CPRQ / 32; ++it) {
          const int f = it * 32 + lane;
          const int e = pw * ROWS + f / Sh::CPRQ, c = f % Sh::CPRQ;
          const int ra = __shfl_sync(0xffffffffu, rows[0], e & 31);
          const int rb = __shfl_sync(0xffffffffu, rows[1], e & 31);
          const int r = e < 32 ? ra : rb;
          const bool okr = r >= 0;
          const size_t go = ((size_t)(okr ? r : 0) * p.Hkv + g) * Sh::CB + c * 16;
          const uint32_t so = (Sh::A0 + c / 8) * Sh::KV_ATOM + e * 128 + (((c & 7) ^ (e & 7)) << 4);
          cp_async16(Ks + so, kb + go, okr);
          cp_async16(Vs + so, vb + go, okr);
        }
        cp_async_commit();
      }
      cp_async_wait<0>();
      if (!*abort_flag)
        for (int t = published; t < T; ++t) publish(t);
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      // With at most 16 query vectors their S rows fit an M=64 product (rows
      // 0-15 land in tensor-memory lanes 0-15), which the tensor pipe runs in
      // about two thirds of the M=128 time at N=64; PV stays at M=128, where
      // M=64 takes as long.
      const uint32_t id_qk = make_idesc_f16(QVP <= 16 ? 64 : 128, BN, bf16, false);
      const uint32_t id_pv = make_idesc_f16(128, D, bf16, true);
      // operand descriptors built once; each MMA adds a constant offset
      const uint64_t dQ = sdesc_sw128(smem_u32(sm + Sh::OFF_Q), 16, 1024);
      const uint64_t dK = sdesc_sw128(smem_u32(sm + Sh::OFF_K), 16, 1024);
      const uint64_t dV = sdesc_sw128(smem_u32(sm + Sh::OFF_V), Sh::KV_ATOM, 1024);
      const uint32_t tO = tbase + Sh::COL_O;
      bool ok = mbar_wait(q_full, 0, abort_flag, wait_ns);
      tc_fence_after();
      // Event-driven issue: QK of the next tile as soon as its K/V have landed
      // (and its S buffer is free: at most one tile ahead of the PVs), PV of
      // the oldest tile as soon as its P is written.  Neither waits for the
      // other, so a late tile never holds back the release of earlier stages.
      int nqk = 0, npv = 0;
      unsigned long long t_idle = 0;
      while (ok && npv < T) {
        bool progressed = false;
        if (nqk < T && nqk < npv + 2 && mbar_test_wait(k_full + nqk % NST, (nqk / NST) & 1)) {
          const int st = nqk % NST, b = nqk & 1;
          tc_fence_after();
          // 16-bit stages are written by cp.async copies that arrived on
          // k_full by themselves: order them before the tensor core's reads
          if constexpr (KQ == 0) fence_proxy_async_smem();
          const uint64_t dKs = sdesc_at(dK, st * Sh::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t a_off = (kk >> 2) * Sh::QATOM + (kk & 3) * 32;
            const uint32_t b_off = (kk >> 2) * Sh::KV_ATOM + (kk & 3) * 32;
            mma_ss(tbase + Sh::COL_S + b * BN, sdesc_at(dQ, a_off), sdesc_at(dKs, b_off), id_qk, kk > 0);
          }
          tc_commit(s_full + b);
          tc_commit(k_empty + st);
          ++nqk;
          progressed = true;
        }
        if (npv < nqk && mbar_test_wait(p_full + (npv & 1), (npv >> 1) & 1) &&
            mbar_test_wait(v_full + npv % NST, (npv / NST) & 1)) {
          const int pst = npv % NST, pb = npv & 1;
          tc_fence_after();
          if constexpr (KQ == 0) fence_proxy_async_smem();
          // O += P_hi V + P_lo V (P_hi in S columns 0..BN/2-1, P_lo after it)
          const uint64_t dVs = sdesc_at(dV, pst * Sh::TILE);
#pragma unroll
          for (int kk = 0; kk < 2 * (BN / 16); ++kk)
            mma_ts(tO, tbase + Sh::COL_S + pb * BN + kk * 8, sdesc_at(dVs, (kk % (BN / 16)) * 2048), id_pv,
                   npv > 0 || kk > 0);
          tc_commit(v_empty + pst);
          tc_commit(o_ready);
          ++npv;
          progressed = true;
        }
        if (progressed) {
          t_idle = 0;
          continue;
        }
        if (t_idle == 0) {
          t_idle = globaltimer();
        } else if (*abort_flag) {
          ok = false;
        } else if (globaltimer() - t_idle > wait_ns) {
          *abort_flag = 1;
          ok = false;
        }
      }
      tc_commit(drain);
      wait_drain(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax (warp 0)
    dk_softmax<D, QVP, KQ, NS>(p, sm, s_full, p_full, o_ready, drain, abort_flag, tbase, T, cnt, j0, n_s, rows_g, unit,
                           split, s, g, ns_unit == 1);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, Sh::TMEM_COLS);
  }
  // An expired wait marks the workspace status word; the CTA still arrives
  // on its split counter (marked as aborted) so the counter ends at zero.
  const bool aborted = *abort_flag != 0;
  if (aborted && threadIdx.x == 0 && kp.err) atomicOr(kp.err, FA_WS_WAIT_EXPIRED);
  if (ns_unit == 1 || p.merge_kernel) return;

  // ---- cross-split merge by the last CTA of this (slice, KV head)
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *am_last = split_arrive_last(p.counters + unit, ns_unit, aborted);
  __syncthreads();
  if (!*am_last) return;
  __threadfence();
  merge_splits<D>(p, unit, QV, QV, s, g, reinterpret_cast<float*>(sm + Sh::OFF_K), ns_unit);
  if (threadIdx.x == 0) p.counters[unit] = 0u;
}

// ---------------------------------------------------------------------------
// host side

namespace {

bool dk_map(CUtensorMap* m, const void* base, bool bf16, int D, int Hkv, long long R) {
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)R};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * Hkv * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)dk::BN};
  return tmap_encode_3d(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, dims,
                        strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int D, int QVP, int KQ, int NS>
int dk_occupancy() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] > 0) return cached[dev];
  using Sh = DkShape<D, QVP, KQ, NS>;
  auto kern = fa_rows_decode_tc_kernel<D, QVP, KQ, NS>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, dk::NWARP * 32, Sh::SMEM) != cudaSuccess) return 0;
  // tensor memory also bounds residency: 512 columns per SM
  const int by_tmem = 512 / (int)Sh::TMEM_COLS;
  n = n < by_tmem ? n : by_tmem;
  cached[dev] = n;
  return n;
}

template <int D, int QVP, int KQ, int NS>
cudaError_t dk_launch(const DecodeParams& a, unsigned int* err, cudaStream_t st) {
  if (dk_occupancy<D, QVP, KQ, NS>() <= 0) return cudaErrorInvalidConfiguration;
  DecodeTcParams kp;
  kp.a = a;
  kp.err = err;
  // TMA tile loads of contiguous runs (16-bit pools only: codes are widened by the producers)
  kp.tma_kv = KQ == 0 && a.R >= dk::BN;
  const bool bf16 = a.q_bf16 != 0;
  CUtensorMap tk, tv;
  memset(&tk, 0, sizeof(tk));
  memset(&tv, 0, sizeof(tv));
  if (kp.tma_kv) {
    if (!dk_map(&tk, a.k, bf16, D, a.Hkv, a.R) || !dk_map(&tv, a.v, bf16, D, a.Hkv, a.R)) return cudaErrorInvalidValue;
  }
  dim3 grid(a.nsplit, a.Hkv, a.S);
  fa_rows_decode_tc_kernel<D, QVP, KQ, NS><<<grid, dk::NWARP * 32, DkShape<D, QVP, KQ, NS>::SMEM, st>>>(kp, tk, tv);
  return cudaGetLastError();
}

}  // namespace

bool decode_tc_supported(int D, int kind, int qv, int mask_kind) {
  return (D == 128 || D == 256) && (kind == KV_BF16 || kind == KV_F16 || kind == KV_I8) && qv >= 1 &&
         qv <= dk::QROWS && mask_kind != FA_MASK_DENSE;
}

// Stages per CTA: the 16-bit kernel runs two CTAs per SM with three stages
// each; an INT8 stage keeps only half its bytes in flight (codes land in the
// upper half of a 16-bit tile), so at D 128 the INT8 kernel runs one CTA per
// SM with six stages.
constexpr int dk_stages(int D, int KQ) { return KQ != 0 && D == 128 ? 6 : dk::NST; }

static int qv_pow2(int qv) {
  int q = 1;
  while (q < qv) q <<= 1;
  return q;
}

template <int D, int KQ>
int dk_occupancy_d(int qvp) {
  switch (qvp) {
    case 1: return dk_occupancy<D, 1, KQ, dk_stages(D, KQ)>();
    case 2: return dk_occupancy<D, 2, KQ, dk_stages(D, KQ)>();
    case 4: return dk_occupancy<D, 4, KQ, dk_stages(D, KQ)>();
    case 8: return dk_occupancy<D, 8, KQ, dk_stages(D, KQ)>();
    case 16: return dk_occupancy<D, 16, KQ, dk_stages(D, KQ)>();
    default: return dk_occupancy<D, 32, KQ, dk_stages(D, KQ)>();
  }
}

template <int D, int KQ>
cudaError_t dk_launch_d(int qvp, const DecodeParams& a, unsigned int* err, cudaStream_t st) {
  switch (qvp) {
    case 1: return dk_launch<D, 1, KQ, dk_stages(D, KQ)>(a, err, st);
    case 2: return dk_launch<D, 2, KQ, dk_stages(D, KQ)>(a, err, st);
    case 4: return dk_launch<D, 4, KQ, dk_stages(D, KQ)>(a, err, st);
    case 8: return dk_launch<D, 8, KQ, dk_stages(D, KQ)>(a, err, st);
    case 16: return dk_launch<D, 16, KQ, dk_stages(D, KQ)>(a, err, st);
    default: return dk_launch<D, 32, KQ, dk_stages(D, KQ)>(a, err, st);
  }
}

int decode_tc_occupancy(int D, int kind, int qv) {
  const int q = qv_pow2(qv);
  const bool quant = kind == KV_I8;
  if (D == 128) return quant ? dk_occupancy_d<128, 1>(q) : dk_occupancy_d<128, 0>(q);
  if (D == 256) return quant ? dk_occupancy_d<256, 1>(q) : dk_occupancy_d<256, 0>(q);
  return 0;
}

int decode_tc_tile() { return dk::BN; }

// Launched as a programmatic dependent of the decode: its CTAs may be
// scheduled while the decode's last CTAs run, and wait (griddepcontrol.wait)
// for the decode grid to complete and its writes to be visible.
cudaError_t decode_merge_launch(const DecodeParams& a, int D, cudaStream_t st) {
  const int items = a.QV * (D / 4);
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)((items + 63) / 64), (unsigned)(a.S * a.Hkv));
  cfg.blockDim = dim3(64);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (D == 128) return cudaLaunchKernelEx(&cfg, merge_splits_kernel<128>, a);
  if (D == 256) return cudaLaunchKernelEx(&cfg, merge_splits_kernel<256>, a);
  return cudaErrorInvalidValue;
}

cudaError_t decode_tc_launch(const DecodeParams& a, int D, int kind, unsigned int* err, cudaStream_t st) {
  const int q = qv_pow2(a.QV);
  const bool quant = kind == KV_I8;
  if (D == 128) return quant ? dk_launch_d<128, 1>(q, a, err, st) : dk_launch_d<128, 0>(q, a, err, st);
  if (D == 256) return quant ? dk_launch_d<256, 1>(q, a, err, st) : dk_launch_d<256, 0>(q, a, err, st);
  return cudaErrorInvalidValue;
}

}  // namespace far
