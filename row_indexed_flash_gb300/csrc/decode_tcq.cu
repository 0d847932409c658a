// Split-KV decode over row-indexed lists for quantised pools (INT8, INT4 or
// FP8 E4M3 codes with one fp16 scale per (row, KV head)), head_dim 128, on the
// 5th-generation tensor cores.
//
// The operation ("llama.cpp 0.9.0 inference boundaries", section 1) is the
// same exact attention over the listed rows as the 16-bit decode; the pool
// format follows the v100llm article (section 2: 64-token pages, INT8/INT4
// KV): codes x = q * s per (row, head), the fp16 scales laid out
// [R/64][Hkv][64].
//
// A quantised tile carries half (INT8) or a quarter (INT4) of the bytes of a
// 16-bit tile, so keeping HBM busy takes many tiles in flight per SM, and the
// codes must be widened before the tensor core can use them.  One CTA per SM,
// each (slice, KV head, split) item streamed in tiles of 64 list entries:
//   gather warp      the listed rows' codes into a ring of NC code stages:
//                    one TMA tile load per matrix when the 64 rows are one
//                    contiguous run (a 64-token page), else cp.async gathers;
//                    it never waits for its copies: they arrive on the
//                    stage's barrier when they land.  It also stages Q as
//                    f16, each query vector times a power of two that puts
//                    its largest element in [2^13, 2^14) (exact for every
//                    element within 2^-29 of the largest; the factor is taken
//                    back out of the logit scale).
//   4 widen warps    16 rows each: codes -> f16 in the MMA's 128-byte-swizzled
//                    layout, into one of NB working buffers: K codes exactly
//                    (|code| <= 127), V as rn_f16(code * s_v) (one rounding,
//                    2^-12 relative); the code stage is released as soon as
//                    its codes are in registers.
//   MMA warp         S = Q K^T into one of NS buffers, O += P V (f16, P from
//                    tensor memory, V MN-major); even tiles accumulate into
//                    O_A, odd tiles into O_B.
//   2 softmax warps  one per parity of the tile index, each with its own
//                    running max/sum and its own O accumulator (warps 0 and
//                    4: both address tensor-memory lanes 0-31, where the
//                    query vectors' rows live).  The K scale is folded into
//                    the logit; P = exp2(x - m) <= 2^8 is rounded once to
//                    f16 (2^-12 relative).  At the end the two streams are
//                    merged like two splits.
// The last CTA to finish a (slice, KV head) merges the splits.  Every wait is
// bounded in time and reported through an error word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

#include "merge.cuh"
#include "tc.cuh"
#include "tmap.cuh"
#include "widen.cuh"

namespace far {

namespace dq {
constexpr int D = 128;
constexpr int BN = 64;        // list entries per tile
constexpr int QROWS = 32;     // query-vector rows kept in shared memory
constexpr int NB = 4;         // 16-bit working buffers (K and V tiles)
constexpr int NS = 4;         // S/P buffers in tensor memory: two per softmax warp
constexpr int NCONV = 4;      // widen warps per group (16 rows each); two groups take alternate tiles
constexpr int NWARP = 12;
// warp roles: 0 softmax (even tiles), 1 MMA, 2 gather, 4 softmax (odd
// tiles), widen group 0: 3, 5, 6, 8; group 1: 7, 9, 10, 11 -- the two softmax
// warps share a scheduler (both address tensor-memory lanes 0-31), each widen
// group spans all four
constexpr int W_SMX0 = 0, W_MMA = 1, W_GATHER = 2, W_SMX1 = 4;
// widen warp -> (group << 2) | index within the group
__device__ __forceinline__ int widen_slot(int warp) {
  switch (warp) {
    case 3: return 0;
    case 5: return 1;
    case 6: return 2;
    case 8: return 3;
    case 7: return 4;
    case 9: return 5;
    case 10: return 6;
    default: return 7;   // 11
  }
}
}  // namespace dq

// KQ: 1 = INT8 codes, 2 = INT4 codes (two per byte), 3 = FP8 E4M3 codes.
template <int QVP, int KQ>
struct DqShape {
  static constexpr int CB = KQ == 2 ? dq::D / 2 : dq::D;   // code bytes of one (row, head)
  static constexpr int CPR = CB / 16;                      // their 16-byte chunks
  static constexpr int QATOM = dq::QROWS * 128;
  static constexpr int Q_BYTES = 2 * QATOM;
  static constexpr int KV_ATOM = dq::BN * 128;
  static constexpr int TILE = 2 * KV_ATOM;                 // one 16-bit K (or V) tile
  static constexpr int CODES = dq::BN * CB;                // one tile's K (or V) codes
  static constexpr int LPR = 32 / QVP;                     // softmax lanes per query vector
  static constexpr int SSTR = dq::BN + (2 * LPR) % 32;     // padded S row stride (floats)
  static constexpr int SPP = dq::BN + LPR % 32;            // padded P row stride (words)
  static constexpr int SROW = SSTR > SPP ? SSTR : SPP;
  static constexpr int STAGE_SM = ((QVP * SROW * 4 + 2 * dq::BN * 4 + 127) / 128) * 128;   // S/P rows + scales
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_B = ((Q_BYTES + 1023) / 1024) * 1024;
  static constexpr int OFF_C = OFF_B + dq::NB * 2 * TILE;
  static constexpr int TAIL = 512 + 128 + 2 * STAGE_SM + 3 * dq::QROWS * 8;   // barriers, misc, staging, exchange, scales
  static constexpr int BUDGET = 227 * 1024 - 1024 - OFF_C - TAIL;
  static constexpr int NC = BUDGET / (2 * CODES) < 8 ? BUDGET / (2 * CODES) : 8;   // code stages
  static constexpr int OFF_BAR = OFF_C + NC * 2 * CODES;
  // q_full, code_full[NC], code_empty[NC], buf_full[NB], buf_empty[NB], s_full[NS], p_full[NS], o_ready[2], drain
  static constexpr int NBAR = 1 + 2 * NC + 2 * dq::NB + 2 * dq::NS + 2 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;      // tmem base, abort flag, last-CTA flag
  static constexpr int OFF_SM = ((OFF_MISC + 16 + 127) / 128) * 128;
  static constexpr int OFF_X = OFF_SM + 2 * STAGE_SM;      // [2][QROWS] (max, sum) of the two streams
  static constexpr int OFF_QS = OFF_X + 2 * dq::QROWS * 8; // [QROWS] logit scale of each query vector
  static constexpr int SMEM_USED = OFF_QS + dq::QROWS * 4;
  static constexpr int SMEM = SMEM_USED + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0;                     // S0..S3: 64 columns each
  static constexpr uint32_t COL_O = dq::NS * dq::BN;       // O_A, O_B: 128 columns each
  static_assert(COL_O + 2 * dq::D <= TMEM_COLS, "tensor memory");
  static_assert(NC >= 3, "code ring too shallow");
  static_assert(NBAR * 8 <= 512, "barrier area");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(OFF_B % 1024 == 0 && TILE % 1024 == 0 && OFF_C % 1024 == 0, "tiles must be 1024-byte aligned");
  static_assert(CODES % 16 == 0 && OFF_SM % 16 == 0 && STAGE_SM % 16 == 0, "16-byte alignment");
  // the 128-row Q operand reads past the 32 stored rows (results never used):
  // those reads stay inside the allocation
  static_assert(OFF_Q + QATOM + 16 * 1024 <= SMEM_USED, "A-operand overrun");
  // split merge scratch (up to 2 * 256 * 32 + 64 floats) reuses the working buffers and code ring
  static_assert(OFF_BAR - OFF_B >= (2 * kDecodeMaxSplits * dq::QROWS + 2 * dq::QROWS) * 4, "merge scratch");
};

struct DqParams {
  DecodeParams a;
  unsigned int* err;
  int tma;   // the code pools have tensor maps
};

namespace {

__device__ __forceinline__ void dq_wait_drain(uint64_t* b, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(b, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

}  // namespace

template <int QVP, int KQ>
__global__ void __launch_bounds__(dq::NWARP * 32, 1)
    fa_rows_decode_tcq_kernel(const DqParams kp, const __grid_constant__ CUtensorMap tk,
                              const __grid_constant__ CUtensorMap tv) {
  using Sh = DqShape<QVP, KQ>;
  using namespace dq;
  constexpr int NC = Sh::NC;
  const DecodeParams& p = kp.a;
  const unsigned long long wait_ns = p.wait_ns;
  const float NEG_INF = __int_as_float(0xff800000);
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Sh::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* code_full = q_full + 1;
  uint64_t* code_empty = code_full + NC;
  uint64_t* buf_full = code_empty + NC;
  uint64_t* buf_empty = buf_full + NB;
  uint64_t* s_full = buf_empty + NB;
  uint64_t* p_full = s_full + NS;
  uint64_t* o_ready = p_full + NS;
  uint64_t* drain = o_ready + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + Sh::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Sh::OFF_MISC + 4);
  int* am_last = reinterpret_cast<int*>(sm + Sh::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int G = p.G, QV = p.QV;
  const bool q_bf16 = p.q_bf16 != 0;
  constexpr bool bf16 = false;   // every MMA operand is f16 here
  int n_s = p.L;
  if (p.kv_len) n_s = min(max(__ldg(p.kv_len + s), 0), p.L);
  const int j0 = split * p.chunk;
  const int cnt = max(min(j0 + p.chunk, n_s) - j0, 0);
  const int T = (cnt + BN - 1) / BN;
  const int32_t* rows_g = p.kv_rows + (size_t)s * p.L + j0;
  const size_t unit = (size_t)s * p.Hkv + g;
  auto entry = [&](int pos) { return pos < cnt ? __ldg(rows_g + pos) : -1; };
  auto valid = [&](int r) { return r >= 0 && (long long)r < p.R; };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NC; ++i) {
      mbar_init(code_full + i, 32);   // one asynchronous arrival per gather lane
      mbar_init(code_empty + i, NCONV);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(buf_full + i, NCONV);
      mbar_init(buf_empty + i, 1);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 1);
    }
    mbar_init(o_ready, 1);
    mbar_init(o_ready + 1, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == W_MMA) {
    tmem_alloc(tmem_holder, Sh::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;

  if (warp == W_GATHER) {
    // ------------------------------------------------------------ gather
    const char* kb = static_cast<const char*>(p.k);
    const char* vb = static_cast<const char*>(p.v);
    if (T > 0) {
      // query vectors -> rows 0..QV-1 of the swizzled Q tile, as f16 times
      // 2^k_r; the row's logit scale becomes qscale * 2^-k_r.  16 lanes per
      // row, 8 elements (one 16-byte chunk) each.
      const uint16_t* qg = static_cast<const uint16_t*>(p.q);
      float* qs = reinterpret_cast<float*>(sm + Sh::OFF_QS);
      for (int r = lane / 16; r < ((QV + 1) & ~1); r += 2) {
        const int c = lane % 16;
        const bool live = r < QV;
        const int i = r / G, h = g * G + r % G;
        float v[8];
        float mx = 0.f;
        if (live) {
          const uint4 w4 = __ldg(reinterpret_cast<const uint4*>(qg + (((size_t)s * p.Nq + i) * p.Hq + h) * D) + c);
          const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            if (q_bf16) {
              v[2 * t] = bf16_lo(wv[t]);
              v[2 * t + 1] = bf16_hi(wv[t]);
            } else {
              const float2 f2 = f16x2_to_f2(wv[t]);
              v[2 * t] = f2.x;
              v[2 * t + 1] = f2.y;
            }
            mx = fmaxf(mx, fmaxf(fabsf(v[2 * t]), fabsf(v[2 * t + 1])));
          }
        }
#pragma unroll
        for (int sh = 1; sh < 16; sh <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, sh));
        // 2^k with the largest |element| * 2^k in [2^13, 2^14); 1 for a zero
        // or non-finite row (its logits are then 0 or NaN either way)
        int k2 = 0;
        if (mx > 0.f && mx <= 3.402823e38f) k2 = min(max(140 - (int)((__float_as_uint(mx) >> 23) & 0xff), -126), 126);
        const float up = __int_as_float((127 + k2) << 23), down = __int_as_float((127 - k2) << 23);
        if (live) {
          uint4 o;
          o.x = pack2h(v[0] * up, v[1] * up, false);
          o.y = pack2h(v[2] * up, v[3] * up, false);
          o.z = pack2h(v[4] * up, v[5] * up, false);
          o.w = pack2h(v[6] * up, v[7] * up, false);
          *reinterpret_cast<uint4*>(sm + Sh::OFF_Q + (c >> 3) * Sh::QATOM + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = o;
          if (c == 0) qs[r] = p.qscale * down;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    }
    int nrow0 = entry(lane), nrow1 = entry(lane + 32);   // the next tile's entries, one tile ahead
    unsigned tma_pend = 0, tma_par = 0;                    // stages with a TMA load issued, and its phase parity
    for (int j = 0; j < T; ++j) {
      const int c = j % NC, u = j / NC;
      if (!__all_sync(0xffffffffu, mbar_wait(code_empty + c, (u & 1) ^ 1, abort_flag, wait_ns))) break;
      const int r0 = valid(nrow0) ? nrow0 : -1, r1 = valid(nrow1) ? nrow1 : -1;
      nrow0 = entry((j + 1) * BN + lane);
      nrow1 = entry((j + 1) * BN + lane + 32);
      unsigned char* Kc = sm + Sh::OFF_C + c * 2 * Sh::CODES;
      unsigned char* Vc = Kc + Sh::CODES;
      const int rbase = __shfl_sync(0xffffffffu, r0, 0);
      const bool contig =
          kp.tma && __all_sync(0xffffffffu, r0 >= 0 && r0 == rbase + lane && r1 >= 0 && r1 == rbase + 32 + lane);
      if (contig) {
        // one 64-row run: a TMA tile load per matrix (x = 0 is 16-byte aligned)
        if (lane == 0) {
          mbar_arrive_expect_tx(code_full + c, 2 * Sh::CODES);
          tma_load_3d(Kc, &tk, 0, g, rbase, code_full + c);
          tma_load_3d(Vc, &tv, 0, g, rbase, code_full + c);
        } else {
          mbar_arrive(code_full + c);
        }
        tma_pend |= 1u << c;
        tma_par = (tma_par & ~(1u << c)) | ((unsigned)(u & 1) << c);
        continue;
      }
#pragma unroll
      for (int it = 0; it < BN * Sh::CPR / 32; ++it) {
        const int f = it * 32 + lane;
        const int e = f / Sh::CPR, q = f % Sh::CPR;   // e < 32 exactly for the first half of the iterations
        const int ra = __shfl_sync(0xffffffffu, r0, e & 31);
        const int rb = __shfl_sync(0xffffffffu, r1, e & 31);
        const int r = e < 32 ? ra : rb;
        const bool okr = r >= 0;
        const size_t go = ((size_t)(okr ? r : 0) * p.Hkv + g) * Sh::CB + q * 16;
        cp_async16(Kc + e * Sh::CB + q * 16, kb + go, okr);
        cp_async16(Vc + e * Sh::CB + q * 16, vb + go, okr);
      }
      cp_async_mbar_arrive_noinc(code_full + c);
    }
    cp_async_wait_all();
    if (lane == 0 && *abort_flag) {   // no TMA load may still be writing when the CTA exits
      for (int c = 0; c < NC; ++c)
        if ((tma_pend >> c) & 1u) dq_wait_drain(code_full + c, (tma_par >> c) & 1u);
    }
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      // With at most 16 query vectors their S rows fit an M = 64 product
      // (rows 0-15 land in tensor-memory lanes 0-15); PV stays at M = 128.
      const uint32_t id_qk = make_idesc_f16(QVP <= 16 ? 64 : 128, BN, bf16, false);
      const uint32_t id_pv = make_idesc_f16(128, D, bf16, true);
      // operand descriptors built once; each MMA only adds a constant offset
      const uint64_t dQ = sdesc_sw128(smem_u32(sm + Sh::OFF_Q), 16, 1024);
      const uint64_t dK = sdesc_sw128(smem_u32(sm + Sh::OFF_B), 16, 1024);
      const uint64_t dV = sdesc_sw128(smem_u32(sm + Sh::OFF_B + Sh::TILE), Sh::KV_ATOM, 1024);
      bool ok = mbar_wait(q_full, 0, abort_flag, wait_ns);
      tc_fence_after();
      int nqk = 0, npv = 0;
      unsigned long long t_idle = 0;
      while (ok && npv < T) {
        bool progressed = false;
        // PV of the oldest tile once its P is written: O_(tile parity) += P V
        if (npv < nqk && mbar_test_wait(p_full + npv % NS, (npv / NS) & 1)) {
          const int b = npv % NB, sb = npv % NS;
          tc_fence_after();
          const uint64_t vb = sdesc_at(dV, b * 2 * Sh::TILE);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tbase + Sh::COL_O + (npv & 1) * D, tbase + Sh::COL_S + sb * BN + kk * 8, sdesc_at(vb, kk * 2048),
                   id_pv, npv > 1 || kk > 0);
          tc_commit(buf_empty + b);
          tc_commit(o_ready + (npv & 1));
          ++npv;
          progressed = true;
        }
        // QK of the next tile once its widened K/V are in a buffer and its S
        // buffer is free (the PV of the tile NS back has been issued)
        if (nqk < T && nqk < npv + NS && mbar_test_wait(buf_full + nqk % NB, (nqk / NB) & 1)) {
          const int b = nqk % NB, sb = nqk % NS;
          tc_fence_after();
          const uint64_t kbd = sdesc_at(dK, b * 2 * Sh::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t a_off = (kk >> 2) * Sh::QATOM + (kk & 3) * 32;
            const uint32_t b_off = (kk >> 2) * Sh::KV_ATOM + (kk & 3) * 32;
            mma_ss(tbase + Sh::COL_S + sb * BN, sdesc_at(dQ, a_off), sdesc_at(kbd, b_off), id_qk, kk > 0);
          }
          tc_commit(s_full + sb);
          ++nqk;
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
      dq_wait_drain(drain, 0);
    }
  } else if (warp == W_SMX0 || warp == W_SMX1) {
    // ------------------------------------------------------------ softmax (tiles of one parity)
    const int w = warp == W_SMX1 ? 1 : 0;
    constexpr int LPR = Sh::LPR, CPL = BN / LPR;   // lanes per row, columns per lane
    const int row = lane / LPR, part = lane % LPR;
    const bool row_ok = row < QV;
    const int lim = (p.mask_kind == FA_MASK_CAUSAL) ? n_s - p.Nq + row / G : n_s - 1;
    float* sS = reinterpret_cast<float*>(sm + Sh::OFF_SM + w * Sh::STAGE_SM);
    uint32_t* sP = reinterpret_cast<uint32_t*>(sS);             // replaces S once every lane has read it
    float* scK = sS + QVP * Sh::SROW;                            // [BN] K scales of the current tile
    bool ok = true;
    const uint32_t tO = tbase + Sh::COL_O + w * D;
    // this row's logit scale (written by the gather warp before q_full)
    float c = 0.f;
    if (T > w) {
      if (!__all_sync(0xffffffffu, mbar_wait(q_full, 0, abort_flag, wait_ns))) ok = false;
      c = row_ok ? reinterpret_cast<const float*>(sm + Sh::OFF_QS)[row] : 0.f;
    }
    float m_used = NEG_INF, l = 0.f;
    auto scale_of = [&](const uint16_t* sc, int r) {
      return valid(r) ? __ldg(sc + ((size_t)(r >> 6) * p.Hkv + g) * kPage + (r & 63)) : (unsigned short)0;
    };
    // entries lane, lane + 32 of this warp's current tile and of its next (two tiles on)
    int cur0 = entry(w * BN + lane), cur1 = entry(w * BN + lane + 32);
    int nx0 = entry((w + 2) * BN + lane), nx1 = entry((w + 2) * BN + lane + 32);
    unsigned short sk0 = scale_of(p.k_scale, cur0), sk1 = scale_of(p.k_scale, cur1);
    int k = 0;
    for (int j = w; ok && j < T; j += 2, ++k) {
      unsigned vb[2];
      vb[0] = __ballot_sync(0xffffffffu, valid(cur0));
      vb[1] = __ballot_sync(0xffffffffu, valid(cur1));
      scK[lane] = __half2float(__ushort_as_half(sk0));
      scK[lane + 32] = __half2float(__ushort_as_half(sk1));
      sk0 = scale_of(p.k_scale, nx0);
      sk1 = scale_of(p.k_scale, nx1);
      cur0 = nx0;
      cur1 = nx1;
      nx0 = entry((j + 4) * BN + lane);
      nx1 = entry((j + 4) * BN + lane + 32);
      const int jb = j0 + j * BN;   // list position of column 0
      // this warp's k-th tile is j = w + 2k; it uses S buffer j % NS
      const int sb = j % NS;
      const uint32_t tS = tbase + Sh::COL_S + sb * BN;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(s_full + sb, (j / NS) & 1, abort_flag, wait_ns)))) break;
      tc_fence_after();
      {
        uint32_t sr[2][32];
        tmem_ld32_nowait(tS, sr[0]);
        tmem_ld32_nowait(tS + 32, sr[1]);
        tmem_wait_ld_tied(sr[0]);
        tmem_wait_ld_tied(sr[1]);
        if (lane < QV) {
          float2* dst = reinterpret_cast<float2*>(sS + lane * Sh::SSTR);
#pragma unroll
          for (int q = 0; q < 16; ++q) dst[q] = make_float2(__uint_as_float(sr[0][2 * q]), __uint_as_float(sr[0][2 * q + 1]));
#pragma unroll
          for (int q = 0; q < 16; ++q)
            dst[16 + q] = make_float2(__uint_as_float(sr[1][2 * q]), __uint_as_float(sr[1][2 * q + 1]));
        }
      }
      __syncwarp();
      // column pairs 2*(part + LPR*kk) of row `row`: logits in log2 units, masked
      const unsigned long long vbits = ((unsigned long long)vb[1] << 32) | vb[0];
      float x[CPL];
      float mx = NEG_INF;
#pragma unroll
      for (int kk = 0; kk < CPL / 2; ++kk) {
        const int col = 2 * (part + LPR * kk);
        const float2 sv = *reinterpret_cast<const float2*>(sS + row * Sh::SSTR + col);
        const float2 sk = *reinterpret_cast<const float2*>(scK + col);
        float v0 = sv.x * (c * sk.x), v1 = sv.y * (c * sk.y);
        if (!(row_ok && ((vbits >> col) & 1ull) && (jb + col <= lim))) v0 = NEG_INF;
        if (!(row_ok && ((vbits >> (col + 1)) & 1ull) && (jb + col + 1 <= lim))) v1 = NEG_INF;
        x[2 * kk] = v0;
        x[2 * kk + 1] = v1;
        mx = fmaxf(mx, fmaxf(v0, v1));
      }
#pragma unroll
      for (int sh = 1; sh < LPR; sh <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, sh));
      const float m_new = fmaxf(m_used, mx);
      const bool need = row_ok && m_new > m_used + 8.f;
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? fast_ex2(m_used - m_new) : 1.f;
        if (need) {
          l *= alpha;
          m_used = m_new;
        }
        if (k > 0) {
          // wait for the PV of this stream's previous tile (the one before it
          // is implied by the S wait: it was issued before this tile's QK)
          const float a_r = __shfl_sync(0xffffffffu, alpha, (lane % QVP) * LPR);
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(o_ready + w, (k - 1) & 1, abort_flag, wait_ns)))) break;
          tc_fence_after();
#pragma unroll
          for (int c4 = 0; c4 < D / 32; ++c4) {
            uint32_t o[32];
            tmem_ld32(tO + c4 * 32, o);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * a_r);
            tmem_st32(tO + c4 * 32, o);
          }
        }
      }
      const float mu = (m_used == NEG_INF) ? 0.f : m_used;
      float sum = 0.f;
      __syncwarp();   // every lane's S reads are done before P overwrites them
#pragma unroll
      for (int kk = 0; kk < CPL / 2; ++kk) {
        const int pp = part + LPR * kk;   // column pair
        const float p0 = fast_ex2(x[2 * kk] - mu), p1 = fast_ex2(x[2 * kk + 1] - mu);
        sum += p0 + p1;
        if (row_ok) sP[row * Sh::SPP + pp] = pack2h(p0, p1, false);
      }
#pragma unroll
      for (int sh = 1; sh < LPR; sh <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
      l += sum;
      __syncwarp();
      {
        uint32_t pk[32];
        if (lane < QV) {
          const uint32_t* src = sP + lane * Sh::SPP;
          if constexpr (Sh::SPP % 4 == 0) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint4 w4 = reinterpret_cast<const uint4*>(src)[q];
              pk[4 * q] = w4.x; pk[4 * q + 1] = w4.y; pk[4 * q + 2] = w4.z; pk[4 * q + 3] = w4.w;
            }
          } else if constexpr (Sh::SPP % 2 == 0) {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const uint2 w2 = reinterpret_cast<const uint2*>(src)[q];
              pk[2 * q] = w2.x; pk[2 * q + 1] = w2.y;
            }
          } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) pk[q] = src[q];
          }
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) pk[q] = 0u;
        }
        tmem_st32_nowait(tS, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full + sb);
    }
    // ---- merge the two streams and write this split's result; warp w
    // writes O columns [64w, 64w + 64)
    const float m_r = __shfl_sync(0xffffffffu, m_used, (lane % QVP) * LPR);
    const float l_r = __shfl_sync(0xffffffffu, l, (lane % QVP) * LPR);
    if (ok && T > 0) ok = __all_sync(0xffffffffu, mbar_wait(drain, 0, abort_flag, wait_ns));
    float2* X = reinterpret_cast<float2*>(sm + Sh::OFF_X);
    if (lane < QROWS) X[w * QROWS + lane] = make_float2(m_r, l_r);
    named_barrier(1, 64);   // both softmax warps, always reached exactly once
    tc_fence_after();
    if (ok && !*abort_flag) {
      const int r = lane;
      const bool own = r < QV;
      const float2 a = X[r], b2 = X[QROWS + r];
      const float M = fmaxf(a.x, b2.x);
      const float wa = (a.x == NEG_INF) ? 0.f : fast_ex2(a.x - M);
      const float wb = (b2.x == NEG_INF) ? 0.f : fast_ex2(b2.x - M);
      const float L = a.y * wa + b2.y * wb;
      const int i = r / G, h = g * G + r % G;
      const size_t oi = ((size_t)s * p.Nq + i) * p.Hq + h;
      const size_t pi = (unit * p.nsplit + split) * QV + r;
      const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col = w * (D / 2) + cc * 32;
        uint32_t oa[32], ob[32];
        if (T > 0) tmem_ld32(tbase + Sh::COL_O + col, oa);
        if (T > 1) tmem_ld32(tbase + Sh::COL_O + D + col, ob);
        float acc[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          float v = 0.f;
          if (T > 0 && wa != 0.f) v = __uint_as_float(oa[q]) * wa;
          if (T > 1 && wb != 0.f) v += __uint_as_float(ob[q]) * wb;
          acc[q] = v;
        }
        if (!own) continue;
        if (p.nsplit == 1) {
#pragma unroll
          for (int q = 0; q < 32; ++q) store_out(p.out, oi * D + col + q, acc[q] * inv, p.out_dtype);
        } else if (M != NEG_INF) {
          float4* dst = reinterpret_cast<float4*>(p.part_o + pi * D + col);
#pragma unroll
          for (int q = 0; q < 8; ++q) dst[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
        }
      }
      if (own && w == 0) {
        if (p.nsplit == 1) {
          if (p.lse) p.lse[oi] = L > 0.f ? (M + __log2f(L)) * kLn2 : NEG_INF;
        } else {
          p.part_ml[pi * 2] = M;
          p.part_ml[pi * 2 + 1] = L;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ widen (16 rows each)
    const int slot = widen_slot(warp);
    const int grp = slot >> 2, cv = slot & 3;   // this warp widens rows 16*cv.. of tiles grp, grp + 2, ...
    constexpr int NIT = 16 * Sh::CPR / 32;
    // V scales of this warp's 16 rows (lane t < 16: row 16*cv + t): each
    // scale is loaded two of this group's tiles before its use, from an entry
    // loaded two tiles before that, so neither load's latency lands on a tile
    auto ventry = [&](int jj) { return lane < 16 ? entry(jj * BN + cv * 16 + lane) : -1; };
    auto vscale = [&](int r) {
      return valid(r) ? __ldg(p.v_scale + ((size_t)(r >> 6) * p.Hkv + g) * kPage + (r & 63)) : (unsigned short)0;
    };
    unsigned short sv0 = vscale(ventry(grp)), sv1 = vscale(ventry(grp + 2));   // tiles j, j + 2
    int re2 = ventry(grp + 4), re3 = ventry(grp + 6);                           // entries of tiles j + 4, j + 6
    for (int j = grp; j < T; j += 2) {
      const unsigned short sv_here = sv0;
      sv0 = sv1;
      sv1 = vscale(re2);
      re2 = re3;
      re3 = ventry(j + 8);
      const int c = j % NC, u = j / NC, b = j % NB, ub = j / NB;
      if (!__all_sync(0xffffffffu, mbar_wait(code_full + c, u & 1, abort_flag, wait_ns))) break;
      const unsigned char* Kc = sm + Sh::OFF_C + c * 2 * Sh::CODES;
      const unsigned char* Vc = Kc + Sh::CODES;
      uint4 ck[NIT], cvv[NIT];
#pragma unroll
      for (int it = 0; it < NIT; ++it) {
        const int f = it * 32 + lane;
        const int e = cv * 16 + f / Sh::CPR, q = f % Sh::CPR;
        ck[it] = *reinterpret_cast<const uint4*>(Kc + e * Sh::CB + q * 16);
        cvv[it] = *reinterpret_cast<const uint4*>(Vc + e * Sh::CB + q * 16);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(code_empty + c);   // the codes are in registers
      if (!__all_sync(0xffffffffu, mbar_wait(buf_empty + b, (ub & 1) ^ 1, abort_flag, wait_ns))) break;
      unsigned char* Kb = sm + Sh::OFF_B + b * 2 * Sh::TILE;
#pragma unroll
      for (int mat = 0; mat < 2; ++mat) {
        unsigned char* tile = Kb + mat * Sh::TILE;
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
          const int f = it * 32 + lane;
          const int e = cv * 16 + f / Sh::CPR, q = f % Sh::CPR;
          const uint4 cw = mat ? cvv[it] : ck[it];
          // V: each value times its row's scale, rounded once to f16
          const unsigned short svr = (unsigned short)__shfl_sync(0xffffffffu, (int)sv_here, f / Sh::CPR);
          const __half2 sv2 = __halves2half2(__ushort_as_half(svr), __ushort_as_half(svr));
          auto vs = [&](uint32_t h2) {
            if (!mat) return h2;
            __half2 x2 = __hmul2(*reinterpret_cast<const __half2*>(&h2), sv2);
            return *reinterpret_cast<uint32_t*>(&x2);
          };
          if constexpr (KQ == 1 || KQ == 3) {
            // 16 codes = columns 16q .. 16q+15: two 16-byte chunks of atom q / 4
            uint2 a, b1, c2, d;
            if constexpr (KQ == 1) {
              a = widen_i8x4(cw.x, bf16), b1 = widen_i8x4(cw.y, bf16);
              c2 = widen_i8x4(cw.z, bf16), d = widen_i8x4(cw.w, bf16);
            } else {
              a = widen_e4m3x4(cw.x), b1 = widen_e4m3x4(cw.y), c2 = widen_e4m3x4(cw.z), d = widen_e4m3x4(cw.w);
            }
            unsigned char* rowp = tile + (q / 4) * Sh::KV_ATOM + e * 128;
            const int k0 = 2 * (q % 4);
            *reinterpret_cast<uint4*>(rowp + ((k0 ^ (e & 7)) << 4)) = make_uint4(vs(a.x), vs(a.y), vs(b1.x), vs(b1.y));
            *reinterpret_cast<uint4*>(rowp + (((k0 + 1) ^ (e & 7)) << 4)) =
                make_uint4(vs(c2.x), vs(c2.y), vs(d.x), vs(d.y));
          } else {
            // 32 codes = columns 32q .. 32q+31: four 16-byte chunks of atom q / 2
            unsigned char* rowp = tile + (q / 2) * Sh::KV_ATOM + e * 128;
            const int k0 = 4 * (q % 2);
            const uint32_t wv[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const uint4 h = widen_i4x8(wv[t], bf16);
              *reinterpret_cast<uint4*>(rowp + (((k0 + t) ^ (e & 7)) << 4)) = make_uint4(vs(h.x), vs(h.y), vs(h.z), vs(h.w));
            }
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(buf_full + b);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, Sh::TMEM_COLS);
  }
  // An expired wait marks the workspace status word; the CTA still arrives
  // on its split counter (marked as aborted) so the counter ends at zero.
  const bool aborted = *abort_flag != 0;
  if (aborted && threadIdx.x == 0 && kp.err) atomicOr(kp.err, FA_WS_WAIT_EXPIRED);
  if (p.nsplit == 1) return;

  // ---- cross-split merge by the last CTA of this (slice, KV head)
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *am_last = split_arrive_last(p.counters + unit, p.nsplit, aborted);
  __syncthreads();
  if (!*am_last) return;
  __threadfence();
  merge_splits<D>(p, unit, QV, QV, s, g, reinterpret_cast<float*>(sm + Sh::OFF_B));
  if (threadIdx.x == 0) p.counters[unit] = 0u;
}

// ---------------------------------------------------------------------------
// host side

namespace {

// Code pool [R][Hkv][CB bytes] as a 3-D byte tensor; box = CB bytes x one
// head x 64 rows, unswizzled (the widen warps read it row-major).
bool dq_map(CUtensorMap* m, const void* base, int CB, int Hkv, long long R) {
  const cuuint64_t dims[3] = {(cuuint64_t)CB, (cuuint64_t)Hkv, (cuuint64_t)R};
  const cuuint64_t strides[2] = {(cuuint64_t)CB, (cuuint64_t)CB * Hkv};
  const cuuint32_t box[3] = {(cuuint32_t)CB, 1, (cuuint32_t)dq::BN};
  return tmap_encode_3d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int QVP, int KQ>
int dq_occupancy() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] > 0) return cached[dev];
  using Sh = DqShape<QVP, KQ>;
  auto kern = fa_rows_decode_tcq_kernel<QVP, KQ>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, dq::NWARP * 32, Sh::SMEM) != cudaSuccess) return 0;
  n = n < 1 ? n : 1;   // 512 tensor-memory columns: one CTA per SM
  cached[dev] = n;
  return n;
}

template <int QVP, int KQ>
cudaError_t dq_launch(const DecodeParams& a, unsigned int* err, cudaStream_t st) {
  if (dq_occupancy<QVP, KQ>() <= 0) return cudaErrorInvalidConfiguration;
  using Sh = DqShape<QVP, KQ>;
  DqParams kp;
  kp.a = a;
  kp.err = err;
  CUtensorMap tk, tv;
  memset(&tk, 0, sizeof(tk));
  memset(&tv, 0, sizeof(tv));
  kp.tma = a.R >= dq::BN && dq_map(&tk, a.k, Sh::CB, a.Hkv, a.R) && dq_map(&tv, a.v, Sh::CB, a.Hkv, a.R);
  dim3 grid(a.nsplit, a.Hkv, a.S);
  fa_rows_decode_tcq_kernel<QVP, KQ><<<grid, dq::NWARP * 32, Sh::SMEM, st>>>(kp, tk, tv);
  return cudaGetLastError();
}

int dq_pow2(int qv) {
  int q = 1;
  while (q < qv) q <<= 1;
  return q;
}

template <int KQ>
int dq_occupancy_q(int qvp) {
  switch (qvp) {
    case 1: return dq_occupancy<1, KQ>();
    case 2: return dq_occupancy<2, KQ>();
    case 4: return dq_occupancy<4, KQ>();
    case 8: return dq_occupancy<8, KQ>();
    case 16: return dq_occupancy<16, KQ>();
    default: return dq_occupancy<32, KQ>();
  }
}

template <int KQ>
cudaError_t dq_launch_q(int qvp, const DecodeParams& a, unsigned int* err, cudaStream_t st) {
  switch (qvp) {
    case 1: return dq_launch<1, KQ>(a, err, st);
    case 2: return dq_launch<2, KQ>(a, err, st);
    case 4: return dq_launch<4, KQ>(a, err, st);
    case 8: return dq_launch<8, KQ>(a, err, st);
    case 16: return dq_launch<16, KQ>(a, err, st);
    default: return dq_launch<32, KQ>(a, err, st);
  }
}

}  // namespace

bool decode_tcq_supported(int D, int kind, int qv, int mask_kind) {
  return D == dq::D && (kind == KV_I8 || kind == KV_I4 || kind == KV_F8) && qv >= 1 && qv <= dq::QROWS &&
         mask_kind != FA_MASK_DENSE;
}

int decode_tcq_occupancy(int kind, int qv) {
  if (kind == KV_I4) return dq_occupancy_q<2>(dq_pow2(qv));
  if (kind == KV_F8) return dq_occupancy_q<3>(dq_pow2(qv));
  return dq_occupancy_q<1>(dq_pow2(qv));
}

cudaError_t decode_tcq_launch(const DecodeParams& a, int kind, unsigned int* err, cudaStream_t st) {
  if (kind == KV_I4) return dq_launch_q<2>(dq_pow2(a.QV), a, err, st);
  if (kind == KV_F8) return dq_launch_q<3>(dq_pow2(a.QV), a, err, st);
  return dq_launch_q<1>(dq_pow2(a.QV), a, err, st);
}

}  // namespace far
