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
// Keys ride in the MMA's M dimension and the query vectors of the KV head (at
// most 32) in N, so a 128-key tile costs 16 small MMAs and the softmax is one
// thread per key.  Per tile of 128 list entries (two 64-row halves, a page
// each):
//   gather warp      the listed rows' K and V codes into a ring of code
//                    stages (128-byte rows swizzled, 64-byte INT4 rows plain):
//                    one TMA tile load per half and matrix when the half is
//                    one contiguous pool run, else cp.async gathers; the
//                    copies arrive on the stage's barrier by themselves.  It
//                    also stages Q^T: the query vectors as f16 rows, each
//                    times a power of two that puts its largest element in
//                    [2^13, 2^14) (exact for every element within 2^-29 of the
//                    largest), taken back out of its logit scale.
//   widen warps (4)  one thread per key: its K codes widened exactly to f16
//                    into a K tile in tensor memory (lane = key).
//   MMA warps (2)    one issues S^T = K Q^T (A = the K tile in tensor
//                    memory, B = Q^T), the other O^T += V^T P^T (A = the V
//                    tile read MN-major, B = P^T in shared memory) into the
//                    O^T accumulator of the tile's softmax group; O^T holds a
//                    lane per head dimension and a column per query vector.
//   softmax (n x 4)  three groups of four warps (two for more than 8 query
//                    vectors) take the tiles in turn, each with its own
//                    references, row sums and O^T, so that one group's
//                    barriers and waits overlap the others' work; one
//                    thread per key.  Each tile starts with its V codes,
//                    widened exactly to f16 in place: the f16 V tile (rows =
//                    keys) takes the whole code stage once the widen warps
//                    hold its K codes, and the stage is released when the PV
//                    that reads it completes.  Then the key's logits (the K
//                    scale folded in),
//                    P = exp2(logit - m) against a reference max m per query
//                    vector that moves only when a logit exceeds it by more
//                    than 2^8 -- detected by each thread and agreed across the
//                    group's four warps at one bounded barrier per tile,
//                    followed only in that rare case by a maximum over the
//                    tile's keys and a rescale of the group's O^T -- then the
//                    O weight P * s_v as f16 into P^T, kept below 2^8 by a
//                    second lazy reference of the same kind over
//                    logit + log2|s_v|.  At the end the first group (now one
//                    thread per head dimension) combines the groups' states
//                    and normalises.
// The last CTA to finish a (slice, KV head) merges the splits.  Every wait is
// bounded in time and reported through the workspace status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "merge.cuh"
#include "tc.cuh"
#include "tmap.cuh"
#include "widen.cuh"

namespace far {

namespace dq {
constexpr int D = 128;
constexpr int BN = 128;       // list entries per tile
constexpr int HB = 64;        // rows per half tile (a 64-token page)
constexpr int QROWS = 32;     // query vectors per KV head, at most
constexpr int NKT = 4;        // K tiles in tensor memory
constexpr int NS = 4;         // S^T buffers in tensor memory
constexpr int NPB = 4;        // P^T buffers (the tile j - 4 of a buffer is a softmax group's earlier tile)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_K = 0;                  // NKT K tiles of 64 columns (128 f16 per key)
constexpr uint32_t COL_S = NKT * 64;           // NS S^T buffers of NQ columns, then two O^T
}  // namespace dq

// KQ: 1 = INT8 codes, 2 = INT4 codes (two per byte), 3 = FP8 E4M3 codes.
template <int QVP, int KQ>
struct DqShape {
  // NGRP softmax groups of four warps; group g takes the tiles j with
  // j % NGRP == g (tensor-memory lane quarter = warp % 4).  Then four widen
  // warps (lane quarter = warp % 4), the gather warp, the QK warp and the PV
  // warp (two issuers, so that neither kind of MMA waits behind the other's
  // operands).
  static constexpr int NGRP = QVP <= 8 ? 3 : 2;
  static constexpr int NWARP = 4 * NGRP + 7;
  static constexpr int W_WID0 = 4 * NGRP, W_GATHER = 4 * NGRP + 4, W_MMA = 4 * NGRP + 5, W_PV = 4 * NGRP + 6;
  // registers per thread: a scheduler holds ceil(NWARP / 4) of the CTA's
  // warps in its 16,384-register file (19 warps: 96, 15 warps: 128)
  static constexpr int MAXREG = (16384 / (32 * ((NWARP + 3) / 4))) & ~7;
  static constexpr int NQ = QVP < 16 ? 16 : QVP;            // MMA N: query vectors, padded
  static constexpr int CB = KQ == 2 ? dq::D / 2 : dq::D;   // code bytes of one (row, head)
  static constexpr int CPR = CB / 16;                      // their 16-byte chunks
  static constexpr int WPC = 64 / CPR;                     // widened f16 pairs per chunk
  static constexpr int CODES = dq::BN * CB;                // one tile's K (or V) codes
  static constexpr int VATOM = dq::BN * 128;               // f16 V tile: 128 keys x 128 B per 64 dimensions
  // a stage holds the K codes at 0 and the V codes at VATOM, then the f16 V
  // tile (atom a at a * VATOM): each key's f16 row covers its own code rows
  // for 128-byte codes; for INT4 the widen warps agree before writing
  static constexpr int STAGE = 2 * VATOM;
  static constexpr int QATOM = NQ * 128;                   // Q^T: NQ rows x 128 B per 64 dimensions
  static constexpr int PATOM = NQ * 128;                   // P^T: NQ rows x 128 B per 64 keys
  static constexpr int PBUF = 2 * PATOM;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_P = ((2 * QATOM + 1023) / 1024) * 1024;
  static constexpr int OFF_C = OFF_P + dq::NPB * PBUF;
  // per group: agreement flags [2][4], tile maxima [2][4][QROWS], row sums
  // [4][QROWS], references [2][3][QROWS]; logit scales [QROWS]
  static constexpr int GRP_FLOATS = 8 + 8 * dq::QROWS + 4 * dq::QROWS + 6 * dq::QROWS + 4 * dq::QROWS;
  static constexpr int TAIL = 512 + 64 + NGRP * GRP_FLOATS * 4 + dq::QROWS * 4;
  static constexpr int BUDGET = 227 * 1024 - 1024 - OFF_C - TAIL;
  static constexpr int NC = BUDGET / STAGE < 8 ? BUDGET / STAGE : 8;   // code stages
  static constexpr int OFF_BAR = OFF_C + NC * STAGE;
  // q_full, code_full[NC], pv_done[NC], kc_read[NC], kt_full[NKT], s_full[NS],
  // p_full[NPB], agree[NGRP], drain
  static constexpr int NBAR = 1 + 3 * NC + dq::NKT + dq::NS + dq::NPB + NGRP + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // tmem base, abort flag, last-CTA flag, final copies [NGRP]
  static constexpr int OFF_GRP = OFF_MISC + 32;         // [NGRP] groups of GRP_FLOATS words
  static constexpr int G_FLAG = 0, G_RED = 8, G_SUM = 8 + 8 * dq::QROWS, G_REF = 8 + 12 * dq::QROWS,
                       G_WSUM = 8 + 18 * dq::QROWS;   // [4][QROWS] sums of the O weights
  static constexpr int OFF_QS = OFF_GRP + NGRP * GRP_FLOATS * 4;   // [QROWS] float
  static constexpr int SMEM_USED = OFF_QS + dq::QROWS * 4;
  static constexpr int SMEM = SMEM_USED + 1024;
  static constexpr uint32_t COL_O = dq::COL_S + dq::NS * NQ;   // O^T of group g: NQ columns at COL_O + g * NQ
  static_assert(COL_O + NGRP * NQ <= dq::TMEM_COLS, "tensor memory");
  // the QK of tile j is issued NGRP tiles before the PV of tile j: its S^T
  // buffer, last read by tile j - NS, must have had its PV waited for
  static_assert(dq::NS >= NGRP + 1 && NGRP <= 3, "S^T ring");
  // the QK of tile j waits for the P^T of tile j - NS (its S^T buffer's last
  // reader): that barrier's next phase, tile j - NS + NPB, needs the QK of j
  static_assert(dq::NPB >= dq::NS, "P^T ring");
  static_assert(dq::NKT == dq::NS, "a K tile is released by the QK that fills the S^T buffer of the same index");
  // a PV is waited for through its stage's barrier: by the next user of its
  // P^T buffer (NPB tiles on) and of its group's O^T (NGRP tiles on) before
  // the stage's next PV (NC tiles on) can complete
  static_assert(NC > dq::NPB && NC > NGRP, "pv_done ring");
  static_assert(NC >= 3, "code ring too shallow");
  static_assert(NBAR * 8 <= 512, "barrier area");
  static_assert(SMEM_USED - OFF_BAR <= TAIL, "tail area");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(OFF_P % 1024 == 0 && OFF_C % 1024 == 0 && STAGE % 1024 == 0 &&
                    CODES % 1024 == 0 && QATOM % 1024 == 0 && PATOM % 1024 == 0,
                "operand tiles and swizzled stages must be 1024-byte aligned");
  // split merge scratch (up to 2 * 256 * 32 + 64 floats) reuses the code ring
  static_assert(NC * STAGE >= (2 * kDecodeMaxSplits * dq::QROWS + 2 * dq::QROWS) * 4, "merge scratch");
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

// Widened f16 pairs of 16-byte code chunk `cw`: INT8 / FP8 chunks hold 16
// codes (8 words out), INT4 chunks 32 codes (16 words out); word t holds the
// chunk's elements 2t and 2t + 1.
template <int KQ>
__device__ __forceinline__ void widen_chunk(const uint4& cw, uint32_t* w) {
  if constexpr (KQ == 1) {
    const uint2 a = widen_i8x4(cw.x, false), b = widen_i8x4(cw.y, false);
    const uint2 c = widen_i8x4(cw.z, false), d = widen_i8x4(cw.w, false);
    w[0] = a.x; w[1] = a.y; w[2] = b.x; w[3] = b.y; w[4] = c.x; w[5] = c.y; w[6] = d.x; w[7] = d.y;
  } else if constexpr (KQ == 3) {
    const uint2 a = widen_e4m3x4(cw.x), b = widen_e4m3x4(cw.y), c = widen_e4m3x4(cw.z), d = widen_e4m3x4(cw.w);
    w[0] = a.x; w[1] = a.y; w[2] = b.x; w[3] = b.y; w[4] = c.x; w[5] = c.y; w[6] = d.x; w[7] = d.y;
  } else {
    const uint32_t v[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint4 h = widen_i4x8(v[t], false);
      w[4 * t] = h.x; w[4 * t + 1] = h.y; w[4 * t + 2] = h.z; w[4 * t + 3] = h.w;
    }
  }
}

// V codes widened with a constant offset: INT8 code c -> f16 1152 + c (the
// byte c + 128 under the f16 bits 0x6400), INT4 code c -> 1032 + c, both
// exact and one subtraction per pair cheaper than the exact widening; FP8
// codes are widened exactly (offset 0), and so are all codes for more than
// 16 query vectors (whose registers the weight sums would cost).  The offset
// is taken back out of O^T at the end with the sum of the O weights (Vᵀ Pᵀ
// holds offset * that sum).
template <int KQ, int QVP>
constexpr float v_offset() { return QVP > 16 ? 0.f : KQ == 1 ? 1152.f : KQ == 2 ? 1032.f : 0.f; }
template <int KQ, int QVP>
__device__ __forceinline__ void widen_chunk_off(const uint4& cw, uint32_t* w) {
  if constexpr (v_offset<KQ, QVP>() == 0.f) {
    widen_chunk<KQ>(cw, w);
  } else if constexpr (KQ == 1) {
    const uint32_t v[4] = {cw.x ^ 0x80808080u, cw.y ^ 0x80808080u, cw.z ^ 0x80808080u, cw.w ^ 0x80808080u};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      w[2 * t] = __byte_perm(v[t], 0x64646464u, 0x4140u);
      w[2 * t + 1] = __byte_perm(v[t], 0x64646464u, 0x4342u);
    }
  } else if constexpr (KQ == 2) {
    const uint32_t v[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t x = v[t] ^ 0x88888888u;
      const uint32_t even = x & 0x0F0F0F0Fu, odd = (x >> 4) & 0x0F0F0F0Fu;   // elements 0,2,4,6 / 1,3,5,7
      const uint32_t p0 = __byte_perm(even, odd, 0x5140u), p1 = __byte_perm(even, odd, 0x7362u);
      w[4 * t] = __byte_perm(p0, 0x64646464u, 0x4140u);
      w[4 * t + 1] = __byte_perm(p0, 0x64646464u, 0x4342u);
      w[4 * t + 2] = __byte_perm(p1, 0x64646464u, 0x4140u);
      w[4 * t + 3] = __byte_perm(p1, 0x64646464u, 0x4342u);
    }
  }
}

// Byte offset of 16-byte chunk ch of code row k within one matrix of a stage:
// 128-byte rows in the 128-byte swizzle (what the TMA writes), 64-byte rows plain.
template <int CB>
__device__ __forceinline__ uint32_t code_off(int k, int ch) {
  if constexpr (CB == 128) return (uint32_t)(k * 128 + ((ch ^ (k & 7)) << 4));
  return (uint32_t)(k * CB + ch * 16);
}

}  // namespace

// One CTA per SM (all 512 tensor-memory columns); the register cap keeps the
// warps that share a scheduler within its register file.
template <int QVP, int KQ>
__global__ void __maxnreg__((DqShape<QVP, KQ>::MAXREG))
    fa_rows_decode_tcq_kernel(const DqParams kp, const __grid_constant__ CUtensorMap tk,
                              const __grid_constant__ CUtensorMap tv) {
  using Sh = DqShape<QVP, KQ>;
  using namespace dq;
  constexpr int NC = Sh::NC, NQ = Sh::NQ, CB = Sh::CB, CPR = Sh::CPR;
  constexpr int NGRP = Sh::NGRP, W_WID0 = Sh::W_WID0, W_GATHER = Sh::W_GATHER, W_MMA = Sh::W_MMA, W_PV = Sh::W_PV;
  const DecodeParams& p = kp.a;
  const unsigned long long wait_ns = p.wait_ns;
  const float NEG_INF = __int_as_float(0xff800000);
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Sh::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* code_full = q_full + 1;
  // One commit per MMA group: pv_done[t % NC] completes with the PV of tile
  // t (its code stage, its P^T buffer and its group's O^T are free again),
  // s_full[j % NS] with the QK of tile j (its S^T is ready and its K tile,
  // j % NKT with NKT = NS, may be overwritten).
  uint64_t* pv_done = code_full + NC;
  uint64_t* kc_read = pv_done + NC;        // the widen warps hold the stage's K codes
  uint64_t* kt_full = kc_read + NC;
  uint64_t* s_full = kt_full + NKT;
  uint64_t* p_full = s_full + NS;
  uint64_t* agree = p_full + NPB;      // [NGRP]: a group's four warps
  uint64_t* drain = agree + NGRP;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + Sh::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Sh::OFF_MISC + 4);
  int* am_last = reinterpret_cast<int*>(sm + Sh::OFF_MISC + 8);
  int* final_copy = reinterpret_cast<int*>(sm + Sh::OFF_MISC + 16);   // [NGRP]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the KV heads vary fastest in the launch order, so the CTAs resident
  // together read the same pages' rows for neighbouring heads (1-2% faster
  // on ragged paged lists than splits fastest)
  const int split = blockIdx.y, g = blockIdx.x, s = blockIdx.z;
  const int G = p.G, QV = p.QV;
  const bool q_bf16 = p.q_bf16 != 0;
  int n_s = p.L;
  if (p.kv_len) n_s = min(max(__ldg(p.kv_len + s), 0), p.L);
  // splits past the sequence's last entry do nothing and are not merged; a
  // sequence that fits one split writes its result directly
  const int ns_unit = n_s > 0 && p.chunk > 0 ? (n_s + p.chunk - 1) / p.chunk : 1;
  if (split >= ns_unit) return;
  const bool single = ns_unit == 1;
  const int j0 = split * p.chunk;
  const int cnt = max(min(j0 + p.chunk, n_s) - j0, 0);
  const int T = (cnt + BN - 1) / BN;
  const int32_t* rows_g = p.kv_rows + (size_t)s * p.L + j0;
  const size_t unit = (size_t)s * p.Hkv + g;
  // List loads run tiles ahead of their use: each reads a clamped (always
  // valid) position and returns the raw entry, and the range test is applied
  // where the value is used, so no instruction waits on the load at issue.
  const int32_t* rows_safe = cnt > 0 ? rows_g : p.kv_rows;
  const int pos_max = cnt > 0 ? cnt - 1 : 0;
  auto entry_raw = [&](int pos) { return __ldg(rows_safe + min(pos, pos_max)); };
  auto live = [&](int pos, int e) { return pos < cnt ? e : -1; };
  auto valid = [&](int r) { return r >= 0 && (long long)r < p.R; };
  auto grp_words = [&](int grp) { return reinterpret_cast<float*>(sm + Sh::OFF_GRP) + grp * Sh::GRP_FLOATS; };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NC; ++i) {
      mbar_init(code_full + i, 32);   // one arrival per gather lane
      mbar_init(pv_done + i, 1);
      mbar_init(kc_read + i, 4);
    }
    for (int i = 0; i < NKT; ++i) {
      mbar_init(kt_full + i, 4);
    }
    for (int i = 0; i < NS; ++i) mbar_init(s_full + i, 1);
    for (int i = 0; i < NPB; ++i) {
      mbar_init(p_full + i, 4);
    }
    for (int i = 0; i < NGRP; ++i) {
      mbar_init(agree + i, 4);
    }
    mbar_init(drain, 2);   // one commit from each MMA issuer
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == W_MMA) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp < W_WID0 && (warp & 3) == 0) {   // each group's first reference copy: ml = mo = -inf, cw = 0
    float* refs = grp_words(warp >> 2) + Sh::G_REF;
    refs[lane] = NEG_INF;
    refs[QROWS + lane] = NEG_INF;
    refs[2 * QROWS + lane] = 0.f;
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
      // Q^T: query vector r -> row r of the swizzled tile (two 64-dimension
      // atoms), as f16 times 2^k_r; the row's logit scale becomes
      // qscale * 2^-k_r.  Rows QV..NQ-1 are zero.  16 lanes per row, 8
      // elements (one 16-byte chunk) each.
      const uint16_t* qg = static_cast<const uint16_t*>(p.q);
      float* qs = reinterpret_cast<float*>(sm + Sh::OFF_QS);
      for (int r = lane / 16; r < NQ; r += 2) {
        const int c = lane % 16;
        const bool live_r = r < QV;
        const int i = r / G, h = g * G + r % G;
        float v[8];
        float mx = 0.f;
        if (live_r) {
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
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (live_r) {
          o.x = pack2h(v[0] * up, v[1] * up, false);
          o.y = pack2h(v[2] * up, v[3] * up, false);
          o.z = pack2h(v[4] * up, v[5] * up, false);
          o.w = pack2h(v[6] * up, v[7] * up, false);
          if (c == 0) qs[r] = p.qscale * down;
        }
        *reinterpret_cast<uint4*>(sm + Sh::OFF_Q + (c >> 3) * Sh::QATOM + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = o;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    }
    // entries lane + 32t of the next two tiles, loaded two tiles ahead
    int nx[4], nx2[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      nx[t] = entry_raw(lane + 32 * t);
      nx2[t] = entry_raw(BN + lane + 32 * t);
    }
    unsigned tma_pend = 0, tma_par = 0;   // stages with a TMA load issued, and its phase parity
    for (int j = 0; j < T; ++j) {
      const int c = j % NC, u = j / NC;
      int r[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int e = live(j * BN + lane + 32 * t, nx[t]);
        r[t] = valid(e) ? e : -1;
        nx[t] = nx2[t];
        nx2[t] = entry_raw((j + 2) * BN + lane + 32 * t);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(pv_done + c, (u & 1) ^ 1, abort_flag, wait_ns))) break;
      unsigned char* Kc = sm + Sh::OFF_C + c * Sh::STAGE;
      unsigned char* Vc = Kc + Sh::VATOM;
      // half h holds entries 64h .. 64h + 63 (lane values r[2h], r[2h + 1]);
      // a half that is one contiguous pool run goes by TMA
      bool contig[2];
      int rb[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        rb[h] = __shfl_sync(0xffffffffu, r[2 * h], 0);
        contig[h] = kp.tma != 0 && __all_sync(0xffffffffu, r[2 * h] >= 0 && r[2 * h] == rb[h] + lane &&
                                                               r[2 * h + 1] >= 0 && r[2 * h + 1] == rb[h] + 32 + lane);
      }
      if (contig[0] || contig[1]) {
        if (lane == 0) {
          // the bytes the loads will bring, counted before any arrival
          mbar_expect_tx(code_full + c, (uint32_t)(((contig[0] ? 1 : 0) + (contig[1] ? 1 : 0)) * 2 * HB * CB));
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (!contig[h]) continue;
            tma_load_3d(Kc + h * HB * CB, &tk, 0, g, rb[h], code_full + c);
            tma_load_3d(Vc + h * HB * CB, &tv, 0, g, rb[h], code_full + c);
          }
        }
        tma_pend |= 1u << c;
        tma_par = (tma_par & ~(1u << c)) | ((unsigned)(u & 1) << c);
      }
      if (!(contig[0] && contig[1])) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (contig[h]) continue;
          // 64 rows x CPR chunks over 32 lanes: row e = f / CPR of the half
#pragma unroll
          for (int it = 0; it < HB * CPR / 32; ++it) {
            const int f = it * 32 + lane;
            const int e = f / CPR, q = f % CPR;   // e < 32 exactly for the first half of the iterations
            const int ra = __shfl_sync(0xffffffffu, r[2 * h], e & 31);
            const int rc = __shfl_sync(0xffffffffu, r[2 * h + 1], e & 31);
            const int row = e < 32 ? ra : rc;
            const bool okr = row >= 0;
            const size_t go = ((size_t)(okr ? row : 0) * p.Hkv + g) * CB + q * 16;
            const uint32_t so = code_off<CB>(h * HB + e, q);
            cp_async16(Kc + so, kb + go, okr);
            cp_async16(Vc + so, vb + go, okr);
          }
        }
        cp_async_mbar_arrive_noinc(code_full + c);
      } else {
        mbar_arrive(code_full + c);
      }
    }
    cp_async_wait_all();
    if (lane == 0 && *abort_flag) {   // no TMA load may still be writing when the CTA exits
      for (int c = 0; c < NC; ++c)
        if ((tma_pend >> c) & 1u) dq_wait_drain(code_full + c, (tma_par >> c) & 1u);
    }
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ QK issuer
    if (lane == 0 && T > 0) {
      // S^T = K Q^T: M = 128 keys (A in tensor memory), N = NQ, K = 128 dims;
      // the Q^T descriptor is built once and each MMA adds a constant offset
      const uint32_t id_qk = make_idesc_f16_ab(128, NQ, false, false, false);
      const uint64_t dQ = sdesc_sw128(smem_u32(sm + Sh::OFF_Q), 16, 1024);
      bool ok = mbar_wait(q_full, 0, abort_flag, wait_ns);
      tc_fence_after();
      for (int j = 0; ok && j < T; ++j) {
        // S^T buffer j % NS last held tile j - NS, whose softmax has read it
        // once that tile's P^T is written
        if (j >= NS) {
          const int t = j - NS;
          ok = mbar_wait(p_full + t % NPB, (t / NPB) & 1, abort_flag, wait_ns);
          if (!ok) break;
        }
        ok = mbar_wait(kt_full + j % NKT, (j / NKT) & 1, abort_flag, wait_ns);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ak = tbase + COL_K + (j % NKT) * 64;
        const uint32_t dS = tbase + COL_S + (j % NS) * NQ;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ts(dS, ak + kk * 8, sdesc_at(dQ, (kk >> 2) * Sh::QATOM + (kk & 3) * 32), id_qk, kk > 0);
        tc_commit(s_full + j % NS);
      }
      tc_commit(drain);
      dq_wait_drain(drain, 0);
    }
  } else if (warp == W_PV) {
    // ------------------------------------------------------------ PV issuer
    if (lane == 0 && T > 0) {
      // O^T += V^T P^T: M = 128 dims (A = the V tile read MN-major), N = NQ,
      // K = 16 keys each, into the O^T of the tile's group
      const uint32_t id_pv = make_idesc_f16_ab(128, NQ, false, true, false);
      const uint64_t dP = sdesc_sw128(smem_u32(sm + Sh::OFF_P), 16, 1024);
      const uint64_t dV = sdesc_sw128(smem_u32(sm + Sh::OFF_C), Sh::VATOM, 1024);
      bool ok = true;
      for (int t = 0; ok && t < T; ++t) {
        // the group arrives after its V tile and then its P^T are written
        ok = mbar_wait(p_full + t % NPB, (t / NPB) & 1, abort_flag, wait_ns);
        if (!ok) break;
        tc_fence_after();
        const int c = t % NC;
        const uint64_t av = sdesc_at(dV, c * Sh::STAGE);
        const uint64_t bp = sdesc_at(dP, (t % NPB) * Sh::PBUF);
        const uint32_t tO = tbase + Sh::COL_O + (t % NGRP) * NQ;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ss(tO, sdesc_at(av, kk * 2048), sdesc_at(bp, (kk >> 2) * Sh::PATOM + (kk & 3) * 32), id_pv,
                 t >= NGRP || kk > 0);
        tc_commit(pv_done + c);
      }
      tc_commit(drain);
      dq_wait_drain(drain, 0);
    }
  } else if (warp >= W_WID0) {
    // ------------------------------------------------------------ widen: one thread per key
    const int k = (warp - W_WID0) * 32 + lane;   // tensor-memory lane = key within the tile
    const uint32_t lane_sel = (uint32_t)((warp - W_WID0) * 32) << 16;
    constexpr int HC = CPR / 2;
    bool ok = true;
    for (int j = 0; ok && j < T; ++j) {
      const int c = j % NC, kt = j % NKT;
      const unsigned char* stg = sm + Sh::OFF_C + c * Sh::STAGE;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(code_full + c, (j / NC) & 1, abort_flag, wait_ns)))) break;
      // dimensions 0..63, then 64..127 (half the row's codes and 32 f16
      // pairs in registers at a time) into K tile kt
      uint4 ca[HC], cb[HC];
#pragma unroll
      for (int ch = 0; ch < HC; ++ch) {
        ca[ch] = *reinterpret_cast<const uint4*>(stg + code_off<CB>(k, ch));
        cb[ch] = *reinterpret_cast<const uint4*>(stg + code_off<CB>(k, HC + ch));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(kc_read + c);   // the f16 V tile may now cover the K codes
      // K tile kt last held tile j - NKT, whose QK completed with s_full[kt]
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(s_full + kt, ((j / NKT) & 1) ^ 1, abort_flag, wait_ns)))) break;
      tc_fence_after();
      {
        uint32_t w[32];
#pragma unroll
        for (int ch = 0; ch < HC; ++ch) widen_chunk<KQ>(ca[ch], w + ch * Sh::WPC);
        tmem_st32_nowait(tbase + lane_sel + COL_K + kt * 64, w);
      }
      {
        uint32_t w[32];
#pragma unroll
        for (int ch = 0; ch < HC; ++ch) widen_chunk<KQ>(cb[ch], w + ch * Sh::WPC);
        tmem_st32_nowait(tbase + lane_sel + COL_K + kt * 64 + 32, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(kt_full + kt);
    }
  } else {
    // ------------------------------------------------------------ softmax, one thread per key
    const int grp = warp >> 2, wq = warp & 3;
    const int k = wq * 32 + lane;
    const uint32_t lane_sel = (uint32_t)(wq * 32) << 16;
    float* gw = grp_words(grp);
    int* flags = reinterpret_cast<int*>(gw + Sh::G_FLAG);   // [2][4]
    float* red = gw + Sh::G_RED;                            // [2][4][QROWS] tile maxima: logit, logit + log2|s_v|
    float* rsum = gw + Sh::G_SUM;                           // [4][QROWS] final row sums
    // Two lazy references per query vector: ml for the row sum l = sum of
    // 2^(x - ml), and mo for the weights that go into O^T, 2^(x + log2|s_v| - mo)
    // * sign(s_v), so that every weight sits below 2^8 in magnitude and the
    // largest ones near the top of the f16 range whatever the V scales are.
    // cw = 2^(ml - mo) turns a row-sum term into an O weight: w = p * s_v * cw.
    // The three are the same for every thread of the group and live in shared
    // memory, two copies that alternate at each move (copy 0 starts at -inf,
    // -inf, 0); l is this thread's partial sum.
    float* refs = gw + Sh::G_REF;   // [2][3][QROWS]
    const float* qs = reinterpret_cast<const float*>(sm + Sh::OFF_QS);
    uint64_t* agr = agree + grp;
    const uint32_t colO = Sh::COL_O + grp * NQ;
    const bool causal = p.mask_kind == FA_MASK_CAUSAL;
    bool ok = true;
    int rp = 0;        // current reference copy
    uint32_t ph = 0;   // completed phases of the group's agreement barrier
    auto agree_wait = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(agr);
      const bool r = __all_sync(0xffffffffu, mbar_wait(agr, ph & 1, abort_flag, wait_ns));
      ++ph;
      return r;
    };
    // l: this thread's partial row sums; wsum: its partial sums of the f16 O
    // weights, which take the V offset back out of O^T at the end
    float l[QVP], wsum[QVP];
#pragma unroll
    for (int q = 0; q < QVP; ++q) {
      l[q] = 0.f;
      wsum[q] = 0.f;
    }
    // the logit scales qs[] are read from shared memory once q_full has completed
    if (T > grp && !__all_sync(0xffffffffu, mbar_wait(q_full, 0, abort_flag, wait_ns))) ok = false;
    // this group's tiles are grp, grp + NGRP, ...; this key's list entries three
    // of them ahead and its raw fp16 scales two ahead; a scale is read at row
    // 0 for a dead entry and zeroed at use
    auto tile_of = [&](int i) { return grp + NGRP * i; };
    auto scale_raw = [&](const uint16_t* sc, int r) {
      const int rr = valid(r) ? r : 0;
      return __ldg(sc + ((size_t)(rr >> 6) * p.Hkv + g) * kPage + (rr & 63));
    };
    const bool has_rows = p.R > 0;
    int e1 = entry_raw(tile_of(0) * BN + k), e2 = entry_raw(tile_of(1) * BN + k), e3 = entry_raw(tile_of(2) * BN + k);
    int r1 = live(tile_of(0) * BN + k, e1), r2 = live(tile_of(1) * BN + k, e2);
    uint16_t hk1 = 0, hv1 = 0, hk2 = 0, hv2 = 0;
    if (has_rows) {
      hk1 = scale_raw(p.k_scale, r1);
      hv1 = scale_raw(p.v_scale, r1);
      hk2 = scale_raw(p.k_scale, r2);
      hv2 = scale_raw(p.v_scale, r2);
    }
    for (int i = 0; ok && tile_of(i) < T; ++i) {
      const int j = tile_of(i);
      const int r = valid(r1) ? r1 : -1;
      const float sk = r >= 0 ? __half2float(__ushort_as_half(hk1)) : 0.f;
      const float sv = r >= 0 ? __half2float(__ushort_as_half(hv1)) : 0.f;
      r1 = r2;
      hk1 = hk2;
      hv1 = hv2;
      r2 = live(tile_of(i + 2) * BN + k, e3);   // loaded an iteration ago
      e3 = entry_raw(tile_of(i + 3) * BN + k);
      if (has_rows) {
        hk2 = scale_raw(p.k_scale, r2);
        hv2 = scale_raw(p.v_scale, r2);
      }
      const float lsv = __log2f(fabsf(sv));   // -inf for a zero scale
      const int pos = j0 + j * BN + k;        // list position of this key
      {
        // V of this tile, widened in place: this key's codes into registers;
        // once the widen warps hold the stage's K codes (and, for INT4, the
        // group's four warps hold their V codes: the f16 rows then cover
        // other keys' code rows), row k of the f16 tile: dimensions
        // 8t..8t+7 (words 4t..4t+3) in 16-byte chunk t % 8 of atom t / 8,
        // swizzled by the row; atom a holds dimensions 64a..64a+63, widened
        // from half a of the codes
        constexpr int HC = CPR / 2;
        const int c = j % NC;
        unsigned char* stg = sm + Sh::OFF_C + c * Sh::STAGE;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(code_full + c, (j / NC) & 1, abort_flag, wait_ns)))) break;
        uint4 ca[HC], cb[HC];
#pragma unroll
        for (int ch = 0; ch < HC; ++ch) {
          ca[ch] = *reinterpret_cast<const uint4*>(stg + Sh::VATOM + code_off<CB>(k, ch));
          cb[ch] = *reinterpret_cast<const uint4*>(stg + Sh::VATOM + code_off<CB>(k, HC + ch));
        }
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(kc_read + c, (j / NC) & 1, abort_flag, wait_ns)))) break;
        if constexpr (CB != 128) {
          if (!(ok = agree_wait())) break;
        }
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          uint32_t w[32];
#pragma unroll
          for (int ch = 0; ch < HC; ++ch) widen_chunk_off<KQ, QVP>(a ? cb[ch] : ca[ch], w + ch * Sh::WPC);
#pragma unroll
          for (int t = 0; t < 8; ++t)
            *reinterpret_cast<uint4*>(stg + a * Sh::VATOM + k * 128 + ((t ^ (k & 7)) << 4)) =
                make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
        }
        fence_proxy_async_smem();
      }
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(s_full + j % NS, (j / NS) & 1, abort_flag, wait_ns)))) break;
      tc_fence_after();
      uint32_t sr[32];
      if constexpr (NQ == 16) {
        tmem_ld16(tbase + lane_sel + COL_S + (j % NS) * NQ, *reinterpret_cast<uint32_t(*)[16]>(sr));
      } else {
        tmem_ld32(tbase + lane_sel + COL_S + (j % NS) * NQ, sr);
      }
      // logits in log2 units with the K scale folded in; masked: -inf
      float x[QVP];
      bool exceed = false;
      const float* ml = refs + rp * 3 * QROWS;
      const float* mo = ml + QROWS;
#pragma unroll
      for (int q = 0; q < QVP; ++q) {
        const int lim = causal ? n_s - p.Nq + q / G : n_s - 1;
        const bool vis = q < QV && valid(r) && pos <= lim;
        x[q] = vis ? __uint_as_float(sr[q]) * (qs[q] * sk) : NEG_INF;
        exceed = exceed || (x[q] > ml[q] + 8.f) || (x[q] + lsv > mo[q] + 8.f);
      }
      // do the group's four warps agree that no reference has to move?
      const bool wex = __any_sync(0xffffffffu, exceed);
      if (lane == 0) flags[(i & 1) * 4 + wq] = wex ? 1 : 0;
      if (!(ok = agree_wait())) break;
      const int* fl = flags + (i & 1) * 4;
      if (fl[0] | fl[1] | fl[2] | fl[3]) {
        // rare: each query vector's maxima over the tile's keys
#pragma unroll
        for (int q = 0; q < QVP; ++q) {
          float v = x[q], vo = x[q] + lsv;
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) {
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            vo = fmaxf(vo, __shfl_xor_sync(0xffffffffu, vo, o));
          }
          if (lane == 0) {
            red[wq * QROWS + q] = v;
            red[(4 + wq) * QROWS + q] = vo;
          }
        }
        if (!(ok = agree_wait())) break;
        // new references into the other copy (the group's first warp, a lane
        // per query vector); each thread scales its own partial sums and
        // keeps the O^T factors
        float* nref = refs + (rp ^ 1) * 3 * QROWS;
        float alpha[QVP];
        bool any_scale = false;
#pragma unroll
        for (int q = 0; q < QVP; ++q) {
          const float* rl = red + q;
          const float* ro = red + 4 * QROWS + q;
          const float mt = fmaxf(fmaxf(rl[0], rl[QROWS]), fmaxf(rl[2 * QROWS], rl[3 * QROWS]));
          const float mto = fmaxf(fmaxf(ro[0], ro[QROWS]), fmaxf(ro[2 * QROWS], ro[3 * QROWS]));
          float nl = ml[q], no = mo[q];
          if (mt > nl + 8.f) {
            l[q] *= nl == NEG_INF ? 0.f : fast_ex2(nl - mt);
            nl = mt;
          }
          alpha[q] = 1.f;
          if (mto > no + 8.f) {
            alpha[q] = no == NEG_INF ? 0.f : fast_ex2(no - mto);
            no = mto;
            any_scale = true;
          }
          if constexpr (v_offset<KQ, QVP>() != 0.f) wsum[q] *= alpha[q];
          if (wq == 0 && lane == q) {
            nref[q] = nl;
            nref[QROWS + q] = no;
            nref[2 * QROWS + q] = no == NEG_INF || nl == NEG_INF ? 0.f : fast_ex2(nl - no);
          }
        }
        // the new copy is complete, and every thread has read the reductions
        // and the old copy, before any thread goes on
        if (!(ok = agree_wait())) break;
        rp ^= 1;
        if (any_scale && i > 0) {
          // the group's O^T (this thread's lane = head dimension k) times
          // alpha per query vector, once the PV of its previous tile has
          // completed
          const int jp = j - NGRP;
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(pv_done + jp % NC, (jp / NC) & 1, abort_flag, wait_ns)))) break;
          tc_fence_after();
          uint32_t o[32];
          if constexpr (NQ == 16) {
            tmem_ld16(tbase + lane_sel + colO, *reinterpret_cast<uint32_t(*)[16]>(o));
          } else {
            tmem_ld32(tbase + lane_sel + colO, o);
          }
#pragma unroll
          for (int q = 0; q < QVP; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha[q]);
          if constexpr (NQ == 16) {
            tmem_st16(tbase + lane_sel + colO, *reinterpret_cast<uint32_t(*)[16]>(o));
          } else {
            tmem_st32(tbase + lane_sel + colO, o);
          }
        }
      }
      // P^T row q, key k: the O weight as f16, once the PV that last read this
      // buffer has completed
      const int pb = j % NPB;
      if (j >= NPB) {
        const int jp = j - NPB;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(pv_done + jp % NC, (jp / NC) & 1, abort_flag, wait_ns)))) break;
      }
      unsigned char* Pb = sm + Sh::OFF_P + pb * Sh::PBUF + (k >> 6) * Sh::PATOM + (k & 7) * 2;
      const float* mlc = refs + rp * 3 * QROWS;
      const float* cw = mlc + 2 * QROWS;
#pragma unroll
      for (int q = 0; q < QVP; ++q) {
        const float pq = x[q] == NEG_INF ? 0.f : fast_ex2(x[q] - mlc[q]);
        l[q] += pq;
        if (q < QV) {
          const __half wq = __float2half_rn(pq * (sv * cw[q]));
          if constexpr (v_offset<KQ, QVP>() != 0.f) wsum[q] += __half2float(wq);
          *reinterpret_cast<__half*>(Pb + q * 128 + ((((k & 63) >> 3) ^ (q & 7)) << 4)) = wq;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full + pb);
    }
    // ---- each group's row sums, then the first group (this thread's lane
    // now head dimension k) combines the groups' states and normalises
    if (ok && T > 0) ok = __all_sync(0xffffffffu, mbar_wait(drain, 0, abort_flag, wait_ns));
#pragma unroll
    for (int q = 0; q < QVP; ++q) {
      float v = l[q];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) rsum[wq * QROWS + q] = v;
      if constexpr (v_offset<KQ, QVP>() != 0.f) {
        float u = wsum[q];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
        if (lane == 0) gw[Sh::G_WSUM + wq * QROWS + q] = u;
      }
    }
    if (wq == 0 && lane == 0) final_copy[grp] = rp;
    named_barrier(1, NGRP * 4 * 32);   // the softmax warps; every wait before it is bounded
    tc_fence_after();
    if (grp == 0 && ok && !*abort_flag) {
      // per query vector: m = the largest group reference, L = the groups'
      // sums relative to m, and O^T relative to m (a group's O^T holds the
      // sum of 2^(x - mo) s_v v, so it enters times 2^(mo - m)); a group with
      // no tile has ml = mo = -inf and contributes nothing
      float mq[QVP], ov[QVP];
#pragma unroll
      for (int q = 0; q < QVP; ++q) {
        float m = NEG_INF;
        for (int gi = 0; gi < NGRP; ++gi) m = fmaxf(m, grp_words(gi)[Sh::G_REF + final_copy[gi] * 3 * QROWS + q]);
        mq[q] = m;
        ov[q] = 0.f;
      }
      for (int gi = 0; gi < NGRP && gi < T; ++gi) {
        const float* fr = grp_words(gi) + Sh::G_REF + final_copy[gi] * 3 * QROWS;
        uint32_t o[32];
        if constexpr (NQ == 16) {
          tmem_ld16(tbase + lane_sel + Sh::COL_O + gi * NQ, *reinterpret_cast<uint32_t(*)[16]>(o));
        } else {
          tmem_ld32(tbase + lane_sel + Sh::COL_O + gi * NQ, o);
        }
#pragma unroll
        for (int q = 0; q < QVP; ++q) {
          const float mo = fr[QROWS + q];
          if (mq[q] != NEG_INF && mo != NEG_INF) {
            // the V offset out: O^T holds sum w (offset + v) over the group's keys
            float oq = __uint_as_float(o[q]);
            if constexpr (v_offset<KQ, QVP>() != 0.f) {
              const float* ws = grp_words(gi) + Sh::G_WSUM + q;
              oq -= v_offset<KQ, QVP>() * (ws[0] + ws[QROWS] + ws[2 * QROWS] + ws[3 * QROWS]);
            }
            ov[q] += oq * exp2f(mo - mq[q]);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < QVP; ++q) {
        if (q >= QV) continue;
        const float m = mq[q];
        float L = 0.f;
        if (m != NEG_INF) {
          for (int gi = 0; gi < NGRP; ++gi) {
            const float ml = grp_words(gi)[Sh::G_REF + final_copy[gi] * 3 * QROWS + q];
            const float* sg = grp_words(gi) + Sh::G_SUM;
            if (ml != NEG_INF) L += (sg[q] + sg[QROWS + q] + sg[2 * QROWS + q] + sg[3 * QROWS + q]) * exp2f(ml - m);
          }
        }
        const int qi = q / G, h = g * G + q % G;
        const size_t oi = ((size_t)s * p.Nq + qi) * p.Hq + h;
        const size_t pi = (unit * p.nsplit + split) * QV + q;
        if (single) {
          store_out(p.out, oi * D + k, L > 0.f ? ov[q] / L : 0.f, p.out_dtype);
          if (k == 0 && p.lse) p.lse[oi] = L > 0.f ? (m + __log2f(L)) * kLn2 : NEG_INF;
        } else {
          if (m != NEG_INF) p.part_o[pi * D + k] = ov[q];
          if (k == 0) {
            p.part_ml[pi * 2] = m;
            p.part_ml[pi * 2 + 1] = L;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
  // An expired wait marks the workspace status word; the CTA still arrives
  // on its split counter (marked as aborted) so the counter ends at zero.
  const bool aborted = *abort_flag != 0;
  if (aborted && threadIdx.x == 0 && kp.err) atomicOr(kp.err, FA_WS_WAIT_EXPIRED);
  if (single) return;

  // ---- cross-split merge by the last CTA of this (slice, KV head)
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *am_last = split_arrive_last(p.counters + unit, ns_unit, aborted);
  __syncthreads();
  if (!*am_last) return;
  __threadfence();
  merge_splits<D>(p, unit, QV, QV, s, g, reinterpret_cast<float*>(sm + Sh::OFF_C), ns_unit);
  if (threadIdx.x == 0) p.counters[unit] = 0u;
}

// ---------------------------------------------------------------------------
// host side

namespace {

// Code pool [R][Hkv][CB bytes] as a 3-D byte tensor; box = CB bytes x one
// head x 64 rows, 128-byte swizzled for 128-byte rows (the widen threads each
// read a row), plain for INT4's 64-byte rows.
bool dq_map(CUtensorMap* m, const void* base, int CB, int Hkv, long long R) {
  const cuuint64_t dims[3] = {(cuuint64_t)CB, (cuuint64_t)Hkv, (cuuint64_t)R};
  const cuuint64_t strides[2] = {(cuuint64_t)CB, (cuuint64_t)CB * Hkv};
  const cuuint32_t box[3] = {(cuuint32_t)CB, 1, (cuuint32_t)dq::HB};
  return tmap_encode_3d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, dims, strides, box,
                        CB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int QVP, int KQ>
int dq_occupancy() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  const int c = cached[dev].load(std::memory_order_relaxed);
  if (c > 0) return c;
  using Sh = DqShape<QVP, KQ>;
  auto kern = fa_rows_decode_tcq_kernel<QVP, KQ>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Sh::NWARP * 32, Sh::SMEM) != cudaSuccess) return 0;
  n = n < 1 ? n : 1;   // 512 tensor-memory columns: one CTA per SM
  if (n > 0) cached[dev].store(n, std::memory_order_relaxed);
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
  kp.tma = a.R >= dq::HB && dq_map(&tk, a.k, Sh::CB, a.Hkv, a.R) && dq_map(&tv, a.v, Sh::CB, a.Hkv, a.R);
  dim3 grid(a.Hkv, a.nsplit, a.S);
  fa_rows_decode_tcq_kernel<QVP, KQ><<<grid, Sh::NWARP * 32, Sh::SMEM, st>>>(kp, tk, tv);
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

int decode_tcq_tile() { return dq::BN; }

cudaError_t decode_tcq_launch(const DecodeParams& a, int kind, unsigned int* err, cudaStream_t st) {
  if (kind == KV_I4) return dq_launch_q<2>(dq_pow2(a.QV), a, err, st);
  if (kind == KV_F8) return dq_launch_q<3>(dq_pow2(a.QV), a, err, st);
  return dq_launch_q<1>(dq_pow2(a.QV), a, err, st);
}

}  // namespace far
