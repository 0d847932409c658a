// Prefill over row-indexed lists on the 5th-generation tensor cores.
//
// The operation ("llama.cpp 0.9.0 inference boundaries", section 1): each
// query slice attends, exactly, to the pool rows its kv_rows list names; a
// negative entry is padding (mask -inf).  Causal prefill of a ubatch at the
// end of a prompt: query i of the slice's Nq sees list positions
// j <= n_s - Nq + i.
//
// One CTA owns two 128-row query tiles of one (slice, KV head).  A tile row
// is one (query position, query head) pair of that KV head's group, so the G
// heads sharing K/V ride in the MMA's M dimension and every K/V tile that is
// staged serves all of them.  Per 128-entry KV tile j:
//
//   producer warp  TMA (3-D tensor map over the pool [R][Hkv][D]) when the 128
//                  listed rows are one contiguous pool run, else a cp.async
//                  gather into the same 128-byte-swizzled layout (padding
//                  rows zero-filled); two K/V stages.
//   MMA warp       S_t = Q_t K_j^T into tensor memory (tcgen05.mma, both
//                  operands in shared memory), then O_t += P_t V_j with P_t read
//                  from tensor memory and V_j in shared memory (MN-major).
//   softmax warpgroup t (one thread per S row)
//                  loads S_t, masks, keeps a running max that is only moved
//                  when it grows by more than 2^8 (then O_t is rescaled in
//                  place), writes P_t = exp2(S*c - m) over S_t as 16-bit
//                  values (bf16: the pair P_hi = rn(P), P_lo = rn(P - P_hi),
//                  which keeps about 16 significant bits of P where one bf16
//                  rounding keeps 8; f16: rn(P) alone, 11 bits), and finally
//                  normalises O_t.
//
// Tensor memory: S0 | S1 | O0 | O1, 128 columns each (all 512).  The two
// warpgroups ping-pong: while one computes softmax, the tensor core runs the
// other tile's PV and next QK.
//
// Every wait is bounded in time; on expiry the CTA drains its own copies and
// MMAs, frees tensor memory, raises an error word and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <string.h>

#include <atomic>
#include <mutex>

#include "tc.cuh"
#include "tmap.cuh"

namespace far {

namespace pf {
constexpr int BM = 128;                    // query rows per tile = TMEM lanes
constexpr int BN = 128;                    // list entries per KV tile
constexpr int HD = 128;                    // head dim
constexpr int NST = 2;                     // K/V stages
constexpr int TILE = BM * HD * 2;          // one 128 x 128 16-bit tile: 32 KB
constexpr int HALF = TILE / 2;             // one 64-column half: 16 KB
// warps 0-3: softmax of Q tile 0, 4-7: Q tile 1, 8: producer (TMA, Q, gather),
// 9: MMA issuer, 10-11: gather producers
constexpr int NWARP = 12;
constexpr int W_PROD = 8, W_MMA = 9;
constexpr int NPROD = 3;                   // warps that gather K/V rows
// registers per thread: the block is launched with 384 x 168; the producer
// and MMA warpgroup keeps 64 and the two softmax warpgroups take 216 each
// (128 x 64 + 256 x 216 = 63,488 <= 64,512 = 384 x 168)
constexpr int REG_LAUNCH = 168, REG_LOW = 64, REG_HIGH = 216;
static_assert(128 * REG_LOW + 256 * REG_HIGH <= NWARP * 32 * REG_LAUNCH, "register split");
constexpr int OFF_Q = 0;
constexpr int OFF_K = 2 * TILE;
constexpr int OFF_V = OFF_K + NST * TILE;
constexpr int OFF_BAR = OFF_V + NST * TILE;
// q_full, k_full[NST], v_full[NST], kv_empty[NST], s_full[2], p_full[2], o_final[2], drain
constexpr int NBAR = 1 + 3 * NST + 2 + 2 + 2 + 1;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int OFF_IDX = OFF_MISC + 16;     // [NPROD][BN] list entries of the tile each gather warp is on
constexpr int SMEM_USED = OFF_IDX + NPROD * BN * 4;
constexpr int SMEM = SMEM_USED + 1024;     // slack for 1024-byte alignment
constexpr uint32_t COL_S = 0, COL_O = 256;
static_assert(SMEM <= 227 * 1024, "shared memory");
}  // namespace pf

struct PrefillKernelParams {
  PrefillParams a;
  int PT;            // query positions per tile (floor(128 / G))
  int tma_kv;        // 1 if the K/V tensor maps may be used
  int q_box;         // positions per Q TMA box
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Drain wait: bounded in time, ignores the abort flag.
__device__ __forceinline__ void mbar_wait_drain(uint64_t* b, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(b, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

// Visibility of column k of KV tile j for this thread's row: a valid entry
// (bit k of the tile's validity mask) within the causal limit.
__device__ __forceinline__ bool col_visible(int k, unsigned vb0, unsigned vb1, unsigned vb2, unsigned vb3, int jbase,
                                            int lim) {
  const unsigned vb = k < 32 ? vb0 : k < 64 ? vb1 : k < 96 ? vb2 : vb3;
  return ((vb >> (k & 31)) & 1u) && (jbase + k <= lim);
}

template <bool BF16>
__global__ void __launch_bounds__(pf::NWARP * 32, 1)
    fa_rows_prefill_kernel(const PrefillKernelParams kp, const __grid_constant__ CUtensorMap tq,
                           const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  using namespace pf;
  const PrefillParams& p = kp.a;
  const unsigned long long wait_ns = p.wait_ns;
  const float NEG_INF = __int_as_float(0xff800000);
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + NST;
  uint64_t* kv_empty = v_full + NST;
  uint64_t* s_full = kv_empty + NST;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_final = p_full + 2;
  uint64_t* drain = o_final + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int G = p.G, PT = kp.PT;
  const bool causal = p.mask_kind == FA_MASK_CAUSAL;
  int n_s = p.L;
  if (p.kv_len) n_s = min(max(__ldg(p.kv_len + s), 0), p.L);
  const int i0 = qb * 2 * PT;
  const int i_last = min(i0 + 2 * PT, p.Nq) - 1;
  const int lim_max = causal ? n_s - p.Nq + i_last : n_s - 1;
  const int n_vis = max(0, min(n_s, lim_max + 1));
  const int T = (n_vis + BN - 1) / BN;
  const int32_t* rows_g = p.kv_rows + (size_t)s * p.L;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NST; ++i) {
      // one arrival per lane of the three producer warps: asynchronous when
      // its gathered copies land, or plain next to the TMA byte count
      mbar_init(k_full + i, NPROD * 32);
      mbar_init(v_full + i, NPROD * 32);
      mbar_init(kv_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 128);
      mbar_init(o_final + i, 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == W_MMA) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;

  if (warp >= 8) {
    // the producer / MMA warpgroup gives registers to the softmax warpgroups
    regs_release<REG_LOW>();
    if (warp == W_PROD || warp >= 10) {
      // ------------------------------------------------------------ producers
      // Per KV tile: one TMA tile load per 64-column half and matrix when the
      // 128 listed rows are one contiguous pool run (warp 8, lane 0), else a
      // cp.async gather of the rows into the same 128-byte-swizzled layout
      // split over the three warps (padding rows zero-filled).  Every lane of
      // the three warps arrives once per stage and matrix; gather copies arrive
      // by themselves when they land, so no warp waits for its own loads.
      static_assert(NST == 2, "the producer tracks two stages in scalars");
      const int pi = warp == W_PROD ? 0 : warp - 9;   // 0, 1, 2
      const bool lead = pi == 0 && lane == 0;
      unsigned pend = 0;       // bit st: a TMA load into stage st may still be in flight
      int iss0 = 0, iss1 = 0;  // use count of the last TMA load into stage 0 / 1
      bool q_pending = false;
      if (lead && T > 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        mbar_arrive_expect_tx(q_full, 2u * 2u * (uint32_t)(kp.q_box * G) * 128u);
        for (int qt = 0; qt < 2; ++qt)
          for (int h = 0; h < 2; ++h)
            tma_load_3d(sm + OFF_Q + qt * TILE + h * HALF, &tq, h * 64, g * G, s * p.Nq + i0 + qt * PT, q_full);
        q_pending = true;
      }
      const char* kb = static_cast<const char*>(p.k);
      const char* vb = static_cast<const char*>(p.v);
      int32_t* idx = reinterpret_cast<int32_t*>(sm + OFF_IDX) + pi * BN;
      // this warp's row pairs of a gathered tile: [it_lo, it_hi) of the 64
      const int it_lo = pi * 22, it_hi = min(BN / 2, it_lo + 22);
      int nxt[4];
      #pragma unroll
      for (int t = 0; t < 4; ++t) nxt[t] = lane + 32 * t < n_s ? __ldg(rows_g + lane + 32 * t) : -1;
      for (int j = 0; j < T; ++j) {
        const int st = j % NST, u = j / NST;
        int rows[4];
        #pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int r = nxt[t];
          rows[t] = (r < 0 || (long long)r >= p.R) ? -1 : r;
          const int pos = (j + 1) * BN + lane + 32 * t;
          nxt[t] = pos < n_s ? __ldg(rows_g + pos) : -1;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(kv_empty + st, (u & 1) ^ 1, abort_flag, wait_ns))) break;
        if (lead) pend &= ~(1u << st);
        const int r0 = __shfl_sync(0xffffffffu, rows[0], 0);
        bool contig = true;
        #pragma unroll
        for (int t = 0; t < 4; ++t) contig = contig && rows[t] >= 0 && rows[t] == r0 + lane + 32 * t;
        contig = __all_sync(0xffffffffu, contig) && kp.tma_kv;
        unsigned char* Ks = sm + OFF_K + st * TILE;
        unsigned char* Vs = sm + OFF_V + st * TILE;
        if (contig) {
          if (lead) {
            mbar_arrive_expect_tx(k_full + st, TILE);
            tma_load_3d(Ks, &tk, 0, g, r0, k_full + st);
            tma_load_3d(Ks + HALF, &tk, 64, g, r0, k_full + st);
            mbar_arrive_expect_tx(v_full + st, TILE);
            tma_load_3d(Vs, &tv, 0, g, r0, v_full + st);
            tma_load_3d(Vs + HALF, &tv, 64, g, r0, v_full + st);
            pend |= 1u << st;
            if (st == 0) iss0 = u; else iss1 = u;
          } else {
            mbar_arrive(k_full + st);
            mbar_arrive(v_full + st);
          }
        } else {
          // this warp's entries of the tile, for any lane to read (the region
          // is this warp's alone: another warp may already be on the next tile)
          __syncwarp();
          #pragma unroll
          for (int t = 0; t < 4; ++t) idx[lane + 32 * t] = rows[t];
          __syncwarp();
          const int c = lane & 15;
          for (int it = it_lo; it < it_hi; ++it) {
            const int e = 2 * it + (lane >> 4);
            const int r = idx[e];
            const bool ok = r >= 0;
            const size_t go = ((size_t)(ok ? r : 0) * p.Hkv + g) * (HD * 2) + c * 16;
            const uint32_t so = (c >> 3) * HALF + e * 128 + (((c & 7) ^ (e & 7)) << 4);
            cp_async16(Ks + so, kb + go, ok);
            cp_async16(Vs + so, vb + go, ok);
          }
          cp_async_mbar_arrive_noinc(k_full + st);
          cp_async_mbar_arrive_noinc(v_full + st);
        }
      }
      cp_async_wait_all();
      // bulk copies still in flight must land before the CTA can exit
      if (lead) {
        if (q_pending && *abort_flag) mbar_wait_drain(q_full, 0);
        if ((pend & 1u) && *abort_flag) {
          mbar_wait_drain(k_full, iss0 & 1);
          mbar_wait_drain(v_full, iss0 & 1);
        }
        if ((pend & 2u) && *abort_flag) {
          mbar_wait_drain(k_full + 1, iss1 & 1);
          mbar_wait_drain(v_full + 1, iss1 & 1);
        }
      }
    } else if (warp == W_MMA) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0 && T > 0) {
        const uint32_t id_qk = make_idesc_f16(128, 128, BF16, false);
        const uint32_t id_pv = make_idesc_f16(128, 128, BF16, true);
        const uint32_t sQ = smem_u32(sm + OFF_Q), sK = smem_u32(sm + OFF_K), sV = smem_u32(sm + OFF_V);
        auto qk = [&](int qt, int st) {
          const uint32_t d = tbase + COL_S + qt * 128;
          #pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * HALF + (kk & 3) * 32;
            mma_ss(d, sdesc_sw128(sQ + qt * TILE + off, 16, 1024), sdesc_sw128(sK + st * TILE + off, 16, 1024), id_qk,
                   kk > 0);
          }
        };
        // P of keys 16kk..16kk+15 (8 packed columns): f16 at column 8kk; bf16
        // P_hi at 16kk and P_lo at 16kk + 8, each multiplied by the same V rows
        auto pv = [&](int qt, int st, bool acc) {
          const uint32_t d = tbase + COL_O + qt * 128;
          const uint32_t a = tbase + COL_S + qt * 128;
          #pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t vd = sdesc_sw128(sV + st * TILE + kk * 2048, HALF, 1024);
            if constexpr (BF16) {
              mma_ts(d, a + kk * 16, vd, id_pv, acc || kk > 0);
              mma_ts(d, a + kk * 16 + 8, vd, id_pv, 1);
            } else {
              mma_ts(d, a + kk * 8, vd, id_pv, acc || kk > 0);
            }
          }
        };
        bool ok = mbar_wait(q_full, 0, abort_flag, wait_ns);
        tc_fence_after();
        // Issue order per KV tile j: [PV_0(j-1), QK_0(j)], [PV_1(j-1), QK_1(j)],
        // so each tile's QK follows the PV that read its S buffer (the tensor
        // pipe runs one thread's MMAs in order).  Gathered stages were written
        // by cp.async copies that arrived on their barrier by themselves: a
        // proxy fence orders them before the tensor core's reads.
        for (int j = 0; ok && j < T; ++j) {
          const int st = j % NST, u = j / NST;
          if (!(ok = mbar_wait(k_full + st, u & 1, abort_flag, wait_ns))) break;
          tc_fence_after();
          fence_proxy_async_smem();
          for (int qt = 0; qt < 2 && ok; ++qt) {
            if (j > 0) {
              const int pj = j - 1, pst = pj % NST, pu = pj / NST;
              if (qt == 0) {
                if (!(ok = mbar_wait(v_full + pst, pu & 1, abort_flag, wait_ns))) break;
                fence_proxy_async_smem();
              }
              if (!(ok = mbar_wait(p_full + qt, pj & 1, abort_flag, wait_ns))) break;
              tc_fence_after();
              pv(qt, pst, pj > 0);
              if (qt == 1) tc_commit(kv_empty + pst);
            }
            qk(qt, st);
            tc_commit(s_full + qt);
          }
        }
        if (ok) {
          const int pj = T - 1, pst = pj % NST, pu = pj / NST;
          ok = mbar_wait(v_full + pst, pu & 1, abort_flag, wait_ns);
          fence_proxy_async_smem();
          for (int qt = 0; qt < 2 && ok; ++qt) {
            if (!(ok = mbar_wait(p_full + qt, pj & 1, abort_flag, wait_ns))) break;
            tc_fence_after();
            pv(qt, pst, pj > 0);
            tc_commit(o_final + qt);
          }
        }
        tc_commit(drain);
        mbar_wait_drain(drain, 0);
      }
    }
  } else {
    regs_acquire<REG_HIGH>();
    // ------------------------------------------------------------ softmax
    // One thread per S row; the whole 128-column row of a tile is loaded from
    // tensor memory once and kept in registers.
    const int qt = warp >> 2, quad = warp & 3;
    const int m = quad * 32 + lane;
    const int i = i0 + qt * PT + m / G;
    const int h = g * G + m % G;
    const bool row_ok = (m < PT * G) && (i < p.Nq);
    const int lim = causal ? n_s - p.Nq + i : n_s - 1;
    const uint32_t lane_sel = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tbase + lane_sel + COL_S + qt * 128;
    const uint32_t tO = tbase + lane_sel + COL_O + qt * 128;
    // c = scale * log2(e); a zero scale is replaced by the smallest normal
    // float, which leaves every logit 0 to within 2^-100 (so P = 1 exactly)
    // while a masked column's infinite fill still maps to -inf
    const float c = p.qscale == 0.f ? 1.17549435e-38f : p.qscale;
    // masked columns take the raw S value whose logit S*c is -inf
    const uint32_t fill = c > 0.f ? 0xff800000u : 0x7f800000u;
    float m_used = NEG_INF, l = 0.f;
    bool ok = true;
    // list entries of the next tile, loaded one tile ahead of their use
    int nxt[4];
    #pragma unroll
    for (int t = 0; t < 4; ++t) nxt[t] = lane + 32 * t < n_s ? __ldg(rows_g + lane + 32 * t) : -1;
    for (int j = 0; j < T; ++j) {
      unsigned vbits[4];
      #pragma unroll
      for (int t = 0; t < 4; ++t) {
        vbits[t] = __ballot_sync(0xffffffffu, nxt[t] >= 0 && (long long)nxt[t] < p.R);
        const int pos = (j + 1) * BN + lane + 32 * t;
        nxt[t] = pos < n_s ? __ldg(rows_g + pos) : -1;
      }
      const bool all_valid = (vbits[0] & vbits[1] & vbits[2] & vbits[3]) == 0xffffffffu;
      // warp-uniform: the tcgen05 loads below need every lane of the warp
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(s_full + qt, j & 1, abort_flag, wait_ns)))) break;
      tc_fence_after();
      uint32_t s0[32], s1[32], s2[32], s3[32];
      tmem_ld32_nowait(tS, s0);
      tmem_ld32_nowait(tS + 32, s1);
      tmem_ld32_nowait(tS + 64, s2);
      tmem_ld32_nowait(tS + 96, s3);
      tmem_wait_ld_tied(s0);
      tmem_wait_ld_tied(s1);
      tmem_wait_ld_tied(s2);
      tmem_wait_ld_tied(s3);
      if (!all_valid || j * BN + BN - 1 > lim) {
        #pragma unroll
        for (int k = 0; k < 32; ++k) {
          if (!col_visible(k, vbits[0], vbits[1], vbits[2], vbits[3], j * BN, lim)) s0[k] = fill;
          if (!col_visible(32 + k, vbits[0], vbits[1], vbits[2], vbits[3], j * BN, lim)) s1[k] = fill;
          if (!col_visible(64 + k, vbits[0], vbits[1], vbits[2], vbits[3], j * BN, lim)) s2[k] = fill;
          if (!col_visible(96 + k, vbits[0], vbits[1], vbits[2], vbits[3], j * BN, lim)) s3[k] = fill;
        }
      }
      // the row maximum of the logits S*c (c = scale*log2e), taken on raw S:
      // max(S)*c for c > 0, min(S)*c for c < 0 (masked columns hold the fill)
      float e[4];
      if (c > 0.f) {
        #pragma unroll
        for (int u = 0; u < 4; ++u) e[u] = __uint_as_float(fill);
        #pragma unroll
        for (int k = 0; k < 32; k += 2) {
          e[0] = fmaxf(e[0], fmaxf(__uint_as_float(s0[k]), __uint_as_float(s0[k + 1])));
          e[1] = fmaxf(e[1], fmaxf(__uint_as_float(s1[k]), __uint_as_float(s1[k + 1])));
          e[2] = fmaxf(e[2], fmaxf(__uint_as_float(s2[k]), __uint_as_float(s2[k + 1])));
          e[3] = fmaxf(e[3], fmaxf(__uint_as_float(s3[k]), __uint_as_float(s3[k + 1])));
        }
        e[0] = fmaxf(fmaxf(e[0], e[1]), fmaxf(e[2], e[3]));
      } else {
        #pragma unroll
        for (int u = 0; u < 4; ++u) e[u] = __uint_as_float(fill);
        #pragma unroll
        for (int k = 0; k < 32; k += 2) {
          e[0] = fminf(e[0], fminf(__uint_as_float(s0[k]), __uint_as_float(s0[k + 1])));
          e[1] = fminf(e[1], fminf(__uint_as_float(s1[k]), __uint_as_float(s1[k + 1])));
          e[2] = fminf(e[2], fminf(__uint_as_float(s2[k]), __uint_as_float(s2[k + 1])));
          e[3] = fminf(e[3], fminf(__uint_as_float(s3[k]), __uint_as_float(s3[k + 1])));
        }
        e[0] = fminf(fminf(e[0], e[1]), fminf(e[2], e[3]));
      }
      const float mx = (__float_as_uint(e[0]) == fill) ? NEG_INF : e[0] * c;
      const float m_new = fmaxf(m_used, mx);
      const bool need = m_new > m_used + 8.f;
      if (__any_sync(0xffffffffu, need)) {
        // rare: move the reference max and rescale O in place (PV of the
        // previous tile has completed: it was issued before this tile's QK)
        const float alpha = need ? fast_ex2(m_used - m_new) : 1.f;
        if (need) {
          l *= alpha;
          m_used = m_new;
        }
        if (j > 0) {
          #pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t r[32];
            tmem_ld32(tO + c4 * 32, r);
            #pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
            tmem_st32(tO + c4 * 32, r);
          }
        }
      }
      // P = exp2(S*c - m), written over S (all of which is in registers), 16
      // keys at a time: keys 16kk..16kk+15 as f16 P to columns 8kk..8kk+7, or
      // as bf16 P_hi = rn(P) to 16kk..16kk+7 and P_lo = rn(P - P_hi) to
      // 16kk+8..16kk+15; a masked column's fill gives exp2(-inf) = 0
      const float nmu = (m_used == NEG_INF) ? 0.f : -m_used;
      const float2 c2v = make_float2(c, c), nmu2 = make_float2(nmu, nmu);
      float2 sum[4];
      auto emit = [&](const uint32_t (&sv)[32], int q) {
        float2 acc = make_float2(0.f, 0.f);
        #pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t w[16];   // bf16: 8 P_hi words then 8 P_lo words; f16: 8 P words
          #pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int x = 16 * h + 2 * k;
            const float2 t =
                __ffma2_rn(make_float2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1])), c2v, nmu2);
            const float2 pr = make_float2(fast_ex2(t.x), fast_ex2(t.y));
            acc = __fadd2_rn(acc, pr);
            const uint32_t hi = pack2(pr.x, pr.y, BF16);
            w[k] = hi;
            if constexpr (BF16) {
              const float2 rem =
                  __fadd2_rn(pr, make_float2(-__uint_as_float(hi << 16), -__uint_as_float(hi & 0xffff0000u)));
              w[8 + k] = pack2(rem.x, rem.y, true);
            }
          }
          const int kk = 2 * q + h;
          if constexpr (BF16) {
            tmem_st16_nowait(tS + kk * 16, w);
          } else {
            tmem_st8_nowait(tS + kk * 8, w);
          }
        }
        sum[q] = acc;
      };
      emit(s0, 0);
      emit(s1, 1);
      emit(s2, 2);
      emit(s3, 3);
      tmem_wait_st();
      const float2 s01 = __fadd2_rn(sum[0], sum[1]), s23 = __fadd2_rn(sum[2], sum[3]);
      const float2 st = __fadd2_rn(s01, s23);
      l += st.x + st.y;
      tc_fence_before();
      mbar_arrive(p_full + qt);
    }
    if (ok && T > 0) ok = mbar_wait(o_final + qt, 0, abort_flag, wait_ns);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t orow = (((size_t)s * p.Nq + i) * p.Hq + h) * HD;
      #pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t r[32];
        if (T > 0) {
          tmem_ld32(tO + c4 * 32, r);
        } else {
          #pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = 0u;
        }
        if (row_ok) {
          if (p.out_dtype == FA_F32) {
            float4* o4 = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow + c4 * 32);
            #pragma unroll
            for (int k = 0; k < 8; ++k)
              o4[k] = make_float4(__uint_as_float(r[4 * k]) * inv, __uint_as_float(r[4 * k + 1]) * inv,
                                  __uint_as_float(r[4 * k + 2]) * inv, __uint_as_float(r[4 * k + 3]) * inv);
          } else {
            const bool ob = p.out_dtype == FA_BF16;
            uint4* o4 = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow + c4 * 32);
            #pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint4 w;
              w.x = pack2(__uint_as_float(r[8 * k + 0]) * inv, __uint_as_float(r[8 * k + 1]) * inv, ob);
              w.y = pack2(__uint_as_float(r[8 * k + 2]) * inv, __uint_as_float(r[8 * k + 3]) * inv, ob);
              w.z = pack2(__uint_as_float(r[8 * k + 4]) * inv, __uint_as_float(r[8 * k + 5]) * inv, ob);
              w.w = pack2(__uint_as_float(r[8 * k + 6]) * inv, __uint_as_float(r[8 * k + 7]) * inv, ob);
              o4[k] = w;
            }
          }
        }
      }
      if (row_ok && p.lse)
        p.lse[((size_t)s * p.Nq + i) * p.Hq + h] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : NEG_INF;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (threadIdx.x == 0 && *abort_flag && p.err) atomicOr(p.err, FA_WS_WAIT_EXPIRED);
}

// ---------------------------------------------------------------------------
// host side

namespace {

bool make_map_3d(CUtensorMap* m, const void* base, bool bf16, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0,
                 uint32_t b1, uint32_t b2) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {b0, b1, b2};
  return tmap_encode_3d(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, dims,
                        strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

bool prefill_supported(int D, int kind) { return D == pf::HD && (kind == KV_BF16 || kind == KV_F16); }

int prefill_positions_per_tile(int G) { return G >= 1 && G <= 128 ? 128 / G : 0; }

cudaError_t prefill_launch(const PrefillParams& a, cudaStream_t st) {
  PrefillKernelParams kp;
  kp.a = a;
  kp.PT = prefill_positions_per_tile(a.G);
  if (kp.PT == 0) return cudaErrorInvalidValue;
  const long long qrows = (long long)a.S * a.Nq;
  kp.q_box = (int)(qrows < kp.PT ? qrows : kp.PT);
  kp.tma_kv = a.R >= pf::BN;
  const bool bf16 = a.is_bf16 != 0;
  CUtensorMap tq, tk, tv;
  memset(&tq, 0, sizeof(tq));
  memset(&tk, 0, sizeof(tk));
  memset(&tv, 0, sizeof(tv));
  if (!make_map_3d(&tq, a.q, bf16, pf::HD, a.Hq, (uint64_t)qrows, 64, a.G, kp.q_box)) return cudaErrorInvalidValue;
  if (kp.tma_kv) {
    if (!make_map_3d(&tk, a.k, bf16, pf::HD, a.Hkv, a.R, 64, 1, pf::BN)) return cudaErrorInvalidValue;
    if (!make_map_3d(&tv, a.v, bf16, pf::HD, a.Hkv, a.R, 64, 1, pf::BN)) return cudaErrorInvalidValue;
  }
  auto kern = bf16 ? fa_rows_prefill_kernel<true> : fa_rows_prefill_kernel<false>;
  static std::atomic<int> attr_done[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  const int bit = bf16 ? 1 : 2;
  if (!(attr_done[dev].load(std::memory_order_relaxed) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pf::SMEM);
    if (e != cudaSuccess) return e;
    attr_done[dev].fetch_or(bit, std::memory_order_relaxed);
  }
  const int qb = (a.Nq + 2 * kp.PT - 1) / (2 * kp.PT);
  dim3 grid(qb, a.Hkv, a.S);
  kern<<<grid, pf::NWARP * 32, pf::SMEM, st>>>(kp, tq, tk, tv);
  return cudaGetLastError();
}

}  // namespace far
