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
constexpr int NWARP = 10;
constexpr int OFF_Q = 0;
constexpr int OFF_K = 2 * TILE;
constexpr int OFF_V = OFF_K + NST * TILE;
constexpr int OFF_BAR = OFF_V + NST * TILE;
// q_full, k_full[NST], v_full[NST], kv_empty[NST], s_full[2], p_full[2], o_final[2], drain
constexpr int NBAR = 1 + 3 * NST + 2 + 2 + 2 + 1;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int OFF_IDX = OFF_MISC + 16;
constexpr int SMEM_USED = OFF_IDX + BN * 4;
constexpr int SMEM = SMEM_USED + 1024;     // slack for 1024-byte alignment
constexpr uint32_t COL_S = 0, COL_O = 256;
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

// 64 raw fp32 columns of this thread's S row starting at column c0, two loads
// in flight per wait.
__device__ __forceinline__ void load_s64(uint32_t (&a)[32], uint32_t (&b)[32], uint32_t tS, int c0) {
  tmem_ld32_nowait(tS + c0, a);
  tmem_ld32_nowait(tS + c0 + 32, b);
  tmem_wait_ld_tied(a);
  tmem_wait_ld_tied(b);
}

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
  int32_t* idx_sm = reinterpret_cast<int32_t*>(sm + OFF_IDX);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int G = p.G, PT = kp.PT;
  const bool bf16 = p.is_bf16 != 0;
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
      mbar_init(k_full + i, 1);
      mbar_init(v_full + i, 1);
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
  if (warp == 9) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    static_assert(NST == 2, "the producer tracks two stages in scalars");
    unsigned pend = 0;       // bit st: a TMA load into stage st may still be in flight
    int iss0 = 0, iss1 = 0;  // use count of the last TMA load into stage 0 / 1
    bool q_pending = false;
    if (lane == 0 && T > 0) {
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
    for (int j = 0; j < T; ++j) {
      const int st = j % NST, u = j / NST;
      if (!__all_sync(0xffffffffu, mbar_wait(kv_empty + st, (u & 1) ^ 1, abort_flag, wait_ns))) break;
      pend &= ~(1u << st);
      int rows[4];
      bool contig = true;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int e = lane + 32 * t, pos = j * BN + e;
        int r = pos < n_s ? __ldg(rows_g + pos) : -1;
        if (r < 0 || (long long)r >= p.R) r = -1;
        rows[t] = r;
      }
      const int r0 = __shfl_sync(0xffffffffu, rows[0], 0);
#pragma unroll
      for (int t = 0; t < 4; ++t) contig = contig && rows[t] >= 0 && rows[t] == r0 + lane + 32 * t;
      contig = __all_sync(0xffffffffu, contig) && kp.tma_kv;
      unsigned char* Ks = sm + OFF_K + st * TILE;
      unsigned char* Vs = sm + OFF_V + st * TILE;
      if (contig) {
        if (lane == 0) {
          mbar_arrive_expect_tx(k_full + st, TILE);
          tma_load_3d(Ks, &tk, 0, g, r0, k_full + st);
          tma_load_3d(Ks + HALF, &tk, 64, g, r0, k_full + st);
          mbar_arrive_expect_tx(v_full + st, TILE);
          tma_load_3d(Vs, &tv, 0, g, r0, v_full + st);
          tma_load_3d(Vs + HALF, &tv, 64, g, r0, v_full + st);
        }
        pend |= 1u << st;
        if (st == 0) iss0 = u; else iss1 = u;
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) idx_sm[lane + 32 * t] = rows[t];
        __syncwarp();
        const int c = lane & 15;
#pragma unroll 4
        for (int it = 0; it < BN / 2; ++it) {
          const int e = 2 * it + (lane >> 4);
          const int r = idx_sm[e];
          const bool ok = r >= 0;
          const size_t go = ((size_t)(ok ? r : 0) * p.Hkv + g) * (HD * 2) + c * 16;
          const uint32_t so = (c >> 3) * HALF + e * 128 + (((c & 7) ^ (e & 7)) << 4);
          cp_async16(Ks + so, kb + go, ok);
          cp_async16(Vs + so, vb + go, ok);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(k_full + st);
          mbar_arrive(v_full + st);
        }
        __syncwarp();
      }
    }
    // bulk copies still in flight must land before the CTA can exit
    if (lane == 0) {
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
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      const uint32_t id_qk = make_idesc_f16(128, 128, bf16, false);
      const uint32_t id_pv = make_idesc_f16(128, 128, bf16, true);
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
      // P_hi at 64(kk/4) + 8(kk%4) and P_lo 32 columns after it, each
      // multiplied by the same V rows
      auto pv = [&](int qt, int st, bool acc) {
        const uint32_t d = tbase + COL_O + qt * 128;
        const uint32_t a = tbase + COL_S + qt * 128;
        if (bf16) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t vd = sdesc_sw128(sV + st * TILE + kk * 2048, HALF, 1024);
            const uint32_t ah = a + (kk >> 2) * 64 + (kk & 3) * 8;
            mma_ts(d, ah, vd, id_pv, acc || kk > 0);
            mma_ts(d, ah + 32, vd, id_pv, 1);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(d, a + kk * 8, sdesc_sw128(sV + st * TILE + kk * 2048, HALF, 1024), id_pv, acc || kk > 0);
        }
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, wait_ns);
      tc_fence_after();
      // Issue order per KV tile j: [PV_0(j-1), QK_0(j)], [PV_1(j-1), QK_1(j)],
      // so each tile's QK follows the PV that read its S buffer (the tensor
      // pipe runs one thread's MMAs in order).
      for (int j = 0; ok && j < T; ++j) {
        const int st = j % NST, u = j / NST;
        if (!(ok = mbar_wait(k_full + st, u & 1, abort_flag, wait_ns))) break;
        tc_fence_after();
        for (int qt = 0; qt < 2 && ok; ++qt) {
          if (j > 0) {
            const int pj = j - 1, pst = pj % NST, pu = pj / NST;
            if (qt == 0 && !(ok = mbar_wait(v_full + pst, pu & 1, abort_flag, wait_ns))) break;
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
  } else {
    // ------------------------------------------------------------ softmax
    const int qt = warp >> 2, quad = warp & 3;
    const int m = quad * 32 + lane;
    const int i = i0 + qt * PT + m / G;
    const int h = g * G + m % G;
    const bool row_ok = (m < PT * G) && (i < p.Nq);
    const int lim = causal ? n_s - p.Nq + i : n_s - 1;
    const uint32_t lane_sel = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tbase + lane_sel + COL_S + qt * 128;
    const uint32_t tO = tbase + lane_sel + COL_O + qt * 128;
    const float c = p.qscale;
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
      const bool need_mask = !all_valid || j * BN + BN - 1 > lim;
      // pass 1: the row maximum of the logits S*c (c = scale*log2e), taken on
      // raw S: max(S*c) = c*max(S) for c >= 0 and c*min(S) for c < 0
      const bool cpos = c >= 0.f;
      const float fill = cpos ? NEG_INF : -NEG_INF;
      float ext = fill;
#pragma unroll
      for (int c8 = 0; c8 < 2; ++c8) {
        uint32_t ra[32], rb[32];
        load_s64(ra, rb, tS, c8 * 64);
        if (need_mask) {
#pragma unroll
          for (int k = 0; k < 64; ++k) {
            float x = __uint_as_float(k < 32 ? ra[k] : rb[k - 32]);
            if (!col_visible(c8 * 64 + k, vbits[0], vbits[1], vbits[2], vbits[3], j * BN, lim)) x = fill;
            ext = cpos ? fmaxf(ext, x) : fminf(ext, x);
          }
        } else if (cpos) {
#pragma unroll
          for (int k = 0; k < 64; ++k) ext = fmaxf(ext, __uint_as_float(k < 32 ? ra[k] : rb[k - 32]));
        } else {
#pragma unroll
          for (int k = 0; k < 64; ++k) ext = fminf(ext, __uint_as_float(k < 32 ? ra[k] : rb[k - 32]));
        }
      }
      const float mx = (ext == fill) ? NEG_INF : ext * c;
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
      // pass 2: P = exp2(S*c - m) as 16-bit pairs, invisible columns 0.  The
      // 64 S columns of half hh are read before anything is written over
      // them: f16 P of those keys goes to columns 32hh..32hh+31; bf16 P_hi to
      // 64hh..64hh+31 and P_lo = rn(P - P_hi) to 64hh+32..64hh+63
      const float nmu = (m_used == NEG_INF) ? 0.f : -m_used;
      const float2 c2v = make_float2(c, c), nmu2 = make_float2(nmu, nmu);
      float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t pk[32], pl[32];
        uint32_t ra[32], rb[32];
        load_s64(ra, rb, tS, hh * 64);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c0 = hh * 64 + cc * 32;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float x0 = __uint_as_float(cc == 0 ? ra[2 * k] : rb[2 * k]);
            const float x1 = __uint_as_float(cc == 0 ? ra[2 * k + 1] : rb[2 * k + 1]);
            const float2 t = __ffma2_rn(make_float2(x0, x1), c2v, nmu2);
            float2 pr = make_float2(fast_ex2(t.x), fast_ex2(t.y));
            if (need_mask) {
              if (!col_visible(c0 + 2 * k, vbits[0], vbits[1], vbits[2], vbits[3], j * BN, lim)) pr.x = 0.f;
              if (!col_visible(c0 + 2 * k + 1, vbits[0], vbits[1], vbits[2], vbits[3], j * BN, lim)) pr.y = 0.f;
            }
            sum2 = __fadd2_rn(sum2, pr);
            const uint32_t hi = pack2(pr.x, pr.y, bf16);
            pk[cc * 16 + k] = hi;
            if (bf16) {
              const float2 rem =
                  __fadd2_rn(pr, make_float2(-__uint_as_float(hi << 16), -__uint_as_float(hi & 0xffff0000u)));
              pl[cc * 16 + k] = pack2(rem.x, rem.y, true);
            }
          }
        }
        if (bf16) {
          tmem_st32_nowait(tS + hh * 64, pk);
          tmem_st32_nowait(tS + hh * 64 + 32, pl);
          tmem_wait_st();
        } else {
          tmem_st32(tS + hh * 32, pk);
        }
      }
      const float sum = sum2.x + sum2.y;
      l += sum;
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
  if (warp == 9) {
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
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(fa_rows_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, pf::SMEM);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int qb = (a.Nq + 2 * kp.PT - 1) / (2 * kp.PT);
  dim3 grid(qb, a.Hkv, a.S);
  fa_rows_prefill_kernel<<<grid, pf::NWARP * 32, pf::SMEM, st>>>(kp, tq, tk, tv);
  return cudaGetLastError();
}

}  // namespace far
