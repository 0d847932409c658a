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
//   converters     (bf16 pools) two warps turn each landed V stage into f16
//                  in place, so that P can be one f16 value: exact for every
//                  bf16 value below 65536 in magnitude (one below 2^-14 becomes
//                  an f16 subnormal, within 2^-25 of it).  A scan of the
//                  listed V rows before the launch finds any finite value of
//                  65536 or more; the launch then keeps V in bf16 and P as the
//                  pair below.
//   MMA warp       S_t = Q_t K_j^T into tensor memory (tcgen05.mma, both
//                  operands in shared memory), then O_t += P_t V_j with P_t read
//                  from tensor memory and V_j in shared memory (MN-major).
//   softmax warpgroup t (one thread per S row)
//                  loads S_t, masks, keeps a running max that is only moved
//                  when it grows by more than 2^8 (then O_t is rescaled in
//                  place), writes P_t = exp2(S*c - m) over S_t as 16-bit
//                  values (f16 rn(P), 11 bits, whenever V is f16; else the bf16
//                  pair P_hi = rn(P), P_lo = rn(P - P_hi), which keeps about 16
//                  significant bits of P where one bf16 rounding keeps 8), and
//                  finally normalises O_t.
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
#include <type_traits>

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
// warps 0-15: softmax, four warpgroups (Q tile 0 columns 0-63, Q tile 0
// columns 64-127, then the same for Q tile 1); 16: producer (TMA, Q,
// gather); 17: MMA issuer; 18-19: gather producers
constexpr int NWARP = 20;
constexpr int NSMX = 16;                   // softmax warps
constexpr int W_PROD = 16, W_MMA = 17;
constexpr int NPROD = 3;                   // warps that gather K/V rows
// 640 threads: at most 96 registers each (enough for every role: a softmax
// thread holds 32 S values at a time)
constexpr int OFF_Q = 0;
constexpr int OFF_K = 2 * TILE;
constexpr int OFF_V = OFF_K + NST * TILE;
constexpr int OFF_BAR = OFF_V + NST * TILE;
// q_full, k_full[NST], v_full[NST], k_empty[NST], v_empty[NST], s_full[2],
// p_full[2], o_final[2], drain, pair[8] (the two warps that share a Q tile's rows),
// v_conv[NST] (bf16: the V stage is ready for the PV)
constexpr int NBAR = 1 + 4 * NST + 2 + 2 + 2 + 1 + 8 + NST;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int OFF_IDX = OFF_MISC + 16;     // [NPROD][BN] list entries of the tile each gather warp is on
// [2 tile parities][2 Q tiles][2 column halves][128 rows] partial row maxima, then
// [2 Q tiles][2 column halves][128 rows] partial row sums
constexpr int OFF_X = OFF_IDX + NPROD * BN * 4;
constexpr int SMEM_USED = OFF_X + (8 + 4) * BM * 4;
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

// MODE 0: f16 pool.  MODE 1: bf16 pool, V converted to f16 (f16 P).
// MODE 2: bf16 pool, V kept in bf16 (the P pair).  A bf16 launch runs modes
// 1 and 2; each CTA of the one the scan before the launch does not select
// exits at once.  Mode 2 is selected when a listed V value is beyond f16's
// range, or when more than a quarter of the KV tiles are gathered (not one
// contiguous pool run): there mode 1 has a single warp gathering K (two
// gather and convert V), mode 2 three warps on both.
template <int MODE>
__global__ void __launch_bounds__(pf::NWARP * 32, 1)
    fa_rows_prefill_kernel(const PrefillKernelParams kp, const __grid_constant__ CUtensorMap tq,
                           const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  using namespace pf;
  constexpr bool BF16 = MODE != 0, VF16 = MODE == 1, PAIR = MODE == 2;
  const PrefillParams& p = kp.a;
  if constexpr (BF16) {
    const bool pair_mode = __ldcg(p.err + 1) != 0u || 4u * __ldcg(p.err + 2) > __ldcg(p.err + 3);
    if (pair_mode != PAIR) return;
  }
  const unsigned long long wait_ns = p.wait_ns;
  const float NEG_INF = __int_as_float(0xff800000);
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + NST;
  uint64_t* k_empty = v_full + NST;    // a K stage is free once both Q tiles' QK have read it
  uint64_t* v_empty = k_empty + NST;   // a V stage once both PV have
  uint64_t* s_full = v_empty + NST;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_final = p_full + 2;
  uint64_t* drain = o_final + 2;
  uint64_t* pair = drain + 1;
  uint64_t* v_conv = pair + 8;
  // V converted to f16: one warp gathers and two convert
  constexpr int NPRODK = VF16 ? 1 : NPROD;
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
      mbar_init(k_full + i, NPRODK * 32);
      mbar_init(v_full + i, NPRODK * 32);
      mbar_init(v_conv + i, 2);
      mbar_init(k_empty + i, 1);
      mbar_init(v_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 256);   // both column halves of the tile's 128 rows
      mbar_init(o_final + i, 1);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < 8; ++i) mbar_init(pair + i, 64);
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

  if (warp >= NSMX) {
    if (VF16 && warp > W_MMA) {
      // ------------------------------------------------------------ V converters (bf16)
      // A V tile that is one contiguous pool run arrives by TMA (the
      // producer's); the converters gather the others themselves with
      // cp.async, one tile ahead, each thread later converting exactly the
      // 16-byte groups it copied.  Thread tid owns groups it * 64 + tid of the
      // tile: row e = group / 16, 16-byte column c = group % 16.
      const int ci = warp - W_MMA - 1;                    // 0, 1
      const int tid = ci * 32 + lane;                     // 0..63
      constexpr int NU = TILE / 16 / 64;                  // 16-byte groups per thread
      const char* vbase = static_cast<const char*>(p.v);
      int32_t* cidx = reinterpret_cast<int32_t*>(sm + OFF_IDX) + (1 + ci) * BN;   // this warp's copy of a tile's rows
      // the tile's 128 entries (lane + 32t), its contiguity as the producer decides it
      int nxt[4];
      #pragma unroll
      for (int t = 0; t < 4; ++t) nxt[t] = lane + 32 * t < n_s ? __ldg(rows_g + lane + 32 * t) : -1;
      auto next_tile = [&](int j, bool& contig) {
        int rows[4];
        #pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int r = nxt[t];
          rows[t] = (r < 0 || (long long)r >= p.R) ? -1 : r;
          const int pos = (j + 1) * BN + lane + 32 * t;
          nxt[t] = pos < n_s ? __ldg(rows_g + pos) : -1;
        }
        const int r0 = __shfl_sync(0xffffffffu, rows[0], 0);
        bool c = true;
        #pragma unroll
        for (int t = 0; t < 4; ++t) c = c && rows[t] >= 0 && rows[t] == r0 + lane + 32 * t;
        contig = __all_sync(0xffffffffu, c) && kp.tma_kv;
        if (!contig) {
          __syncwarp();
          #pragma unroll
          for (int t = 0; t < 4; ++t) cidx[lane + 32 * t] = rows[t];
          __syncwarp();
        }
      };
      // a gathered tile's copies into its stage, once both PVs of the tile two
      // back have read it; one commit group per tile (empty for a TMA tile)
      auto issue = [&](int j, bool contig) -> bool {
        if (!contig) {
          const int st = j % NST;
          if (!__all_sync(0xffffffffu, mbar_wait(v_empty + st, ((j / NST) & 1) ^ 1, abort_flag, wait_ns))) return false;
          unsigned char* dst = sm + OFF_V + st * TILE;
          #pragma unroll 4
          for (int it = 0; it < NU; ++it) {
            const int grp = it * 64 + tid, e = grp >> 4, c = grp & 15;
            const int r = cidx[e];
            const bool ok = r >= 0;
            const size_t go = ((size_t)(ok ? r : 0) * p.Hkv + g) * (HD * 2) + c * 16;
            cp_async16(dst + (c >> 3) * HALF + e * 128 + (((c & 7) ^ (e & 7)) << 4), vbase + go, ok);
          }
        }
        cp_async_commit();
        return true;
      };
      bool contig_cur = true, contig_nxt = true, ok = true;
      if (T > 0) {
        next_tile(0, contig_cur);
        ok = issue(0, contig_cur);
      }
      for (int j = 0; ok && j < T; ++j) {
        const int st = j % NST;
        const bool contig = contig_cur;
        if (j + 1 < T) {
          next_tile(j + 1, contig_nxt);
          if (!(ok = issue(j + 1, contig_nxt))) break;
          contig_cur = contig_nxt;
          cp_async_wait<1>();   // this thread's copies of tile j (not j + 1)
        } else {
          cp_async_wait<0>();
        }
        if (contig && !(ok = __all_sync(0xffffffffu, mbar_wait(v_full + st, (j / NST) & 1, abort_flag, wait_ns)))) break;
        uint4* vt = reinterpret_cast<uint4*>(sm + OFF_V + st * TILE);
        #pragma unroll 8
        for (int it = 0; it < NU; ++it) {
          const int grp = it * 64 + tid, e = grp >> 4, c = grp & 15;
          uint4* at = vt + ((c >> 3) * HALF + e * 128 + (((c & 7) ^ (e & 7)) << 4)) / 16;
          const uint4 w = *at;
          const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
          uint32_t o[4];
          #pragma unroll
          for (int t = 0; t < 4; ++t) {
            const __half2 hv = __floats2half2_rn(__uint_as_float(wv[t] << 16), __uint_as_float(wv[t] & 0xffff0000u));
            o[t] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          *at = make_uint4(o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(v_conv + st);
      }
      cp_async_wait_all();
    } else if (warp == W_PROD || warp > W_MMA) {
      // ------------------------------------------------------------ producers
      // Per KV tile: one TMA tile load per 64-column half and matrix when the
      // 128 listed rows are one contiguous pool run (warp 8, lane 0), else a
      // cp.async gather of the rows into the same 128-byte-swizzled layout
      // split over the three warps (padding rows zero-filled).  Every lane of
      // the three warps arrives once per stage and matrix; gather copies arrive
      // by themselves when they land, so no warp waits for its own loads.
      const int pi = warp == W_PROD ? 0 : warp - W_MMA;   // 0, 1, 2
      const bool lead = pi == 0 && lane == 0;
      // TMA loads that may still be in flight: bit st for K stage st, bit
      // NST + st for V stage st, with the phase parity of each
      unsigned tma_pend = 0, tma_par = 0;
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
      constexpr int PER = (BN / 2 + NPRODK - 1) / NPRODK;
      const int it_lo = pi * PER, it_hi = min(BN / 2, it_lo + PER);
      const int c = lane & 15;
      int nxt[4];
      #pragma unroll
      for (int t = 0; t < 4; ++t) nxt[t] = lane + 32 * t < n_s ? __ldg(rows_g + lane + 32 * t) : -1;
      // one matrix of tile j into stage st: TMA tile loads for a contiguous
      // run, else this warp's share of the gather; every lane arrives once
      auto load = [&](bool contig, int r0, unsigned char* dst, const void* tmap, const char* src, uint64_t* full,
                      int bit, int u) {
        if (contig) {
          if (lead) {
            mbar_arrive_expect_tx(full, TILE);
            tma_load_3d(dst, tmap, 0, g, r0, full);
            tma_load_3d(dst + HALF, tmap, 64, g, r0, full);
            tma_pend |= 1u << bit;
            tma_par = (tma_par & ~(1u << bit)) | ((unsigned)(u & 1) << bit);
          } else {
            mbar_arrive(full);
          }
        } else {
          for (int it = it_lo; it < it_hi; ++it) {
            const int e = 2 * it + (lane >> 4);
            const int r = idx[e];
            const bool ok = r >= 0;
            const size_t go = ((size_t)(ok ? r : 0) * p.Hkv + g) * (HD * 2) + c * 16;
            cp_async16(dst + (c >> 3) * HALF + e * 128 + (((c & 7) ^ (e & 7)) << 4), src + go, ok);
          }
          cp_async_mbar_arrive_noinc(full);
        }
      };
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
        const int r0 = __shfl_sync(0xffffffffu, rows[0], 0);
        bool contig = true;
        #pragma unroll
        for (int t = 0; t < 4; ++t) contig = contig && rows[t] >= 0 && rows[t] == r0 + lane + 32 * t;
        contig = __all_sync(0xffffffffu, contig) && kp.tma_kv;
        if (!contig) {
          // this warp's entries of the tile, for any lane to read (the region
          // is this warp's alone: another warp may already be on the next tile)
          __syncwarp();
          #pragma unroll
          for (int t = 0; t < 4; ++t) idx[lane + 32 * t] = rows[t];
          __syncwarp();
        }
        // K as soon as both QKs of tile j - NST have read the stage, V once both PVs have
        if (!__all_sync(0xffffffffu, mbar_wait(k_empty + st, (u & 1) ^ 1, abort_flag, wait_ns))) break;
        if (lead) tma_pend &= ~(1u << st);
        load(contig, r0, sm + OFF_K + st * TILE, &tk, kb, k_full + st, st, u);
        if (!__all_sync(0xffffffffu, mbar_wait(v_empty + st, (u & 1) ^ 1, abort_flag, wait_ns))) break;
        if (lead) tma_pend &= ~(1u << (NST + st));
        if (VF16 && !contig) {
          mbar_arrive(v_full + st);   // the converters gather this V tile
        } else {
          load(contig, r0, sm + OFF_V + st * TILE, &tv, vb, v_full + st, NST + st, u);
        }
      }
      cp_async_wait_all();
      // bulk copies still in flight must land before the CTA can exit
      if (lead && *abort_flag) {
        if (q_pending) mbar_wait_drain(q_full, 0);
        for (int st = 0; st < NST; ++st) {
          if ((tma_pend >> st) & 1u) mbar_wait_drain(k_full + st, (tma_par >> st) & 1u);
          if ((tma_pend >> (NST + st)) & 1u) mbar_wait_drain(v_full + st, (tma_par >> (NST + st)) & 1u);
        }
      }
    } else if (warp == W_MMA) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0 && T > 0) {
        const uint32_t id_qk = make_idesc_f16(128, 128, BF16, false);
        // PV: f16 P times an f16 V tile, or the bf16 pair times a bf16 tile
        const uint32_t id_pv = make_idesc_f16(128, 128, PAIR, true);
        // operand descriptors built once; each MMA only adds a constant offset
        static_assert(NST == 2, "two K and V stages");
        const uint64_t dQ0 = sdesc_sw128(smem_u32(sm + OFF_Q), 16, 1024), dQ1 = sdesc_at(dQ0, TILE);
        const uint64_t dK0 = sdesc_sw128(smem_u32(sm + OFF_K), 16, 1024), dK1 = sdesc_at(dK0, TILE);
        const uint64_t dV0 = sdesc_sw128(smem_u32(sm + OFF_V), HALF, 1024), dV1 = sdesc_at(dV0, TILE);
        auto qk = [&](int qt, int st) {
          const uint32_t d = tbase + COL_S + qt * 128;
          const uint64_t a = qt ? dQ1 : dQ0, b = st ? dK1 : dK0;
          #pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * HALF + (kk & 3) * 32;
            mma_ss(d, sdesc_at(a, off), sdesc_at(b, off), id_qk, kk > 0);
          }
        };
        // P of keys 16kk..16kk+15 (8 packed columns) at column 16kk; bf16
        // also P_lo at 16kk + 8, multiplied by the same V rows
        auto pv = [&](int qt, int st, bool acc) {
          const uint32_t d = tbase + COL_O + qt * 128;
          const uint32_t a = tbase + COL_S + qt * 128;
          const uint64_t vb = st ? dV1 : dV0;
          #pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t vd = sdesc_at(vb, kk * 2048);
            if constexpr (PAIR) {
              mma_ts(d, a + kk * 16, vd, id_pv, acc || kk > 0);
              mma_ts(d, a + kk * 16 + 8, vd, id_pv, 1);
            } else {
              mma_ts(d, a + kk * 16, vd, id_pv, acc || kk > 0);
            }
          }
        };
        bool ok = mbar_wait(q_full, 0, abort_flag, wait_ns);
        tc_fence_after();
        // Event-driven issue, per Q tile: QK(j), then once its P is written
        // PV(j), then QK(j + 1) into the same S buffer (the tensor pipe runs
        // one thread's MMAs in order, so a QK never overwrites P before the
        // PV that reads it).  Each operation goes out as soon as its own
        // inputs are ready; neither Q tile waits for the other, and no PV
        // waits for the next tile's loads.  A K stage is released after both
        // Q tiles' QK of its tile, a V stage after both PV.  Gathered stages
        // were written by cp.async copies that arrived on their barrier by
        // themselves: a proxy fence orders them before the tensor core's reads.
        int nq[2] = {0, 0}, np[2] = {0, 0};   // next tile of QK / PV per Q tile
        unsigned long long t_idle = 0;
        while (ok && (np[0] < T || np[1] < T)) {
          bool progressed = false;
          #pragma unroll
          for (int qt = 0; qt < 2; ++qt) {
            if (np[qt] < nq[qt]) {
              const int j = np[qt], st = j % NST;
              if (mbar_test_wait(p_full + qt, j & 1) && mbar_test_wait((VF16 ? v_conv : v_full) + st, (j / NST) & 1)) {
                tc_fence_after();
                fence_proxy_async_smem();
                pv(qt, st, j > 0);
                ++np[qt];
                if (np[qt ^ 1] > j) tc_commit(v_empty + st);   // both PV of tile j issued
                if (np[qt] == T) tc_commit(o_final + qt);
                progressed = true;
              }
            }
            if (nq[qt] < T && nq[qt] == np[qt]) {
              const int j = nq[qt], st = j % NST;
              if (mbar_test_wait(k_full + st, (j / NST) & 1)) {
                tc_fence_after();
                fence_proxy_async_smem();
                qk(qt, st);
                tc_commit(s_full + qt);
                ++nq[qt];
                if (nq[qt ^ 1] > j) tc_commit(k_empty + st);   // both QK of tile j issued
                progressed = true;
              }
            }
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
        mbar_wait_drain(drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Two threads per S row, one per 64-column half: each reads its half of
    // a tile's row from tensor memory in two 32-column chunks, once for the
    // row maximum and once to turn it into P.  The two halves' maxima are
    // exchanged through shared memory and a bounded pair barrier, so both
    // apply the same reference max; their sums are added at the end.
    const int qt = warp >> 3, half = (warp >> 2) & 1, quad = warp & 3;
    const int m = quad * 32 + lane;
    const int i = i0 + qt * PT + m / G;
    const int h = g * G + m % G;
    const bool row_ok = (m < PT * G) && (i < p.Nq);
    const int lim = causal ? n_s - p.Nq + i : n_s - 1;
    const uint32_t lane_sel = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tbase + lane_sel + COL_S + qt * 128 + half * 64;
    const uint32_t tO = tbase + lane_sel + COL_O + qt * 128 + half * 64;
    uint64_t* pb = pair + qt * 4 + quad;
    float* xmax = reinterpret_cast<float*>(sm + OFF_X);                   // [parity][qt][half][row]
    float* xsum = xmax + 8 * BM;                                            // [qt][half][row]
    // c = scale * log2(e); a zero scale is replaced by the smallest normal
    // float, which leaves every logit 0 to within 2^-100 (so P = 1 exactly)
    // while a masked column's infinite fill still maps to -inf
    const float c = p.qscale == 0.f ? 1.17549435e-38f : p.qscale;
    // masked columns take the raw S value whose logit S*c is -inf
    const uint32_t fill = c > 0.f ? 0xff800000u : 0x7f800000u;
    float m_used = NEG_INF, l = 0.f;
    bool ok = true;
    // this half's list entries of the next tile, loaded one tile ahead
    const int c0 = half * 64;   // first column of this half within a tile
    int nxt[2];
    #pragma unroll
    for (int t = 0; t < 2; ++t) nxt[t] = c0 + lane + 32 * t < n_s ? __ldg(rows_g + c0 + lane + 32 * t) : -1;
    int j = 0;
    for (; j < T; ++j) {
      unsigned vbits[2];
      #pragma unroll
      for (int t = 0; t < 2; ++t) {
        vbits[t] = __ballot_sync(0xffffffffu, nxt[t] >= 0 && (long long)nxt[t] < p.R);
        const int pos = (j + 1) * BN + c0 + lane + 32 * t;
        nxt[t] = pos < n_s ? __ldg(rows_g + pos) : -1;
      }
      // warp-uniform: the tcgen05 loads below need every lane of the warp
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(s_full + qt, j & 1, abort_flag, wait_ns)))) break;
      tc_fence_after();
      // pass 1: the row extreme of raw S over this half, 32 columns at a time
      // (max for c > 0, min for c < 0: the logits' max is then ext * c;
      // masked columns take the fill)
      const int jb = j * BN + c0;   // list position of this half's first column
      const bool masked = (vbits[0] & vbits[1]) != 0xffffffffu || jb + 63 > lim;
      auto load_chunk = [&](uint32_t (&sv)[32], int q) {
        tmem_ld32(tS + q * 32, sv);
        if (masked) {
          #pragma unroll
          for (int k = 0; k < 32; ++k)
            if (!(((vbits[q] >> k) & 1u) && jb + 32 * q + k <= lim)) sv[k] = fill;
        }
      };
      float e[4];
      #pragma unroll
      for (int u = 0; u < 4; ++u) e[u] = __uint_as_float(fill);
      #pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t sv[32];
        load_chunk(sv, q);
        if (c > 0.f) {
          #pragma unroll
          for (int k = 0; k < 32; k += 8) {
            e[0] = fmaxf(e[0], fmaxf(__uint_as_float(sv[k]), __uint_as_float(sv[k + 1])));
            e[1] = fmaxf(e[1], fmaxf(__uint_as_float(sv[k + 2]), __uint_as_float(sv[k + 3])));
            e[2] = fmaxf(e[2], fmaxf(__uint_as_float(sv[k + 4]), __uint_as_float(sv[k + 5])));
            e[3] = fmaxf(e[3], fmaxf(__uint_as_float(sv[k + 6]), __uint_as_float(sv[k + 7])));
          }
        } else {
          #pragma unroll
          for (int k = 0; k < 32; k += 8) {
            e[0] = fminf(e[0], fminf(__uint_as_float(sv[k]), __uint_as_float(sv[k + 1])));
            e[1] = fminf(e[1], fminf(__uint_as_float(sv[k + 2]), __uint_as_float(sv[k + 3])));
            e[2] = fminf(e[2], fminf(__uint_as_float(sv[k + 4]), __uint_as_float(sv[k + 5])));
            e[3] = fminf(e[3], fminf(__uint_as_float(sv[k + 6]), __uint_as_float(sv[k + 7])));
          }
        }
      }
      e[0] = c > 0.f ? fmaxf(fmaxf(e[0], e[1]), fmaxf(e[2], e[3])) : fminf(fminf(e[0], e[1]), fminf(e[2], e[3]));
      // exchange with the other half of the row (slots alternate with the
      // tile parity, so the partner's next write cannot overwrite a slot this
      // thread has yet to read)
      float* xm = xmax + (((j & 1) * 2 + qt) * 2) * BM + m;
      xm[half * BM] = e[0];
      mbar_arrive(pb);
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(pb, j & 1, abort_flag, wait_ns)))) break;
      const float eo = xm[(half ^ 1) * BM];
      const float ext = c > 0.f ? fmaxf(e[0], eo) : fminf(e[0], eo);
      const float mx = (__float_as_uint(ext) == fill) ? NEG_INF : ext * c;
      const float m_new = fmaxf(m_used, mx);
      const bool need = m_new > m_used + 8.f;
      if (__any_sync(0xffffffffu, need)) {
        // rare: move the reference max and rescale this half of O in place
        // (PV of the previous tile has completed: it was issued before this
        // tile's QK)
        const float alpha = need ? fast_ex2(m_used - m_new) : 1.f;
        if (need) {
          l *= alpha;
          m_used = m_new;
        }
        if (j > 0) {
          #pragma unroll
          for (int c4 = 0; c4 < 2; ++c4) {
            uint32_t r[32];
            tmem_ld32(tO + c4 * 32, r);
            #pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
            tmem_st32(tO + c4 * 32, r);
          }
        }
      }
      // P = exp2(S*c - m), written over this half's S columns (in registers),
      // 16 keys at a time: keys 16kk..16kk+15 of the tile to columns
      // 16kk..16kk+7 (f16 P, or bf16 P_hi = rn(P)) and, for bf16, P_lo =
      // rn(P - P_hi) to 16kk+8..16kk+15; a masked column's fill gives 0
      const float nmu = (m_used == NEG_INF) ? 0.f : -m_used;
      const float2 c2v = make_float2(c, c), nmu2 = make_float2(nmu, nmu);
      float2 acc = make_float2(0.f, 0.f);
      auto emit = [&](const uint32_t (&sv)[32], int q, auto pair_t) {
        constexpr bool PAIR = decltype(pair_t)::value;
        #pragma unroll
        for (int o = 0; o < 4; ++o) {
          // keys 8o..8o+7 of this 32-column chunk: 4 P (or P_hi) words, and
          // for bf16 4 P_lo words
          uint32_t w[8];
          #pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int x = 8 * o + 2 * k;
            const float2 t =
                __ffma2_rn(make_float2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1])), c2v, nmu2);
            const float2 pr = make_float2(fast_ex2(t.x), fast_ex2(t.y));
            acc = __fadd2_rn(acc, pr);
            const uint32_t hi = pack2(pr.x, pr.y, PAIR);
            w[k] = hi;
            if constexpr (PAIR) {
              const float2 rem =
                  __fadd2_rn(pr, make_float2(-__uint_as_float(hi << 16), -__uint_as_float(hi & 0xffff0000u)));
              w[4 + k] = pack2(rem.x, rem.y, true);
            }
          }
          // this half's keys 32q + 8o ..: column 16 * (2q + o/2) + 4 * (o%2) of its 64
          const uint32_t col = tS + (2 * q + (o >> 1)) * 16 + (o & 1) * 4;
          tmem_st4_nowait(col, w[0], w[1], w[2], w[3]);
          if constexpr (PAIR) tmem_st4_nowait(col + 8, w[4], w[5], w[6], w[7]);
        }
      };
      // pass 2: the same 32-column chunks read again, turned into P
      #pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t sv[32];
        load_chunk(sv, q);
        emit(sv, q, std::integral_constant<bool, PAIR>{});
      }
      tmem_wait_st();
      l += acc.x + acc.y;
      tc_fence_before();
      mbar_arrive(p_full + qt);
    }
    if (ok && T > 0) ok = mbar_wait(o_final + qt, 0, abort_flag, wait_ns);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok) {
      // the row sum is the two halves' sums (added in the same order by both)
      xsum[(qt * 2 + half) * BM + m] = l;
      mbar_arrive(pb);
      ok = __all_sync(0xffffffffu, mbar_wait(pb, T & 1, abort_flag, wait_ns));
    }
    if (ok) {
      const float lt = xsum[(qt * 2) * BM + m] + xsum[(qt * 2 + 1) * BM + m];
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const size_t orow = (((size_t)s * p.Nq + i) * p.Hq + h) * HD + half * 64;
      #pragma unroll
      for (int c4 = 0; c4 < 2; ++c4) {
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
              uint4 wv;
              wv.x = pack2(__uint_as_float(r[8 * k + 0]) * inv, __uint_as_float(r[8 * k + 1]) * inv, ob);
              wv.y = pack2(__uint_as_float(r[8 * k + 2]) * inv, __uint_as_float(r[8 * k + 3]) * inv, ob);
              wv.z = pack2(__uint_as_float(r[8 * k + 4]) * inv, __uint_as_float(r[8 * k + 5]) * inv, ob);
              wv.w = pack2(__uint_as_float(r[8 * k + 6]) * inv, __uint_as_float(r[8 * k + 7]) * inv, ob);
              o4[k] = wv;
            }
          }
        }
      }
      if (row_ok && half == 0 && p.lse)
        p.lse[((size_t)s * p.Nq + i) * p.Hq + h] = lt > 0.f ? (m_used + __log2f(lt)) * kLn2 : NEG_INF;
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

// Before a bf16 launch, per 128-entry KV tile of every slice (one warp each):
// is any listed V value finite and of magnitude 65536 or more (not an f16
// value: word 1 of the status block gets 1), and is the tile not one
// contiguous pool run (word 2 counts those, word 3 all tiles)?  The words
// were zeroed before.
__global__ void __launch_bounds__(256) prefill_v_scan_kernel(const uint4* v, const int32_t* kv_rows,
                                                             const int32_t* kv_len, int S, int L, long long R,
                                                             int row_chunks, int tma_kv, unsigned int* words) {
  const int lane = threadIdx.x & 31;
  const int tiles_per = (L + pf::BN - 1) / pf::BN;
  const long long nw = (long long)gridDim.x * (blockDim.x >> 5);
  uint32_t bad = 0;
  unsigned gathered = 0, tiles = 0;
  for (long long e = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); e < (long long)S * tiles_per;
       e += nw) {
    const int s = (int)(e / tiles_per), j0 = (int)(e % tiles_per) * pf::BN;
    const int n_s = kv_len ? min(max(__ldg(kv_len + s), 0), L) : L;
    if (j0 >= n_s) continue;
    const int32_t* rows = kv_rows + (size_t)s * L + j0;
    int r[4];
    #pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int pos = lane + 32 * t;
      const int x = j0 + pos < n_s ? __ldg(rows + pos) : -1;
      r[t] = (x < 0 || (long long)x >= R) ? -1 : x;
    }
    const int r0 = __shfl_sync(0xffffffffu, r[0], 0);
    bool contig = tma_kv != 0;
    #pragma unroll
    for (int t = 0; t < 4; ++t) contig = contig && r[t] >= 0 && r[t] == r0 + lane + 32 * t;
    contig = __all_sync(0xffffffffu, contig);
    ++tiles;
    if (!contig) ++gathered;
    // the tile's rows four at a time, each read by the whole warp (coalesced),
    // all of a group's loads issued before any is examined
    #pragma unroll
    for (int t = 0; t < 4; ++t) {
      for (int rr = 0; rr < 32; rr += 4) {
        int row[4];
        #pragma unroll
        for (int u = 0; u < 4; ++u) row[u] = __shfl_sync(0xffffffffu, r[t], rr + u);
        for (int i0 = 0; i0 < row_chunks; i0 += 64) {
          uint4 w[4][2];
          #pragma unroll
          for (int u = 0; u < 4; ++u) {
            #pragma unroll
            for (int c = 0; c < 2; ++c) {
              const int i = i0 + lane + 32 * c;
              w[u][c] = (row[u] >= 0 && i < row_chunks) ? __ldg(v + (size_t)row[u] * row_chunks + i)
                                                        : make_uint4(0u, 0u, 0u, 0u);
            }
          }
          #pragma unroll
          for (int u = 0; u < 4; ++u) {
            #pragma unroll
            for (int c = 0; c < 2; ++c) {
              const uint32_t wv[4] = {w[u][c].x, w[u][c].y, w[u][c].z, w[u][c].w};
              #pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint32_t a = wv[q] & 0x7fff7fffu;
                bad |= __vcmpgeu2(a, 0x47804780u) & __vcmpltu2(a, 0x7f807f80u);
              }
            }
          }
        }
      }
    }
  }
  if (__any_sync(0xffffffffu, bad != 0) && lane == 0) atomicOr(words, 1u);
  if (lane == 0 && tiles) {
    atomicAdd(words + 1, gathered);
    atomicAdd(words + 2, tiles);
  }
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
  if (bf16) {
    // words 1-3 of the status block: the scan's V-range flag, gathered and all KV tiles
    cudaError_t e = cudaMemsetAsync(a.err + 1, 0, 3 * sizeof(unsigned int), st);
    if (e != cudaSuccess) return e;
    const long long tiles = (long long)a.S * ((a.L + pf::BN - 1) / pf::BN);   // one warp each, 8 per block
    const long long blocks = (tiles + 7) / 8;
    if (blocks > 0) {
      prefill_v_scan_kernel<<<(unsigned)(blocks < 152 * 16 ? blocks : 152 * 16), 256, 0, st>>>(
          static_cast<const uint4*>(a.v), a.kv_rows, a.kv_len, a.S, a.L, a.R, a.Hkv * pf::HD / 8, kp.tma_kv,
          a.err + 1);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  static std::atomic<int> attr_done[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  const int qb = (a.Nq + 2 * kp.PT - 1) / (2 * kp.PT);
  dim3 grid(qb, a.Hkv, a.S);
  // f16: mode 0; bf16: modes 1 (V to f16) and 2 (V kept), one of which exits
  const int modes[2] = {bf16 ? 1 : 0, bf16 ? 2 : -1};
  for (int mode : modes) {
    if (mode < 0) continue;
    auto kern = mode == 0 ? fa_rows_prefill_kernel<0> : mode == 1 ? fa_rows_prefill_kernel<1> : fa_rows_prefill_kernel<2>;
    const int bit = 1 << mode;
    if (!(attr_done[dev].load(std::memory_order_relaxed) & bit)) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pf::SMEM);
      if (e != cudaSuccess) return e;
      attr_done[dev].fetch_or(bit, std::memory_order_relaxed);
    }
    kern<<<grid, pf::NWARP * 32, pf::SMEM, st>>>(kp, tq, tk, tv);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace far
