// The C ABI of fa_rows: argument checks, the decode split planner and the
// launches.  Nothing here allocates device memory or synchronises.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "decode.cuh"
#include "fa_internal.cuh"

namespace {

thread_local char g_err[512] = "";

// Limit of a pipeline wait in the tensor-core kernels launched from now on
// (0 = the kernels' default).
std::atomic<unsigned long long> g_wait_limit_ns{0};

unsigned long long wait_limit() {
  const unsigned long long v = g_wait_limit_ns.load(std::memory_order_relaxed);
  return v ? v : 1000ull * 1000ull * 1000ull;
}

fa_status fail(fa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

fa_status cuda_fail(cudaError_t e, const char* where) {
  return fail(FA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// SM count of the current device, cached per device once it has been read
// (a failed query is not cached: it answers 1 and is retried next time).
int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
  cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

int kv_kind(fa_dtype d) {
  switch (d) {
    case FA_BF16: return far::KV_BF16;
    case FA_F16: return far::KV_F16;
    case FA_I8: return far::KV_I8;
    case FA_I4: return far::KV_I4;
    case FA_F8E4M3: return far::KV_F8;
    default: return -1;
  }
}

// Shape and pointer checks shared by decode and prefill.
fa_status check_common(const fa_rows_args* a) {
  if (!a) return fail(FA_ERR_INVALID_ARG, "args is NULL");
  if (a->S < 0 || a->Nq < 0 || a->Hq <= 0 || a->Hkv <= 0 || a->D <= 0 || a->list_len < 0 || a->n_pool_rows < 0)
    return fail(FA_ERR_INVALID_ARG, "negative or zero size (S=%d Nq=%d Hq=%d Hkv=%d D=%d L=%d R=%lld)", a->S, a->Nq,
                a->Hq, a->Hkv, a->D, a->list_len, (long long)a->n_pool_rows);
  if (a->Hq % a->Hkv != 0) return fail(FA_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", a->Hq, a->Hkv);
  if (a->n_pool_rows > 0x7fffffffLL) return fail(FA_ERR_UNSUPPORTED, "pool rows must fit int32 row indices");
  if (a->q_dtype != FA_F16 && a->q_dtype != FA_BF16) return fail(FA_ERR_UNSUPPORTED, "q dtype must be f16 or bf16");
  if (kv_kind(a->kv_dtype) < 0) return fail(FA_ERR_UNSUPPORTED, "kv dtype must be f16, bf16, i8, i4 or f8e4m3");
  const bool quant = a->kv_dtype == FA_I8 || a->kv_dtype == FA_I4 || a->kv_dtype == FA_F8E4M3;
  if (!quant && a->kv_dtype != a->q_dtype) return fail(FA_ERR_UNSUPPORTED, "a 16-bit pool must have the dtype of q");
  if (a->out_dtype != FA_F32 && a->out_dtype != FA_BF16 && a->out_dtype != FA_F16)
    return fail(FA_ERR_UNSUPPORTED, "out dtype must be f32, bf16 or f16");
  if (a->mask_kind != FA_MASK_NONE && a->mask_kind != FA_MASK_DENSE && a->mask_kind != FA_MASK_CAUSAL)
    return fail(FA_ERR_INVALID_ARG, "unknown mask kind %d", (int)a->mask_kind);
  const bool empty = (long long)a->S * a->Nq == 0;
  if (empty) return FA_OK;
  if (!a->q || !a->out) return fail(FA_ERR_INVALID_ARG, "q and out are required");
  if (a->list_len > 0 && (!a->kv_rows || !a->k || !a->v)) return fail(FA_ERR_INVALID_ARG, "kv_rows, k and v are required");
  if (a->mask_kind == FA_MASK_DENSE && a->list_len > 0 && !a->mask)
    return fail(FA_ERR_INVALID_ARG, "FA_MASK_DENSE needs a mask");
  if (quant) {
    if (a->list_len > 0 && (!a->k_scale || !a->v_scale))
      return fail(FA_ERR_INVALID_ARG, "a quantised pool needs k_scale and v_scale");
    if (a->n_pool_rows % far::kPage != 0) return fail(FA_ERR_UNSUPPORTED, "quantised pool rows must be a multiple of 64");
    if (a->kv_dtype == FA_I4 && a->D % 32 != 0) return fail(FA_ERR_UNSUPPORTED, "INT4 pools need D % 32 == 0");
    if (!aligned(a->k_scale, 4) || !aligned(a->v_scale, 4)) return fail(FA_ERR_INVALID_ARG, "scales must be 4-byte aligned");
  }
  if (!aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->q, 4) || !aligned(a->out, 4) || !aligned(a->kv_rows, 4) ||
      !aligned(a->lse, 4) || !aligned(a->mask, 4) || !aligned(a->kv_len, 4))
    return fail(FA_ERR_INVALID_ARG, "k and v need 16-byte alignment, other tensors 4-byte alignment");
  return FA_OK;
}

struct DecodePlan {
  bool tc = false;   // tensor-core kernel (either of the two below)
  bool tcq = false;  // the quantised-pool tensor-core kernel
  int qvp = 0, rows = 0, chunk = 0, nsplit = 0;
  bool merge_kernel = false;   // the splits are merged by a kernel of their own
  size_t ws = 0;     // workspace bytes: status block, counters, partials
  size_t off_cnt = 0, off_ml = 0, off_o = 0;
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kMaxSplits = far::kDecodeMaxSplits;
constexpr long long kMergeMaxFloats = 32 * 1024;   // partial floats one merging CTA reads, at most (16-bit tc decode)

// The prefill workspace is the status block alone.
constexpr size_t kPrefillWorkspace = far::kStatusBytes;

// Chooses the kernel and how the list is cut into per-CTA chunks.  Cost model
// in units of rows streamed by one CTA: waves * (chunk + fixed cost) + merge
// cost, where ragged lists (n_valid_hint given) are costed by their mean
// length and the all-padding CTAs they leave add a small per-CTA cost.
fa_status plan_decode(const fa_rows_args* a, DecodePlan* pl) {
  const int G = a->Hq / a->Hkv;
  const long long qv = (long long)a->Nq * G;
  if (qv > 32) return fail(FA_ERR_UNSUPPORTED, "decode packs Nq*Hq/Hkv <= 32 query vectors per KV head (got %lld)", qv);
  const int qvp = next_pow2((int)(qv < 1 ? 1 : qv));
  const int kind = kv_kind(a->kv_dtype);
  const int qv1 = (int)(qv < 1 ? 1 : qv);
  pl->tcq = far::decode_tcq_supported(a->D, kind, qv1, a->mask_kind) && aligned(a->q, 16);
  pl->tc = pl->tcq || (far::decode_tc_supported(a->D, kind, qv1, a->mask_kind) && aligned(a->q, 16) &&
                       a->n_pool_rows * a->Hkv < 0x7fffffffLL);  // TMA rows are int32 coordinates r * Hkv + g
  if ((kind == far::KV_I4 || kind == far::KV_F8) && !pl->tcq)
    return fail(FA_ERR_UNSUPPORTED, "INT4/FP8 pools are decoded at D=128 with at most 32 query vectors and no dense mask");
  pl->qvp = qvp;
  pl->rows = pl->tc ? (int)qv : qvp;
  int align = 0, chunk_max = 0;
  if (pl->tc) {
    align = pl->tcq ? far::decode_tcq_tile() : far::decode_tc_tile();
    chunk_max = 1 << 30;
  } else {
    far::DecodeConfig cfg;
    bool built = false;
    if (kind == far::KV_BF16) built = far::decode_config_bf16(a->D, qvp, &cfg);
    if (kind == far::KV_F16) built = far::decode_config_f16(a->D, qvp, &cfg);
    if (kind == far::KV_I8) built = far::decode_config_i8(a->D, qvp, &cfg);
    if (!built)
      return fail(FA_ERR_UNSUPPORTED,
                  "decode is built for D in {64,128,256} with (Nq*G padded) * D <= 2048; got D=%d, %d query vectors",
                  a->D, qvp);
    align = cfg.rt * far::kDecodeWarps;
    chunk_max = far::kDecodeChunkMax;
  }
  const int L = a->list_len;
  pl->off_cnt = far::kStatusBytes;
  if ((long long)a->S * a->Nq == 0 || L == 0) {
    pl->chunk = 0;
    pl->nsplit = 1;
    pl->ws = far::kStatusBytes;
    return FA_OK;
  }
  int occ = 0;
  if (pl->tcq) occ = far::decode_tcq_occupancy(kind, qv1);
  else if (pl->tc) occ = far::decode_tc_occupancy(a->D, kind, qv1);
  else if (kind == far::KV_BF16) occ = far::decode_occupancy_bf16(a->D, qvp);
  else if (kind == far::KV_F16) occ = far::decode_occupancy_f16(a->D, qvp);
  else if (kind == far::KV_I8) occ = far::decode_occupancy_i8(a->D, qvp);
  if (occ <= 0) return fail(FA_ERR_CUDA, "decode kernel cannot be resident (no device, or shared memory too small)");
  const long long slots = (long long)sm_count() * occ;
  const long long units = (long long)a->S * a->Hkv;
  const bool ragged = a->n_valid_hint > 0;
  const double lavg = ragged ? (double)a->n_valid_hint / a->S : (double)L;
  // fixed cost of a CTA (start-up, pipeline fill, merge), in streamed rows
  const double c_cta = pl->tc ? 256.0 : 64.0, c_split = 2.0, c_empty = 16.0, c_cta_q = 1536.0;
  const int ns_lo = (int)((L + chunk_max - 1) / chunk_max);
  if (ns_lo > kMaxSplits)
    return fail(FA_ERR_UNSUPPORTED, "list length %d needs more than %d splits of %d entries", L, kMaxSplits, chunk_max);
  const int ns_hi = (L + align - 1) / align;
  double best = 1e300;
  int best_ns = ns_lo;
  for (int ns = ns_lo; ns <= ns_hi && ns <= kMaxSplits; ++ns) {
    const long long chunk = round_up((L + ns - 1) / ns, align);
    if (chunk > chunk_max) continue;
    const long long ns_eff = (L + chunk - 1) / chunk;
    double cost;
    if (!ragged) {
      const long long waves = (units * ns_eff + slots - 1) / slots;
      cost = waves * (chunk + c_cta) + c_split * ns_eff;
    } else if (pl->tcq) {
      // ragged lists on the quantised kernel (one CTA per SM): CTAs of unequal
      // length backfill the SMs, so the step is about the rows streamed plus
      // a fixed cost per busy CTA (pipeline fill, the groups' combine, the
      // split's share of the merge: about 1 536 rows), over the slots, plus
      // half a chunk of tail; a slice of the mean length holds lavg / chunk
      // + 1/2 busy splits on average over a spread of lengths.  Measured on
      // 32 paged sequences of 1k-128k tokens: 6 / 8 / 10 / 13 splits 0.467 /
      // 0.450 / 0.441 / 0.455 ms, the wave model's 31 splits 0.534.
      const double per_unit = lavg / (double)chunk + 0.5;
      const double busy = units * per_unit;
      cost = (units * lavg + busy * c_cta_q) / slots + 0.5 * (double)chunk +
             c_empty * ((double)units * ns_eff - busy) / slots + c_split * per_unit;
    } else {
      const double per_unit = ceil(lavg / (double)chunk);
      const long long busy = (long long)(units * per_unit);
      const long long waves = (busy + slots - 1) / slots;
      cost = waves * (chunk + c_cta) + c_empty * (double)(units * ns_eff - busy) / slots + c_split * per_unit;
    }
    if (cost < best - 1e-9) {
      best = cost;
      best_ns = (int)ns_eff;
    }
  }
  // The last CTA of a (slice, KV head) merges ns * QV * D fp32 partials with
  // a few loads in flight per thread; when each CTA streams only a few tiles,
  // past 32K floats (128 KB) those load rounds outlast what a finer split
  // saves (measured on the sparse D 256 workload: 32 splits of one tile
  // 13.7 us in the kernel, 16 splits of two tiles 11.4 us).
  if (pl->tc && !pl->tcq) {
    const long long per_split = qv1 * (long long)a->D;
    while (best_ns > 1 && best_ns * per_split > kMergeMaxFloats &&
           round_up((L + best_ns - 1) / best_ns, align) <= 4 * (size_t)align) {
      const int ns_next = (best_ns + 1) / 2;
      const long long chunk_next = round_up((L + ns_next - 1) / ns_next, align);
      if (chunk_next > chunk_max) break;
      best_ns = (int)((L + chunk_next - 1) / chunk_next);
    }
  }
  pl->chunk = (int)round_up((L + best_ns - 1) / best_ns, align);
  pl->nsplit = (L + pl->chunk - 1) / pl->chunk;
  // A latency-bound 16-bit decode (one wave of CTAs, each streaming at most
  // four tiles) merges its splits in a kernel of its own: its last CTA per
  // (slice, KV head) would merge on the critical path with six warps, one
  // L2 round trip per 16 splits per thread; the merge kernel gives every
  // (row, 4 dimensions) a thread and costs one launch gap (sparse D 256, 16
  // splits: 4.9 us of in-kernel merge).
  pl->merge_kernel = pl->tc && !pl->tcq && pl->nsplit > 1 && units * pl->nsplit <= slots &&
                     pl->chunk <= 4 * align;
  // [status block][counters][(max, sum) partials][O partials]
  const size_t nunit = (size_t)units;
  const size_t cnt_bytes = round_up(nunit * sizeof(unsigned int), 256);
  pl->ws = pl->off_cnt + cnt_bytes;
  if (pl->nsplit > 1) {
    const size_t ml_bytes = round_up(nunit * pl->nsplit * pl->rows * 2 * sizeof(float), 256);
    const size_t o_bytes = nunit * pl->nsplit * pl->rows * (size_t)a->D * sizeof(float);
    pl->off_ml = pl->ws;
    pl->off_o = pl->off_ml + ml_bytes;
    pl->ws = pl->off_o + o_bytes;
  }
  return FA_OK;
}

}  // namespace

namespace far {
void set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }
}  // namespace far

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
    case FA_ERR_INDEX_OOB: return "FA_ERR_INDEX_OOB";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_WAIT_EXPIRED: return "FA_ERR_WAIT_EXPIRED";
  }
  return "FA_ERR_UNKNOWN";
}

const char* fa_last_error(void) { return g_err; }

const char* fa_version(void) { return "fa_rows 0.1 sm_103a"; }

size_t fa_rows_workspace_size(const fa_rows_args* a, int is_prefill) {
  g_err[0] = 0;
  if (check_common(a) != FA_OK) return 0;
  if (is_prefill) return kPrefillWorkspace;
  DecodePlan pl;
  if (plan_decode(a, &pl) != FA_OK) return 0;
  return pl.ws;
}

int fa_rows_decode_launches(const fa_rows_args* a) {
  g_err[0] = 0;
  if (check_common(a) != FA_OK) return -1;
  DecodePlan pl;
  if (plan_decode(a, &pl) != FA_OK) return -1;
  if ((long long)a->S * a->Nq == 0) return 0;
  return pl.merge_kernel ? 2 : 1;
}

fa_status fa_rows_workspace_init(void* ws, size_t ws_bytes, fa_stream_t stream) {
  g_err[0] = 0;
  if (ws_bytes == 0) return FA_OK;
  if (!ws) return fail(FA_ERR_INVALID_ARG, "workspace is NULL");
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "workspace init");
}

fa_status fa_rows_status(void* ws, size_t ws_bytes, uint32_t* d_status, int clear, fa_stream_t stream) {
  g_err[0] = 0;
  if (!ws || ws_bytes < far::kStatusBytes || !aligned(ws, 4))
    return fail(FA_ERR_WORKSPACE, "a workspace of at least %zu bytes is required", far::kStatusBytes);
  if (!d_status || !aligned(d_status, 4)) return fail(FA_ERR_INVALID_ARG, "d_status must be a device uint32");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(d_status, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), st);
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "status copy");
}

fa_status fa_set_wait_limit_ns(uint64_t limit_ns) {
  g_err[0] = 0;
  g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed);
  return FA_OK;
}

fa_status fa_rows_decode(const fa_rows_args* a, void* ws, size_t ws_bytes, fa_stream_t stream) {
  g_err[0] = 0;
  fa_status st = check_common(a);
  if (st != FA_OK) return st;
  DecodePlan pl;
  st = plan_decode(a, &pl);
  if (st != FA_OK) return st;
  if ((long long)a->S * a->Nq == 0) return FA_OK;
  if (!ws || ws_bytes < pl.ws || !aligned(ws, 256))
    return fail(FA_ERR_WORKSPACE, "decode needs %zu bytes of 256-byte aligned, zero-initialised workspace (got %zu)",
                pl.ws, ws_bytes);
  far::DecodeParams p;
  memset(&p, 0, sizeof(p));
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.k_scale = a->k_scale;
  p.v_scale = a->v_scale;
  p.kv_rows = a->kv_rows;
  p.kv_len = a->kv_len;
  p.mask = a->mask;
  p.out = a->out;
  p.lse = a->lse;
  {
    char* w = static_cast<char*>(ws);
    p.counters = reinterpret_cast<unsigned int*>(w + pl.off_cnt);
    if (pl.nsplit > 1) {
      p.part_ml = reinterpret_cast<float*>(w + pl.off_ml);
      p.part_o = reinterpret_cast<float*>(w + pl.off_o);
    }
  }
  p.R = a->n_pool_rows;
  p.S = a->S;
  p.Nq = a->Nq;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.L = a->list_len;
  p.G = a->Hq / a->Hkv;
  p.QV = a->Nq * p.G;
  p.chunk = pl.chunk;
  p.nsplit = pl.nsplit;
  p.q_bf16 = a->q_dtype == FA_BF16;
  p.out_dtype = a->out_dtype;
  p.mask_kind = a->mask_kind;
  p.qscale = a->scale * far::kLog2e;
  p.wait_ns = wait_limit();
  p.merge_kernel = pl.merge_kernel ? 1 : 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaErrorInvalidValue;
  const int kind = kv_kind(a->kv_dtype);
  if (pl.tc) {
    unsigned int* err = static_cast<unsigned int*>(ws);   // the status word
    e = pl.tcq ? far::decode_tcq_launch(p, kind, err, s) : far::decode_tc_launch(p, a->D, kind, err, s);
    if (e == cudaSuccess && pl.merge_kernel) e = far::decode_merge_launch(p, a->D, s);
  } else if (kind == far::KV_BF16) {
    e = far::decode_launch_bf16(p, a->D, pl.qvp, s);
  } else if (kind == far::KV_F16) {
    e = far::decode_launch_f16(p, a->D, pl.qvp, s);
  } else if (kind == far::KV_I8) {
    e = far::decode_launch_i8(p, a->D, pl.qvp, s);
  }
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "decode launch");
}

fa_status fa_rows_prefill(const fa_rows_args* a, void* ws, size_t ws_bytes, fa_stream_t stream) {
  g_err[0] = 0;
  fa_status st = check_common(a);
  if (st != FA_OK) return st;
  if (!far::prefill_supported(a->D, kv_kind(a->kv_dtype)))
    return fail(FA_ERR_UNSUPPORTED, "prefill is built for D=128 with a bf16 or f16 pool");
  if (a->mask_kind == FA_MASK_DENSE) return fail(FA_ERR_UNSUPPORTED, "prefill takes FA_MASK_NONE or FA_MASK_CAUSAL");
  if (a->Hq / a->Hkv > 128) return fail(FA_ERR_UNSUPPORTED, "prefill packs at most 128 query heads per KV head");
  if (!aligned(a->q, 16)) return fail(FA_ERR_INVALID_ARG, "prefill needs 16-byte aligned q");
  if ((a->out_dtype == FA_F32 && !aligned(a->out, 16)) || !aligned(a->out, 8))
    return fail(FA_ERR_INVALID_ARG, "prefill needs a 16-byte aligned out");
  if ((long long)a->S * a->Nq == 0) return FA_OK;
  if (!ws || ws_bytes < kPrefillWorkspace || !aligned(ws, 16))
    return fail(FA_ERR_WORKSPACE, "prefill needs a zero-initialised workspace of %zu bytes, 16-byte aligned (it holds "
                                  "the status word)", kPrefillWorkspace);
  far::PrefillParams p;
  memset(&p, 0, sizeof(p));
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.kv_rows = a->kv_rows;
  p.kv_len = a->kv_len;
  p.mask = a->mask;
  p.out = a->out;
  p.lse = a->lse;
  p.R = a->n_pool_rows;
  p.S = a->S;
  p.Nq = a->Nq;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.L = a->list_len;
  p.G = a->Hq / a->Hkv;
  p.out_dtype = a->out_dtype;
  p.mask_kind = a->mask_kind;
  p.is_bf16 = a->q_dtype == FA_BF16;
  p.qscale = a->scale * far::kLog2e;
  p.err = static_cast<unsigned int*>(ws);   // the status word
  p.wait_ns = wait_limit();
  cudaError_t e = far::prefill_launch(p, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "prefill launch");
}

fa_status fa_rows_validate(const fa_rows_args* a, int64_t* d_status, fa_stream_t stream) {
  g_err[0] = 0;
  if (!a) return fail(FA_ERR_INVALID_ARG, "args is NULL");
  if (!d_status || !aligned(d_status, 8)) return fail(FA_ERR_INVALID_ARG, "d_status must be an 8-byte aligned device int64[2]");
  if (a->S < 0 || a->list_len < 0 || a->n_pool_rows < 0) return fail(FA_ERR_INVALID_ARG, "negative size");
  if ((long long)a->S * a->list_len > 0 && !a->kv_rows) return fail(FA_ERR_INVALID_ARG, "kv_rows is NULL");
  cudaError_t e = far::launch_validate(a->kv_rows, a->kv_len, a->S, a->list_len, a->n_pool_rows,
                                       reinterpret_cast<long long*>(d_status), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "validate launch");
}

fa_status fa_kv_page_table_to_rows(const int32_t* page_table, int32_t max_pages, const int32_t* seq_len,
                                   int32_t n_seq, int32_t page_size, int32_t* kv_rows, int32_t list_len,
                                   fa_stream_t stream) {
  g_err[0] = 0;
  if (n_seq < 0 || max_pages < 0 || list_len < 0 || page_size <= 0)
    return fail(FA_ERR_INVALID_ARG, "bad sizes (n_seq=%d max_pages=%d list_len=%d page=%d)", n_seq, max_pages, list_len, page_size);
  if ((long long)max_pages * page_size > 0x7fffffffLL) return fail(FA_ERR_INVALID_ARG, "max_pages*page_size overflows int32");
  if ((long long)n_seq * list_len == 0) return FA_OK;
  if (!seq_len || !kv_rows || (max_pages > 0 && !page_table)) return fail(FA_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(kv_rows, 16) && (list_len & 3) == 0) return fail(FA_ERR_INVALID_ARG, "kv_rows must be 16-byte aligned");
  cudaError_t e = far::launch_page_table_to_rows(page_table, max_pages, seq_len, n_seq, page_size, kv_rows, list_len,
                                                 reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "page table launch");
}

fa_status fa_kv_quantize_int8(const void* x, fa_dtype x_dtype, int64_t n_rows, int32_t Hkv, int32_t D,
                              const int32_t* dst_rows, int8_t* q, uint16_t* scale, int64_t n_pool_rows,
                              fa_stream_t stream) {
  g_err[0] = 0;
  if (x_dtype != FA_BF16 && x_dtype != FA_F16) return fail(FA_ERR_UNSUPPORTED, "x must be bf16 or f16");
  if (n_rows < 0 || Hkv <= 0 || D <= 0 || D > 256 || n_pool_rows < 0)
    return fail(FA_ERR_INVALID_ARG, "bad sizes (n_rows=%lld Hkv=%d D=%d)", (long long)n_rows, Hkv, D);
  if (n_pool_rows % far::kPage) return fail(FA_ERR_UNSUPPORTED, "INT8 pool rows must be a multiple of 64");
  if (!dst_rows && n_rows > n_pool_rows) return fail(FA_ERR_INVALID_ARG, "identity append needs n_rows <= pool rows");
  if (n_rows == 0) return FA_OK;
  if (!x || !q || !scale) return fail(FA_ERR_INVALID_ARG, "NULL pointer");
  cudaError_t e = far::launch_quantize_int8(x, x_dtype == FA_BF16, n_rows, Hkv, D, dst_rows, q, scale, n_pool_rows,
                                            reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "quantize launch");
}

fa_status fa_kv_dequantize_int8(const int8_t* q, const uint16_t* scale, int64_t n_rows, int32_t Hkv, int32_t D,
                                float* out, fa_stream_t stream) {
  g_err[0] = 0;
  if (n_rows < 0 || Hkv <= 0 || D <= 0) return fail(FA_ERR_INVALID_ARG, "bad sizes");
  if (n_rows % far::kPage) return fail(FA_ERR_UNSUPPORTED, "INT8 pool rows must be a multiple of 64");
  if (n_rows == 0) return FA_OK;
  if (!q || !scale || !out) return fail(FA_ERR_INVALID_ARG, "NULL pointer");
  cudaError_t e = far::launch_dequantize_int8(q, scale, n_rows, Hkv, D, out, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "dequantize launch");
}

fa_status fa_kv_quantize_int4(const void* x, fa_dtype x_dtype, int64_t n_rows, int32_t Hkv, int32_t D,
                              const int32_t* dst_rows, uint8_t* q, uint16_t* scale, int64_t n_pool_rows,
                              fa_stream_t stream) {
  g_err[0] = 0;
  if (x_dtype != FA_BF16 && x_dtype != FA_F16) return fail(FA_ERR_UNSUPPORTED, "x must be bf16 or f16");
  if (n_rows < 0 || Hkv <= 0 || D <= 0 || D > 256 || (D & 1) || n_pool_rows < 0)
    return fail(FA_ERR_INVALID_ARG, "bad sizes (n_rows=%lld Hkv=%d D=%d; D must be even, <= 256)", (long long)n_rows, Hkv,
                D);
  if (n_pool_rows % far::kPage) return fail(FA_ERR_UNSUPPORTED, "INT4 pool rows must be a multiple of 64");
  if (!dst_rows && n_rows > n_pool_rows) return fail(FA_ERR_INVALID_ARG, "identity append needs n_rows <= pool rows");
  if (n_rows == 0) return FA_OK;
  if (!x || !q || !scale) return fail(FA_ERR_INVALID_ARG, "NULL pointer");
  cudaError_t e = far::launch_quantize_int4(x, x_dtype == FA_BF16, n_rows, Hkv, D, dst_rows, q, scale, n_pool_rows,
                                            reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "quantize launch");
}

fa_status fa_kv_dequantize_int4(const uint8_t* q, const uint16_t* scale, int64_t n_rows, int32_t Hkv, int32_t D,
                                float* out, fa_stream_t stream) {
  g_err[0] = 0;
  if (n_rows < 0 || Hkv <= 0 || D <= 0 || (D & 1)) return fail(FA_ERR_INVALID_ARG, "bad sizes");
  if (n_rows % far::kPage) return fail(FA_ERR_UNSUPPORTED, "INT4 pool rows must be a multiple of 64");
  if (n_rows == 0) return FA_OK;
  if (!q || !scale || !out) return fail(FA_ERR_INVALID_ARG, "NULL pointer");
  cudaError_t e = far::launch_dequantize_int4(q, scale, n_rows, Hkv, D, out, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "dequantize launch");
}

fa_status fa_kv_quantize_fp8(const void* x, fa_dtype x_dtype, int64_t n_rows, int32_t Hkv, int32_t D,
                             const int32_t* dst_rows, uint8_t* q, uint16_t* scale, int64_t n_pool_rows,
                             fa_stream_t stream) {
  g_err[0] = 0;
  if (x_dtype != FA_BF16 && x_dtype != FA_F16) return fail(FA_ERR_UNSUPPORTED, "x must be bf16 or f16");
  if (n_rows < 0 || Hkv <= 0 || D <= 0 || D > 256 || n_pool_rows < 0)
    return fail(FA_ERR_INVALID_ARG, "bad sizes (n_rows=%lld Hkv=%d D=%d)", (long long)n_rows, Hkv, D);
  if (n_pool_rows % far::kPage) return fail(FA_ERR_UNSUPPORTED, "FP8 pool rows must be a multiple of 64");
  if (!dst_rows && n_rows > n_pool_rows) return fail(FA_ERR_INVALID_ARG, "identity append needs n_rows <= pool rows");
  if (n_rows == 0) return FA_OK;
  if (!x || !q || !scale) return fail(FA_ERR_INVALID_ARG, "NULL pointer");
  cudaError_t e = far::launch_quantize_fp8(x, x_dtype == FA_BF16, n_rows, Hkv, D, dst_rows, q, scale, n_pool_rows,
                                           reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "quantize launch");
}

fa_status fa_kv_dequantize_fp8(const uint8_t* q, const uint16_t* scale, int64_t n_rows, int32_t Hkv, int32_t D,
                               float* out, fa_stream_t stream) {
  g_err[0] = 0;
  if (n_rows < 0 || Hkv <= 0 || D <= 0) return fail(FA_ERR_INVALID_ARG, "bad sizes");
  if (n_rows % far::kPage) return fail(FA_ERR_UNSUPPORTED, "FP8 pool rows must be a multiple of 64");
  if (n_rows == 0) return FA_OK;
  if (!q || !scale || !out) return fail(FA_ERR_INVALID_ARG, "NULL pointer");
  cudaError_t e = far::launch_dequantize_fp8(q, scale, n_rows, Hkv, D, out, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "dequantize launch");
}

size_t fa_kv_sparse_rows_workspace_size(int32_t S, int32_t n_max) {
  g_err[0] = 0;
  if (S <= 0 || n_max < 0) return 0;
  return far::sparse_rows_workspace(S, n_max);
}

fa_status fa_kv_sparse_rows(const float* score, int32_t n_max, const int32_t* n_len, int32_t S, int32_t sinks,
                            int32_t recent, int32_t k, const int32_t* row_map, int32_t* kv_rows, int32_t list_len,
                            void* ws, size_t ws_bytes, fa_stream_t stream) {
  g_err[0] = 0;
  if (S < 0 || n_max < 0 || sinks < 0 || recent < 0 || k < 0 || list_len < 0)
    return fail(FA_ERR_INVALID_ARG, "negative size");
  if ((long long)sinks + recent + k > list_len)
    return fail(FA_ERR_INVALID_ARG, "list_len %d < sinks + recent + k = %lld", list_len,
                (long long)sinks + recent + k);
  if (S == 0 || list_len == 0) return FA_OK;
  if (!kv_rows || (n_max > 0 && !score)) return fail(FA_ERR_INVALID_ARG, "NULL pointer");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (ws) {
    const size_t need = far::sparse_rows_workspace(S, n_max);
    if (ws_bytes < need || !aligned(ws, 16))
      return fail(FA_ERR_WORKSPACE, "sparse rows workspace must be %zu bytes, 16-byte aligned", need);
    e = far::launch_sparse_rows_ws(score, n_max, n_len, S, sinks, recent, k, row_map, kv_rows, list_len, ws, st);
  } else {
    e = far::launch_sparse_rows(score, n_max, n_len, S, sinks, recent, k, row_map, kv_rows, list_len, st);
  }
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "sparse rows launch");
}

fa_status fa_kv_append(const void* x, fa_dtype dtype, int64_t n_rows, int32_t Hkv, int32_t D, const int32_t* dst_rows,
                       void* pool, int64_t n_pool_rows, fa_stream_t stream) {
  g_err[0] = 0;
  if (dtype != FA_BF16 && dtype != FA_F16) return fail(FA_ERR_UNSUPPORTED, "append is for 16-bit pools");
  if (n_rows < 0 || Hkv <= 0 || D <= 0 || n_pool_rows < 0) return fail(FA_ERR_INVALID_ARG, "bad sizes");
  const long long row_bytes = (long long)Hkv * D * 2;
  if (row_bytes % 16) return fail(FA_ERR_UNSUPPORTED, "Hkv*D*2 must be a multiple of 16 bytes");
  if (n_rows == 0) return FA_OK;
  if (!x || !dst_rows || !pool) return fail(FA_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(x, 16) || !aligned(pool, 16)) return fail(FA_ERR_INVALID_ARG, "x and pool must be 16-byte aligned");
  cudaError_t e = far::launch_kv_append(x, n_rows, (int)row_bytes, dst_rows, pool, n_pool_rows,
                                        reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "append launch");
}

}  // extern "C"
