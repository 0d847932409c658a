"""Benchmark of row-indexed attention over a unified KV pool on GB300.

Headline workload: decode, bf16, 4 sequences x 16,384 rows in a 65,536-row
shuffled pool, 32 query / 8 KV heads, head_dim 128, one query token per
sequence (lists sorted ascending).  Metric: gathered-KV GB/s = listed rows x
(K + V bytes) per KV head, per second; padding, indices, Q and O excluded.

A default run on one GPU also measures, in the same JSON line under
``configs``, the other configurations: the small fp16 decode, the prefill
chunk (4 x 2,048 query rows over 99,936-row lists in a 400,000-row pool,
causal; tensor TFLOP/s with 4*D FLOPs per visible (query, key, head) triple)
in its ubatch-run layout and with every row shuffled over the pool, the paged
INT8 decode and the sparse long-context decode -- each with its own roofline,
clocks, end-to-end figure and oracle baseline.

``--workload NAME`` measures one workload alone.  Workloads:
``paged_int8`` / ``paged_int4`` / ``paged_fp8`` (page tables expanded to row
lists, then the quantised-pool decode), ``sparse_bf16`` (sink + recent +
selected list, D 256), ``sparse_select_bf16`` (the list built from a score each
step, then the decode), ``decode_f16_small``, the profiling sizes
``prefill_bf16_small`` / ``paged_int8_small``, and ``kv_append_int8`` (a
ubatch of new rows quantised into fresh pages; GB/s of its input, codes,
scales and destination indices).

One JSON line on stdout (rank 0).  Under torchrun each rank runs an
independent replica of the workload (the path shards by sequence with no
exchange), timing is the max over ranks.

``--impl reference`` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import os

# the CPU oracle legs run one BLAS thread per worker process
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "row-indexed attention: decode gathered-KV GB/s, prefill TFLOP/s (vs GB300 roofline)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {
    "decode": ["row_indexed_flash_gb300/csrc/decode_tc.cu", "row_indexed_flash_gb300/csrc/tc.cuh",
               "row_indexed_flash_gb300/csrc/merge.cuh", "row_indexed_flash_gb300/csrc/widen.cuh",
               "row_indexed_flash_gb300/csrc/fa_internal.cuh"],
    "decode_q": ["row_indexed_flash_gb300/csrc/decode_tcq.cu", "row_indexed_flash_gb300/csrc/tc.cuh",
                 "row_indexed_flash_gb300/csrc/merge.cuh", "row_indexed_flash_gb300/csrc/widen.cuh",
                 "row_indexed_flash_gb300/csrc/fa_internal.cuh"],
    "prefill": ["row_indexed_flash_gb300/csrc/prefill.cu", "row_indexed_flash_gb300/csrc/tc.cuh",
                "row_indexed_flash_gb300/csrc/fa_internal.cuh"],
    "append": ["row_indexed_flash_gb300/csrc/kvcache.cu", "row_indexed_flash_gb300/csrc/fa_internal.cuh"],
}
KERNEL_NAMES = {"decode": "fa_rows_decode_tc_kernel", "prefill": "fa_rows_prefill_kernel",
                "decode_q": "fa_rows_decode_tcq_kernel", "append": "quantize_rows_staged_kernel"}
PROFILE_FILES = {
    "decode_bf16": "profiles/decode_bf16_4x16384_ncu.txt",
    "prefill_bf16": "profiles/prefill_bf16_4x2048x99936_ncu.txt",
    "prefill_bf16_shuffled": "profiles/prefill_bf16_shuffled_4x2048x99936_ncu.txt",
    "prefill_bf16_small": "profiles/prefill_bf16_4x2048x16384_ncu.txt",
    "paged_int8": "profiles/paged_int8_32seq_ncu.txt",
    "paged_int8_small": "profiles/paged_int8_16seq_ncu.txt",
    "kv_append_int8": "profiles/kv_append_int8_4x2048_ncu.txt",
}


# ---------------------------------------------------------------------------
# ranks: each rank runs an independent replica of the workload


def max_over_ranks(vals, dist_mod=None, device=None):
    """Each value's maximum over all ranks of the default process group (the
    values themselves when there is one rank or no group)."""
    vals = [float(x) for x in vals]
    if dist_mod is None or not dist_mod.is_available() or not dist_mod.is_initialized():
        return vals
    if dist_mod.get_world_size() == 1:
        return vals
    import torch
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(world: int, work_per_rank: float, step_ms: float, scale: float) -> float:
    """Work of all ranks per second of the slowest rank's step, in units of scale."""
    return world * work_per_rank / (step_ms * 1e-3) / scale


# ---------------------------------------------------------------------------
# workload accounting


def decode_bytes(p, quant=None) -> int:
    """Algorithmic bytes: each listed row is read once per KV head (K and V
    codes, plus their two fp16 scales for a quantised pool)."""
    per = {None: 4 * p.D, "int8": 2 * p.D + 4, "fp8": 2 * p.D + 4, "int4": p.D + 4}[quant]
    return p.n_valid() * p.Hkv * per


def prefill_flops(p) -> int:
    """4*D per visible (query, key, head): QK^T and PV, 2*D each."""
    n = p.L
    vis = 0
    for i in range(p.Nq):
        vis += max(0, min(n, n - p.Nq + i + 1))
    return 4 * p.D * p.Hq * p.S * vis


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        out = dict(FALLBACK_PEAKS)
        for k in out:
            for cand in (k, k.replace("_gbs", "_GBs")):
                if isinstance(d.get(cand), (int, float)):
                    out[k] = float(d[cand])
        return out, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def code_only(text: str) -> str:
    """C/C++/CUDA source with its comments removed and every run of
    whitespace collapsed to one space (string and character literals kept)."""
    out, i, n = [], 0, len(text)
    while i < n:
        ch = text[i]
        if ch in "\"'":
            j = i + 1
            while j < n and text[j] != ch:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(ch)
            i += 1
    return " ".join("".join(out).split())


def source_sha(kind: str, read=None) -> str:
    """Hash of the code (comments and layout excluded) of a kernel's sources:
    the key under which ncu summaries in profiles/ record what they measured."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        if read is None:
            with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
                text = f.read()
        else:
            text = read(rel)
        h.update(code_only(text).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kind: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, PROFILE_FILES.get(workload, ""))
    if not os.path.isfile(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.strip().split("=", 1)
                kv[k.strip()] = v.strip()
    if kv.get("kernel_source_sha") != source_sha(kind):
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# CPU oracle legs (fork pool, created before any CUDA call)

_P = None
_PAGED = None   # paged sample: quantiser name and, per sampled slice, its pages' codes and scales


def quant_of(workload: str):
    """Pool codec of a workload (None for 16-bit pools)."""
    if not workload.startswith("paged"):
        return None
    return {"paged_int4": "int4", "paged_fp8": "fp8"}.get(workload, "int8")


def _oracle_unit(args):
    import oracle
    s, g, qrows = args
    p = _P
    G = p.Hq // p.Hkv
    if _PAGED is not None:
        # paged decode of (slice s, KV head g): expand the slice's page table
        # over a pool of its own pages, dequantise them, attend over the list
        kc, ks, vc, vs = _PAGED[s]
        deq = {"int8": oracle.dequantize_int8, "int4": oracle.dequantize_int4,
               "fp8": oracle.dequantize_fp8}[_PAGED["quant"]]
        n_pages = kc.shape[0] // p.page_size
        rows = oracle.page_table_to_rows(np.arange(n_pages, dtype=np.int32)[None, :], p.seq_len[s:s + 1], p.L,
                                         p.page_size)
        k = deq(kc[:, g:g + 1], ks[:, g:g + 1]).astype(np.float64)
        v = deq(vc[:, g:g + 1], vs[:, g:g + 1]).astype(np.float64)
        q = oracle.widen(p.q[s:s + 1, :, g * G:(g + 1) * G], p.dtype)
        oracle.attend_rows(q, k, v, rows, p.scale)
        return s, g
    if qrows is None:
        q = oracle.widen(p.q[s:s + 1, :, g * G:(g + 1) * G], p.dtype)
        extra = {}
    else:
        q = oracle.widen(p.q[s:s + 1, list(qrows), g * G:(g + 1) * G], p.dtype)
        extra = dict(query_rows=list(qrows), n_query=p.Nq)
    oracle.attend_rows(q, p.k[:, g:g + 1], p.v[:, g:g + 1], p.kv_rows[s:s + 1], p.scale, causal=p.causal,
                       kv_len=None if p.kv_len is None else p.kv_len[s:s + 1], kv_format=p.dtype, **extra)
    return s, g


def oracle_units(p, prefill: bool, q_sample: int = 4):
    """(slice, KV head, query rows) units of the oracle legs and the work of
    each: gathered K+V bytes for decode, 4*D FLOPs per visible (query, key,
    head) for prefill, whose units take ``q_sample`` query rows spread over the
    chunk."""
    units, work = [], []
    G = p.Hq // p.Hkv
    for s in range(p.S):
        for g in range(p.Hkv):
            if prefill:
                qrows = tuple(sorted({(p.Nq - 1) * t // max(1, q_sample - 1) for t in range(q_sample)}))
                vis = sum(max(0, min(p.L, p.L - p.Nq + i + 1)) if p.causal else p.L for i in qrows)
                units.append((s, g, qrows))
                work.append(4 * p.D * G * vis)
            else:
                units.append((s, g, None))
                work.append(int((p.kv_rows[s] >= 0).sum()) * 2 * p.D * 2)
    return units, work


def paged_oracle_units(p, quant: str, min_rows: int = 65536):
    """Units of the paged oracle leg: the (slice, KV head) pairs of a seeded
    sample of slices holding at least ``min_rows`` listed rows.  Each sampled
    slice's pages are quantised by the oracle's own codec beforehand (the write
    path, not timed); a unit then expands the page table, dequantises and
    attends.  Work = listed rows x (codes + two fp16 scales) per KV head."""
    global _PAGED
    import oracle
    quantise = {"int8": oracle.quantize_int8, "int4": oracle.quantize_int4, "fp8": oracle.quantize_fp8}[quant]
    order = synth.rng(synth.SEED_BASE + 99).permutation(p.S)
    chosen, total = [], 0
    for s in order:
        chosen.append(int(s))
        total += int(p.seq_len[s])
        if total >= min_rows:
            break
    paged = {"quant": quant}
    for s in chosen:
        n_pages = (int(p.seq_len[s]) + p.page_size - 1) // p.page_size
        pages = p.page_table[s, :n_pages].astype(np.int64)
        rows = (pages[:, None] * p.page_size + np.arange(p.page_size)[None, :]).ravel()
        kc, ks = quantise(oracle.widen(p.k[rows], p.dtype).astype(np.float32))
        vc, vs = quantise(oracle.widen(p.v[rows], p.dtype).astype(np.float32))
        paged[s] = (kc, ks, vc, vs)
    _PAGED = paged
    per_row = {"int8": 2 * p.D + 4, "fp8": 2 * p.D + 4, "int4": p.D + 4}[quant]
    units = [(s, g, None) for s in chosen for g in range(p.Hkv)]
    work = [int(p.seq_len[s]) * per_row for s in chosen for g in range(p.Hkv)]
    return units, work, f"{len(chosen)} of {p.S} slices ({total} listed rows, pages quantised beforehand)"


def oracle_rate(p, units, work, procs: int, min_seconds: float = 0.0, max_passes: int = 1):
    """Work per second of the oracle over ``units``: whole passes over them,
    repeated until ``min_seconds`` have elapsed (at most ``max_passes``)."""
    global _P
    _P = p
    ctx = mp.get_context("fork")
    passes = 0
    with ctx.Pool(procs) as pool:
        t0 = time.perf_counter()
        while True:
            pool.map(_oracle_unit, units, chunksize=1)
            passes += 1
            dt = time.perf_counter() - t0
            if dt >= min_seconds or passes >= max_passes:
                break
    return passes * sum(work) / dt, dt, passes


def cpu_leg(p, workload: str, procs: int, min_seconds: float):
    """The oracle, as it stands, on the host cores over a bounded sample of the
    workload: whole passes over its units for about ``min_seconds``."""
    global _PAGED
    prefill = workload.startswith("prefill")
    unit, div = ("TFLOP/s", 1e12) if prefill else ("GB/s", 1e9)
    if p.kv_rows is None:
        units, work, what = paged_oracle_units(p, quant_of(workload))
    else:
        units, work = oracle_units(p, prefill)
        what = f"{len(units)} (slice, KV head) units" + (
            f" x {len(units[0][2])} query rows" if prefill else " (whole workload)")
    try:
        v, dt, passes = oracle_rate(p, units, work, procs, min_seconds=min_seconds, max_passes=1000)
    finally:
        _PAGED = None
    return {"value": round(v / div, 6), "unit": unit, "cores": procs, "kind": "oracle",
            "sample": f"{what} x {passes} passes, {dt:.1f} s wall"}


# ---------------------------------------------------------------------------
# clocks during the timed region


def queue_ahead(torch, steps: int, host_us_per_step: float = 60.0) -> None:
    """Holds the stream on a device-side sleep long enough for the host to
    enqueue every timed step behind it, so that the timed region measures the
    GPU running the steps back to back rather than the host's launch rate (a
    step of a few microseconds is otherwise timed at the Python loop's pace).
    The sleep ends before the first timing event, outside the timed region."""
    seconds = min(20e-3, 0.5e-3 + steps * host_us_per_step * 1e-6)
    torch.cuda._sleep(int(seconds * 2.1e9))


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.out:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm

# The configurations measured beside the headline decode in a default run
# (one GPU): the small fp16 decode, the prefill chunk in its ubatch-run layout
# and fully shuffled, the paged INT8 decode and the sparse long-context decode.
CONFIG_WORKLOADS = ["decode_f16_small", "prefill_bf16", "prefill_bf16_shuffled", "paged_int8", "sparse_bf16"]
WORKLOAD_CHOICES = ["decode_bf16", "decode_f16_small", "prefill_bf16", "prefill_bf16_shuffled", "prefill_bf16_small",
                    "paged_int8", "paged_int8_small", "paged_int4", "paged_fp8", "sparse_bf16", "sparse_select_bf16",
                    "kv_append_int8"]


def build_problem(workload: str, cache=None):
    cache = {} if cache is None else cache
    if workload == "decode_bf16":
        return synth.decode_bf16_large()
    if workload in ("prefill_bf16", "prefill_bf16_shuffled"):
        if "prefill_bf16" not in cache:
            cache["prefill_bf16"] = synth.prefill_bf16()
        p = cache["prefill_bf16"]
        if workload == "prefill_bf16":
            return p
        # the same pool, every listed row at a random slot: all K/V tiles gathered
        return synth.relabel_rows(p, synth.SEED_BASE + 13,
                                  p.name.replace("(2048-row runs)", "(rows shuffled over the pool)"))
    if workload in ("paged_int8", "paged_int4", "paged_fp8"):
        return synth.paged_int8()   # the paged layout; the pool is quantised by each side
    if workload == "paged_int8_small":
        # profiling size: 16 sequences of 1k-32k tokens (about 250 MB of codes, above L2)
        return synth.paged_int8(n_seq=16, lo=1024, hi=32768)
    if workload in ("sparse_bf16", "sparse_select_bf16"):
        return synth.sparse_bf16()
    if workload == "decode_f16_small":
        return synth.decode_fp16_small()
    if workload == "prefill_bf16_small":
        # profiling size: 4 x 16,384-row lists in a 65,536-row pool (268 MB of K/V, above L2)
        return synth.prefill_bf16(n_seq=4, seq_rows=16384, pool_rows=65536)
    raise SystemExit(f"unknown workload {workload}")


def kernel_kind(workload: str) -> str:
    if workload.startswith("prefill"):
        return "prefill"
    return "decode_q" if workload.startswith("paged") else "decode"


def measure(args, rank, world, p, workload, cpu_baseline):
    """Times one workload on this rank's GPU: warm-up, then args.steps steps
    (one replayed CUDA graph holding the steps' launches) with CUDA events on the
    launching stream, clocks sampled meanwhile; then the same call end to end
    with host inputs.  Returns the result dict on rank 0."""
    import ctypes

    import torch
    import torch.distributed as dist

    import row_indexed_flash_gb300 as far

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    tdt = torch.bfloat16 if p.dtype == "bf16" else torch.float16

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(tdt).to(dev)

    is_prefill = workload.startswith("prefill")
    paged = p.kv_rows is None
    quant = quant_of(workload)
    quantise = {"int4": far.fa_kv_quantize_int4, "fp8": far.fa_kv_quantize_fp8}.get(quant, far.fa_kv_quantize_int8)
    q = to_dev(p.q)
    if paged:
        # write path (not timed): quantise the bf16 pool into codes + fp16 scales
        kb, vb = to_dev(p.k), to_dev(p.v)
        kq, ks = quantise(kb, p.R)
        vq, vs = quantise(vb, p.R)
        del kb, vb
        torch.cuda.synchronize(dev)
        base = (kq, vq, ks, vs)
        pt = torch.from_numpy(p.page_table).to(dev)
        sl = torch.from_numpy(p.seq_len).to(dev)
        rows = torch.empty((p.S, p.L), dtype=torch.int32, device=dev)
    else:
        base = (to_dev(p.k), to_dev(p.v), None, None)
        rows = torch.from_numpy(p.kv_rows).to(dev)
    select = workload == "sparse_select_bf16"
    if select:
        # each step builds the list (4 sinks + 1,532 by score + 512 recent) from a
        # seeded fp32 score per position, then decodes over it
        sel_score = torch.from_numpy(synth.rng(9).standard_normal((1, p.R)).astype(np.float32)).to(dev)
        sel_ws = torch.empty(max(far.lib().fa_kv_sparse_rows_workspace_size(1, p.R), 16), dtype=torch.uint8,
                             device=dev)
    pool_bytes = sum(t.numel() * t.element_size() for t in base if t is not None)
    # rotate over enough pool copies that each step reads data not left in L2
    n_copies = max(1, min(3, int(math.ceil(3 * 129e6 / pool_bytes)) + 1)) if not is_prefill else 1
    pools = [base] + [tuple(None if t is None else t.clone() for t in base) for _ in range(n_copies - 1)]
    out = torch.empty((p.S, p.Nq, p.Hq, p.D), dtype=torch.float32, device=dev)
    a_list = []
    for (k, v, ksc, vsc) in pools:
        kw = {}
        if paged:
            kw = dict(k_scale=ksc, v_scale=vsc, kv_len=sl, n_valid_hint=p.n_valid())
        a, _, _ = far.make_args(q, k, v, rows, p.scale, causal=p.causal, out=out, **kw)
        a_list.append(a)
    lib = far.lib()
    entry = lib.fa_rows_prefill if is_prefill else lib.fa_rows_decode
    need = far.fa_rows_workspace_size(a_list[0], is_prefill)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    sh = stream.cuda_stream

    def call(st):
        if st != 0:
            raise far.FaRowsError(st, far.fa_last_error())

    def step(i, sh=sh, a=None):
        if select:
            call(lib.fa_kv_sparse_rows(sel_score.data_ptr(), p.R, None, 1, 4, 512, 1532, None, rows.data_ptr(),
                                       rows.shape[1], sel_ws.data_ptr(), sel_ws.numel(), sh))
        if paged:   # page tables -> row lists, then the decode (both kernels of the step)
            call(lib.fa_kv_page_table_to_rows(pt.data_ptr(), pt.shape[1], sl.data_ptr(), p.S, p.page_size,
                                              rows.data_ptr(), p.L, sh))
        call(entry(ctypes.byref(a_list[i % len(a_list)] if a is None else a), ws.data_ptr(), ws.numel(), sh))

    # a bf16 prefill is three kernels: the V-range scan, then the two prefill
    # modes (V to f16, V kept in bf16), one of which exits at once
    # a decode whose splits are merged by a kernel of their own is two
    launches_per_step = ((1 if is_prefill else lib.fa_rows_decode_launches(ctypes.byref(a_list[0])))
                         + (1 if paged else 0) + (8 if select else 0) + (2 if is_prefill and p.dtype == "bf16" else 0))

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)

    # The K timed steps are captured, in order, into one CUDA graph that is
    # replayed once: a graph per step, or a launch per kernel from Python,
    # leaves gaps of several microseconds between the small steps on the
    # device.  The captured kernels and arguments are exactly those of step(i).
    graph = None
    if not args.no_graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(args.steps):
                    step(i, torch.cuda.current_stream(dev).cuda_stream)
            graph.replay()   # untimed: the first replay uploads the graph
            torch.cuda.synchronize(dev)
        except Exception as exc:   # fall back to direct launches
            print(f"# CUDA graph capture failed ({exc}); timing direct launches", file=sys.stderr)
            graph = None

    def timed_steps():
        if graph is not None:
            graph.replay()
        else:
            for i in range(args.steps):
                step(i)

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        queue_ahead(torch, args.steps)
        t0.record(stream)
        timed_steps()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    total_ms = t0.elapsed_time(t1)
    # one event pair over the whole region: events between the steps would
    # each add a device-side gap of about a microsecond to the small steps
    mean_launch_ms = total_ms / args.steps
    # a wait that ran out would have made every number above meaningless
    if far.fa_rows_status(ws, clear=True) & far.FA_WS_WAIT_EXPIRED:
        raise SystemExit(f"{workload}: a pipeline wait ran out during the timed steps")

    # end to end through the public API: the step's inputs copied in from
    # pinned host memory every step (Q, the pool, the lists -- for a paged
    # pool its codes, scales, page table and lengths), the output read back
    k0, v0, ks0, vs0 = base
    host = {"q": q, "k": k0, "v": v0}
    if paged:
        host.update(ks=ks0, vs=vs0, pt=pt, sl=sl)
    else:
        host["rows"] = rows
    pinned = {n: t.cpu().pin_memory() for n, t in host.items()}
    dbuf = {n: torch.empty_like(t) for n, t in host.items()}
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e_rows = rows if paged else dbuf["rows"]
    kw = {}
    if paged:
        kw = dict(k_scale=dbuf["ks"], v_scale=dbuf["vs"], kv_len=dbuf["sl"], n_valid_hint=p.n_valid())
    a_e2e, _, _ = far.make_args(dbuf["q"], dbuf["k"], dbuf["v"], e_rows, p.scale, causal=p.causal, out=out, **kw)
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = hout.numel() * hout.element_size()
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        for n, t in pinned.items():
            dbuf[n].copy_(t, non_blocking=True)
        if select:
            call(lib.fa_kv_sparse_rows(sel_score.data_ptr(), p.R, None, 1, 4, 512, 1532, None, e_rows.data_ptr(),
                                       rows.shape[1], sel_ws.data_ptr(), sel_ws.numel(), sh))
        if paged:
            call(lib.fa_kv_page_table_to_rows(dbuf["pt"].data_ptr(), pt.shape[1], dbuf["sl"].data_ptr(), p.S,
                                              p.page_size, e_rows.data_ptr(), p.L, sh))
        call(entry(ctypes.byref(a_e2e), ws.data_ptr(), ws.numel(), sh))
        hout.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if far.fa_rows_status(ws, clear=True) & far.FA_WS_WAIT_EXPIRED:
        raise SystemExit(f"{workload}: a pipeline wait ran out during the end-to-end steps")

    step_ms = total_ms / args.steps
    if world > 1:
        step_ms, e2e_ms, mean_launch_ms = max_over_ranks([step_ms, e2e_ms, mean_launch_ms], dist, dev)
    launch_mode = "cuda_graph of the K timed steps" if graph is not None else "direct"
    del graph, pools, a_list, base, pinned, dbuf
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    if rank != 0:
        return None

    pk, pk_src = peaks()
    kind = kernel_kind(workload)
    if is_prefill:
        work = prefill_flops(p)
        unit, scale_ = "TFLOP/s", 1e12
        peak_key = "bf16_tflops_sustained" if args.steps * step_ms > 2000 else "bf16_tflops"
        bound = "tensor"
    else:
        work = decode_bytes(p, quant)
        unit, scale_ = "GB/s", 1e9
        peak_key = "hbm_gbs"
        bound = "hbm"
    peak = pk[peak_key]
    value = whole_job_rate(world, work, step_ms, scale_)
    achieved = work / (mean_launch_ms * 1e-3) / scale_
    return {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": quant if paged else p.dtype,
        "data": "synthetic (seeded N(0,1) values, generator shapes of the pages' workloads)",
        "config": {
            "workload": p.name,
            "kv_rows": f"[{p.S}, {p.L}] int32" + (" (expanded from page tables each step)" if paged else ""),
            "n_valid_rows": p.n_valid(),
            "l2": (f"inputs larger than L2: {n_copies} pool copies of {pool_bytes / 1e6:.0f} MB rotated"
                   if not is_prefill else f"inputs larger than L2: pool {pool_bytes / 1e9:.2f} GB"),
            "parallelism": f"replicas x{world}",
            "launch": launch_mode,
            "queue": "timed steps enqueued behind a device sleep: host launch time is not timed",
        },
        "roofline": {
            "bound": bound,
            "achieved": round(achieved, 2),
            "peak": peak,
            "peak_source": f"{pk_src} {peak_key}",
            "unit": unit,
            "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic(workload, kind),
            "kernel": KERNEL_NAMES[kind],
            "kernel_ms": round(mean_launch_ms, 5),
            "work_per_launch": work,
        },
        "e2e": {
            "value": round(whole_job_rate(world, work, e2e_ms, scale_), 2),
            "unit": unit,
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "ms_per_step": round(e2e_ms, 4),
        },
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk.summary(),
        "cpu_baseline": cpu_baseline,
    }


# ---------------------------------------------------------------------------


APPEND = dict(n_seq=4, new=2048, R=400000, Hkv=8, D=128)


def append_bytes(n_rows: int, Hkv: int, D: int) -> int:
    """Algorithmic bytes of an INT8 append: per (row, head) the 16-bit input,
    the codes and the fp16 scale; per row its destination index."""
    return n_rows * (Hkv * (2 * D + D + 2) + 4)


def append_oracle_rate(min_seconds: float = 0.0, passes_wanted: int = 0):
    """The oracle's append (quantise + scatter, int8) timed on a bounded
    sample: one sequence's 2,048 new rows into a 16,384-row pool, for
    passes_wanted passes, else until min_seconds have passed."""
    import oracle
    c = APPEND
    g = synth.rng(synth.SEED_BASE + 7)
    x = oracle.widen_bf16(synth.normal_bits(g, (c["new"], c["Hkv"], c["D"]), "bf16")).astype(np.float32)
    pool = np.zeros((16384, c["Hkv"], c["D"]), np.int8)
    sc = np.zeros((16384 // 64, c["Hkv"], 64), np.float16)
    dst = (4096 + np.arange(c["new"])).astype(np.int32)
    passes, t0 = 0, time.perf_counter()
    while True:
        oracle.append_rows(pool, x, dst, sc, fmt="int8")
        passes += 1
        dt = time.perf_counter() - t0
        if (passes >= passes_wanted) if passes_wanted > 0 else (dt >= min_seconds):
            break
    v = passes * append_bytes(c["new"], c["Hkv"], c["D"]) / dt / 1e9
    return v, dt, passes


def run_append(args, rank, world, cpu_baseline):
    """Fused KV append: each step quantises a ubatch of new K rows (bf16,
    4 sequences x 2,048 tokens) to INT8 and writes codes and scales into
    fresh 64-row pages of a 400,000-row pool (one 2,048-row block of pages per
    sequence at a seeded random position): one fa_kv_quantize_int8 call."""
    import ctypes

    import torch
    import torch.distributed as dist

    import row_indexed_flash_gb300 as far

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    c = APPEND
    n_seq, new, R, Hkv, D = c["n_seq"], c["new"], c["R"], c["Hkv"], c["D"]
    n = n_seq * new
    g = synth.rng(synth.SEED_BASE + 6)
    x0 = torch.from_numpy(synth.normal_bits(g, (n, Hkv, D), "bf16").view(np.int16)).view(torch.bfloat16).to(dev)
    x_bytes = x0.numel() * 2
    # inputs larger than L2: rotate over copies of the ubatch, each written to its own pages
    n_copies = int(math.ceil(2 * 129e6 / x_bytes)) + 1
    blocks = g.permutation(R // new)[: n_copies * n_seq]
    dsts = [torch.from_numpy(np.concatenate([blocks[ci * n_seq + si] * new + np.arange(new)
                                             for si in range(n_seq)]).astype(np.int32)).to(dev)
            for ci in range(n_copies)]
    xs = [x0] + [x0.clone() for _ in range(n_copies - 1)]
    q = torch.zeros((R, Hkv, D), dtype=torch.int8, device=dev)
    sc = torch.zeros((R // 64, Hkv, 64), dtype=torch.float16, device=dev)
    lib = far.lib()
    bf = far._DT[torch.bfloat16]

    def step(i, sh=sh):
        st = lib.fa_kv_quantize_int8(xs[i % n_copies].data_ptr(), bf, n, Hkv, D, dsts[i % n_copies].data_ptr(),
                                     q.data_ptr(), sc.data_ptr(), R, sh)
        if st != 0:
            raise far.FaRowsError(st, far.fa_last_error())

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    # the K timed steps captured, in order, into one CUDA graph (see measure)
    graph = None
    if not args.no_graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(args.steps):
                    step(i, torch.cuda.current_stream(dev).cuda_stream)
            graph.replay()   # untimed: the first replay uploads the graph
            torch.cuda.synchronize(dev)
        except Exception as exc:
            print(f"# CUDA graph capture failed ({exc}); timing direct launches", file=sys.stderr)
            graph = None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        queue_ahead(torch, args.steps)
        t0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(args.steps):
                step(i)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    step_ms = t0.elapsed_time(t1) / args.steps
    launch_ms = step_ms   # one launch per step, timed over the whole region

    # end to end: the ubatch and its destinations copied in from pinned host
    # memory, the call, and the written codes and scales copied back
    hx = x0.cpu().pin_memory()
    hd = dsts[0].cpu().pin_memory()
    dx, dd = torch.empty_like(x0), torch.empty_like(dsts[0])
    starts = [int(blocks[si]) * new for si in range(n_seq)]
    hq = [torch.empty((new, Hkv, D), dtype=torch.int8).pin_memory() for _ in range(n_seq)]
    hs = [torch.empty((new // 64, Hkv, 64), dtype=torch.float16).pin_memory() for _ in range(n_seq)]
    h2d = hx.numel() * 2 + hd.numel() * 4
    d2h = sum(t.numel() for t in hq) + sum(t.numel() * 2 for t in hs)

    def e2e_step():
        dx.copy_(hx, non_blocking=True)
        dd.copy_(hd, non_blocking=True)
        st = lib.fa_kv_quantize_int8(dx.data_ptr(), bf, n, Hkv, D, dd.data_ptr(), q.data_ptr(), sc.data_ptr(), R, sh)
        if st != 0:
            raise far.FaRowsError(st, far.fa_last_error())
        for si in range(n_seq):
            r0 = starts[si]
            hq[si].copy_(q[r0:r0 + new], non_blocking=True)
            hs[si].copy_(sc[r0 // 64:(r0 + new) // 64], non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    e2e_steps = max(3, min(args.steps, 20))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if world > 1:
        step_ms, e2e_ms, launch_ms = max_over_ranks([step_ms, e2e_ms, launch_ms], dist, dev)
    if rank != 0:
        return None
    pk, pk_src = peaks()
    work = append_bytes(n, Hkv, D)
    achieved = work / (launch_ms * 1e-3) / 1e9
    return {
        "metric": METRIC,
        "value": round(whole_job_rate(world, work, step_ms, 1e9), 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8",
        "data": "synthetic (seeded N(0,1) bf16 rows)",
        "config": {
            "workload": f"kv-append int8: {n_seq} x {new} new rows into a {R}-row pool, {Hkv} KV heads, D{D}",
            "l2": f"inputs larger than L2: {n_copies} ubatch copies of {x_bytes / 1e6:.1f} MB rotated, "
                  f"each to its own pages",
            "parallelism": f"replicas x{world}",
            "launch": "cuda_graph of the K timed steps" if graph is not None else "direct",
            "queue": "timed steps enqueued behind a device sleep: host launch time is not timed",
        },
        "roofline": {
            "bound": "hbm",
            "achieved": round(achieved, 2),
            "peak": pk["hbm_gbs"],
            "peak_source": pk_src,
            "unit": "GB/s",
            "frac": round(achieved / pk["hbm_gbs"], 4),
            "traffic": profiled_traffic("kv_append_int8", "append"),
            "kernel": KERNEL_NAMES["append"],
            "kernel_ms": round(launch_ms, 5),
            "work_per_launch": work,
        },
        "e2e": {
            "value": round(whole_job_rate(world, work, e2e_ms, 1e9), 2),
            "unit": "GB/s",
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "ms_per_step": round(e2e_ms, 4),
        },
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "cpu_baseline": cpu_baseline,
    }


def reference_arm(args, rank, world, procs):
    """The oracle, as it stands, on the host cores: each step a bounded sample
    of the workload (the first `procs` units), on this arm's metric."""
    if rank != 0:
        return
    workload = args.workload
    p = build_problem(workload)
    prefill = workload.startswith("prefill")
    unit, div = ("TFLOP/s", 1e12) if prefill else ("GB/s", 1e9)
    if p.kv_rows is None:
        units, work, what = paged_oracle_units(p, quant_of(workload))
    else:
        units, work = oracle_units(p, prefill)
        what = None
    units, work = units[:procs], work[:procs]
    for _ in range(args.warmup):
        oracle_rate(p, units[:1], work[:1], 1)
    t0 = time.perf_counter()
    done = 0.0
    for _ in range(args.steps):
        r, dt, _ = oracle_rate(p, units, work, procs)
        done += r * dt
    dt = time.perf_counter() - t0
    v = done / dt / div
    if what is None:
        what = f"{len(units)} of {p.S * p.Hkv} (slice, KV head) units per step" + (
            f", {len(units[0][2])} query rows each" if prefill else "")
    sample = f"{what}, fp64 oracle, {procs} processes"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": p.name},
        "cpu_baseline": {"value": round(v, 6), "unit": unit, "cores": procs, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# keys of a configs entry (the rest is the same as the headline line's)
CONFIG_KEYS = ("value", "unit", "ms_per_step", "dtype", "config", "roofline", "e2e", "gpu_launches", "clocks",
               "cpu_baseline")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=None, choices=WORKLOAD_CHOICES,
                    help="one workload alone (default: the bf16 decode, plus the other configurations on one GPU)")
    ap.add_argument("--no-configs", action="store_true", help="the headline workload alone")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=6.0, help="oracle time per workload (headline: 10 s)")
    ap.add_argument("--no-graph", action="store_true", help="time direct launches instead of CUDA-graph replays")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    explicit = args.workload is not None
    if not explicit:
        args.workload = "decode_bf16"

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    procs = os.cpu_count() or 1

    if args.workload == "kv_append_int8":
        if args.impl == "reference":
            if rank != 0:
                return
            append_oracle_rate(passes_wanted=args.warmup)
            v, dt, passes = append_oracle_rate(passes_wanted=args.steps)
            print(json.dumps({
                "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / passes * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
                "data": "synthetic", "config": {"workload": "kv-append int8 (oracle append_rows, bounded sample)"},
                "cpu_baseline": {"value": round(v, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                 "sample": f"2,048 rows into a 16,384-row pool x {passes} passes"},
                "e2e": {"value": round(v, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            }))
            return
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl")
        cpu_baseline = None
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            v, dt, passes = append_oracle_rate(10.0)
            cpu_baseline = {"value": round(v, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                            "sample": f"append_rows (int8) of 2,048 rows into a 16,384-row pool x {passes} passes, "
                                      f"{dt:.1f} s wall"}
        res = run_append(args, rank, world, cpu_baseline)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        if res is not None:
            print(json.dumps(res))
        return

    if args.impl == "reference":
        reference_arm(args, rank, world, procs)
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    # every problem is built and every oracle leg timed before the first CUDA
    # call (the oracle's worker pool is forked)
    names = [args.workload]
    if not explicit and world == 1 and not args.no_configs:
        names += CONFIG_WORKLOADS
    cache = {}
    problems = {n: build_problem(n, cache) for n in names}
    baselines = {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        for n in names:
            if n == "sparse_select_bf16":
                baselines[n] = None
                continue
            secs = 10.0 if n == names[0] else args.cpu_seconds
            baselines[n] = cpu_leg(problems[n], n, procs, secs)
    res = measure(args, rank, world, problems[names[0]], names[0], baselines.get(names[0]))
    configs = {}
    for n in names[1:]:
        r = measure(args, rank, world, problems[n], n, baselines.get(n))
        if r is not None:
            configs[n] = {k: r[k] for k in CONFIG_KEYS}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if res is not None:
        if configs:
            res["configs"] = configs
        print(json.dumps(res))


if __name__ == "__main__":
    main()
