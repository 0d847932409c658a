"""Decode parity: the CUDA split-KV kernel through the C ABI against the fp64
oracle, on small sweeps (several tiles, ragged tails, padding) and on the
full-size decode workloads."""
import numpy as np
import pytest
import torch

import oracle
import row_indexed_flash_gb300 as far
import synth
from helpers import assert_lse, assert_parity, dev_bits, oracle_for

pytestmark = pytest.mark.gpu


def run_decode(p, out_dtype=torch.float32, **kw):
    q, k, v = dev_bits(p.q, p.dtype), dev_bits(p.k, p.dtype), dev_bits(p.v, p.dtype)
    rows = torch.from_numpy(p.kv_rows).cuda()
    extra = {}
    if p.mask is not None:
        extra["mask"] = torch.from_numpy(p.mask).cuda()
    if p.kv_len is not None:
        extra["kv_len"] = torch.from_numpy(p.kv_len).cuda()
    out, lse = far.fa_rows_decode(q, k, v, rows, p.scale, causal=p.causal, out_dtype=out_dtype, want_lse=True,
                                  **extra, **kw)
    torch.cuda.synchronize()
    return out, lse


SWEEP = [
    dict(D=128, Hq=8, Hkv=2, L=1000, R=4096),
    dict(D=128, Hq=32, Hkv=8, L=777, R=3000, S=3),
    dict(D=256, Hq=16, Hkv=2, L=513, R=2000, S=1),
    dict(D=64, Hq=4, Hkv=4, L=200, R=500),
    dict(D=64, Hq=32, Hkv=1, L=300, R=500),
    dict(D=128, Hq=16, Hkv=1, L=90, R=200),
    dict(D=256, Hq=2, Hkv=1, L=4100, R=5000, S=1),
    dict(D=128, Hq=4, Hkv=2, L=33, R=100, Nq=4),
    dict(D=128, Hq=8, Hkv=8, L=5000, R=6000, S=2, Nq=3),
    dict(D=128, Hq=8, Hkv=2, L=2049, R=3000, dtype="f16"),
    dict(D=64, Hq=16, Hkv=2, L=1, R=10),
]


@pytest.mark.parametrize("i", range(len(SWEEP)))
def test_decode_sweep_matches_oracle(i):
    kw = dict(S=2, Nq=1, pad_frac=0.1)
    kw.update(SWEEP[i])
    p = synth.random_problem(1000 + i, **kw)
    out, lse = run_decode(p)
    ref, ref_lse = oracle_for(p)
    assert_parity(out, ref, f"sweep {i}")
    assert_lse(lse, ref_lse, f"sweep {i}")


@pytest.mark.parametrize("kw", [
    dict(with_mask=True),
    dict(with_mask=True, neg_inf_frac=0.5),
    dict(causal=True, Nq=4, Hq=8, Hkv=2),
    dict(kv_len=True),
    dict(kv_len=True, causal=True, Nq=2),
    dict(distinct=False),
    dict(pad_frac=0.9),
])
def test_decode_masks_lengths_and_duplicates(kw):
    base = dict(S=3, Nq=1, Hq=8, Hkv=2, D=128, R=2000, L=1500)
    base.update(kw)
    p = synth.random_problem(2000 + len(str(kw)), **base)
    out, lse = run_decode(p)
    ref, ref_lse = oracle_for(p)
    assert_parity(out, ref, str(kw))
    assert_lse(lse, ref_lse, str(kw))


@pytest.mark.parametrize("odt", [torch.bfloat16, torch.float16])
def test_decode_low_precision_outputs(odt):
    p = synth.random_problem(3000, S=2, Hq=8, Hkv=2, D=128, R=1000, L=700)
    out, _ = run_decode(p, out_dtype=odt)
    ref, _ = oracle_for(p)
    assert out.dtype == odt
    assert_parity(out, ref, str(odt), out_dtype=odt)


def test_decode_empty_lists_give_zero_and_minus_inf():
    p = synth.random_problem(3100, S=3, Hq=8, Hkv=2, D=128, R=500, L=300)
    p.kv_rows[1] = -1
    out, lse = run_decode(p)
    assert torch.all(out[1] == 0) and torch.all(torch.isinf(lse[1]))
    ref, ref_lse = oracle_for(p)
    assert_parity(out, ref)
    assert_lse(lse, ref_lse)


def test_unlisted_rows_are_never_read_even_when_poisoned():
    p = synth.random_problem(3200, S=2, Hq=8, Hkv=2, D=128, R=3000, L=1200, pad_frac=0.2)
    used = np.zeros(p.R, bool)
    used[p.kv_rows[p.kv_rows >= 0]] = True
    k, v = p.k.copy(), p.v.copy()
    k[~used] = 0x7FC0   # bf16 NaN
    v[~used] = 0x7FC0
    clean, _ = run_decode(p)
    p.k, p.v = k, v
    dirty, _ = run_decode(p)
    assert torch.equal(clean, dirty)


def test_out_of_range_rows_are_skipped_like_padding_and_reported():
    p = synth.random_problem(3300, S=2, Hq=8, Hkv=2, D=128, R=1000, L=400, pad_frac=0.0)
    bad = p.kv_rows.copy()
    bad[0, 5] = p.R + 7
    bad[1, 100] = 2 ** 31 - 1
    p2 = synth.Problem(**{**p.__dict__, "kv_rows": bad})
    out, _ = run_decode(p2)
    fixed = bad.copy()
    fixed[fixed >= p.R] = -1
    ref, _ = oracle_for(p, kv_rows=fixed)
    assert_parity(out, ref)
    cnt, first = far.fa_rows_validate(torch.from_numpy(bad).cuda(), p.R)
    assert (cnt, first) == (2, 5)
    assert far.fa_rows_validate(torch.from_numpy(p.kv_rows).cuda(), p.R) == (0, -1)


@pytest.mark.parametrize("hq,hkv,dtype,causal", [(8, 2, "bf16", False), (16, 1, "bf16", True), (32, 1, "bf16", False),
                                                 (8, 2, "f16", False)])
def test_decode_contiguous_runs(hq, hkv, dtype, causal):
    """Lists made of contiguous pool runs (whole 64-entry tiles of one run take
    the tile-load path, the rest are gathered), with a ragged padded tail."""
    S, L, R = 2, 1500, 6000
    p = synth.random_problem(3500 + hq, S=S, Nq=1, Hq=hq, Hkv=hkv, D=128, R=R, L=L, dtype=dtype, pad_frac=0.0,
                             causal=causal)
    g = np.random.default_rng(11 + hq)
    rows = np.empty((S, L), np.int32)
    rows[0] = 1000 + np.arange(L)                 # one run: every full tile is contiguous
    pos = 0
    while pos < L:                                # runs of 20..300 rows at random starts
        n = min(int(g.integers(20, 300)), L - pos)
        start = int(g.integers(0, R - n))
        rows[1, pos:pos + n] = start + np.arange(n)
        pos += n
    rows[:, -37:] = -1
    p2 = synth.Problem(**{**p.__dict__, "kv_rows": rows})
    out, lse = run_decode(p2)
    ref, ref_lse = oracle_for(p2)
    assert_parity(out, ref, f"runs hq={hq} hkv={hkv} {dtype} causal={causal}")
    assert_lse(lse, ref_lse)


def test_repeated_calls_are_identical_and_split_plans_agree():
    p = synth.random_problem(3400, S=4, Hq=32, Hkv=8, D=128, R=40000, L=16000, pad_frac=0.0)
    a, _ = run_decode(p)
    b, _ = run_decode(p)
    assert torch.equal(a, b)                       # the split counters were reset
    c, _ = run_decode(p, n_valid_hint=100)         # a different split plan
    assert_parity(c, a.double().cpu().numpy())


def _decode_launches(p):
    import ctypes
    q, k, v = dev_bits(p.q, p.dtype), dev_bits(p.k, p.dtype), dev_bits(p.v, p.dtype)
    kw = {} if p.kv_len is None else {"kv_len": torch.from_numpy(p.kv_len).cuda()}
    a, _, _ = far.make_args(q, k, v, torch.from_numpy(p.kv_rows).cuda(), p.scale, causal=p.causal, **kw)
    return far.lib().fa_rows_decode_launches(ctypes.byref(a))


@pytest.mark.parametrize("kw,launches", [
    (dict(S=1, Hq=16, Hkv=2, D=256, R=4096, L=2048), 2),                      # the sparse shape: 16 splits
    (dict(S=3, Hq=8, Hkv=2, D=128, R=8192, L=600, kv_len=True), 2),          # short slices write directly
    (dict(S=2, Hq=32, Hkv=8, D=128, R=9000, L=300, causal=True, Nq=1), 2),
    (dict(S=4, Hq=32, Hkv=8, D=128, R=40000, L=16000), 1),                    # long chunks: merged in the decode
])
def test_split_merge_in_the_decode_and_as_its_own_kernel(kw, launches):
    """Both places the splits of a (slice, KV head) are merged: by the last
    CTA of the decode, or (a latency-bound 16-bit decode) by a merge kernel
    after it.  Parity with the oracle, and a repeated call bit-identical."""
    p = synth.random_problem(3500 + launches + kw["L"], **kw)
    assert _decode_launches(p) == launches
    out, lse = run_decode(p)
    ref, ref_lse = oracle_for(p)
    assert_parity(out, ref, f"merge path {launches}")
    assert_lse(lse, ref_lse)
    out2, lse2 = run_decode(p)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


# --- full-size decode workloads ------------------------------------------------


def test_workload_decode_f16_small():
    p = synth.decode_fp16_small()
    out, lse = run_decode(p)
    ref, ref_lse = oracle_for(p)
    assert_parity(out, ref, "decode_f16_small")
    assert_lse(lse, ref_lse)


def test_workload_decode_bf16_4x16384():
    p = synth.decode_bf16_large()
    out, lse = run_decode(p)
    ref, ref_lse = oracle_for(p)
    assert_parity(out, ref, "decode_bf16")
    assert_lse(lse, ref_lse)


def test_workload_sparse_bf16_d256():
    p = synth.sparse_bf16()
    out, lse = run_decode(p)
    ref, ref_lse = oracle_for(p)
    assert_parity(out, ref, "sparse_bf16")
    assert_lse(lse, ref_lse)
