"""Prefill parity: the tcgen05 kernel through the C ABI against the fp64
oracle.  Contiguous runs exercise the TMA path, shuffled pools and padding the
cp.async gather path; the full-size chunk is checked on sampled query rows."""
import numpy as np
import pytest
import torch

import oracle
import row_indexed_flash_gb300 as far
import synth
from helpers import assert_lse, assert_parity, dev_bits, oracle_for

pytestmark = pytest.mark.gpu


def run_prefill(p, out_dtype=torch.float32):
    q, k, v = dev_bits(p.q, p.dtype), dev_bits(p.k, p.dtype), dev_bits(p.v, p.dtype)
    rows = torch.from_numpy(p.kv_rows).cuda()
    extra = {}
    if p.kv_len is not None:
        extra["kv_len"] = torch.from_numpy(p.kv_len).cuda()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    out, lse = far.fa_rows_prefill(q, k, v, rows, p.scale, causal=p.causal, out_dtype=out_dtype, want_lse=True,
                                   workspace=ws, **extra)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0, "prefill pipeline wait expired"
    return out, lse


CASES = {
    "runs_tma_causal": lambda: synth.prefill_bf16(seed=11, n_seq=2, seq_rows=1500, pool_rows=4096, n_query=300,
                                                  run=256, Hq=8, Hkv=2),
    "runs_tma_g1": lambda: synth.prefill_bf16(seed=12, n_seq=2, seq_rows=700, pool_rows=2048, n_query=130,
                                              run=128, Hq=4, Hkv=4),
    "runs_tma_g8": lambda: synth.prefill_bf16(seed=13, n_seq=1, seq_rows=1200, pool_rows=2048, n_query=200,
                                              run=384, Hq=16, Hkv=2),
    "shuffled_gather": lambda: synth.prefill_bf16(seed=14, n_seq=3, seq_rows=900, pool_rows=3000, n_query=150,
                                                  Hq=8, Hkv=2, shuffled=True),
    "random_padding": lambda: synth.random_problem(15, S=2, Nq=100, Hq=8, Hkv=2, D=128, R=2000, L=700,
                                                   causal=True, pad_frac=0.15),
    "noncausal_kvlen": lambda: synth.random_problem(16, S=3, Nq=70, Hq=8, Hkv=2, D=128, R=2000, L=900,
                                                    kv_len=True, pad_frac=0.05),
    "f16": lambda: synth.random_problem(17, S=2, Nq=64, Hq=4, Hkv=1, D=128, R=1000, L=513, dtype="f16",
                                        causal=True, pad_frac=0.0),
    "one_query": lambda: synth.random_problem(18, S=2, Nq=1, Hq=8, Hkv=2, D=128, R=600, L=300, causal=True),
    "g16_partial_tiles": lambda: synth.random_problem(19, S=1, Nq=45, Hq=32, Hkv=2, D=128, R=1000, L=400,
                                                      causal=True),
    "g6_nonpow2": lambda: synth.random_problem(20, S=2, Nq=50, Hq=12, Hkv=2, D=128, R=1000, L=333, causal=True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_matches_oracle(name):
    p = CASES[name]()
    out, lse = run_prefill(p)
    ref, ref_lse = oracle_for(p)
    assert_parity(out, ref, name)
    assert_lse(lse, ref_lse, name)


@pytest.mark.parametrize("scale", [0.0, -0.08838834764831845, 0.05])
def test_prefill_scale_edge_cases_with_masks(scale):
    p = synth.random_problem(23, S=2, Nq=40, Hq=8, Hkv=2, D=128, R=1500, L=600, causal=True, pad_frac=0.2)
    p.scale = scale
    out, lse = run_prefill(p)
    ref, ref_lse = oracle_for(p)
    assert_parity(out, ref, f"scale {scale}")
    assert_lse(lse, ref_lse, f"scale {scale}")


def _times4(bits, dtype):
    """16-bit patterns of 4*x (exact: a power of two, no overflow for N(0,1) data)."""
    if dtype == "bf16":
        f = (bits.astype(np.uint32) << 16).view(np.float32) * np.float32(4)
        return (f.view(np.uint32) >> 16).astype(np.uint16)
    return (bits.view(np.float16) * np.float16(4)).view(np.uint16)


PEAKED_LAYOUTS = {
    "runs_tma": lambda dt: synth.prefill_bf16(seed=31, n_seq=2, seq_rows=1500, pool_rows=4096, n_query=300,
                                              run=256, Hq=8, Hkv=2, dtype=dt),
    "shuffled_gather": lambda dt: synth.prefill_bf16(seed=32, n_seq=2, seq_rows=1300, pool_rows=3000, n_query=260,
                                                     Hq=8, Hkv=2, shuffled=True, dtype=dt),
}


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("layout", sorted(PEAKED_LAYOUTS))
@pytest.mark.parametrize("peak", ["scale0.3", "scale0.5", "q_times4"])
def test_prefill_peaked_attention(peak, layout, dtype):
    """Concentrated attention (logit spreads of 3-6 standard deviations, a
    few rows taking most of the weight), where a P rounded once to bf16 would
    put about 2^-9 * |V| into the output: the same tolerance holds."""
    p = PEAKED_LAYOUTS[layout](dtype)
    if peak == "q_times4":
        p.q = _times4(p.q, dtype)
    else:
        p.scale = float(peak[5:])
    out, lse = run_prefill(p)
    ref, ref_lse = oracle_for(p)
    assert_parity(out, ref, f"{peak} {layout} {dtype}")
    assert_lse(lse, ref_lse, f"{peak} {layout} {dtype}")


def _bf16_times_pow2(bits, e):
    """16-bit patterns of x * 2^e for bf16 x (exact for N(0,1) data)."""
    f = (bits.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** e)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("layout", sorted(PEAKED_LAYOUTS))
@pytest.mark.parametrize("where", ["all_rows", "one_tile"])
def test_prefill_bf16_values_beyond_f16_range(where, layout):
    """bf16 V tiles go to f16 before PV unless a listed V value is finite and
    2^16 or more, which f16 cannot represent: the launch then keeps V in bf16
    and P as the bf16 pair.  With every V row times 2^17, out / 2^17 must
    match the oracle on the unscaled rows; with only the rows of one 128-entry
    tile of the first slice scaled, the rest of the launch has ordinary values
    (checked at |err| <= 2e-3 + 1e-4 * the softmax-weighted |V|: terms near
    2^17 meet in f32 sums)."""
    p = PEAKED_LAYOUTS[layout]("bf16")
    if where == "all_rows":
        ref, ref_lse = oracle_for(p)
        p.v = _bf16_times_pow2(p.v, 17)
        out, lse = run_prefill(p)
        assert_parity(out / 2.0 ** 17, ref, f"{where} {layout}")
        return
    rows = p.kv_rows[0, 256:384]
    rows = rows[rows >= 0]
    p.v[rows] = _bf16_times_pow2(p.v[rows], 17)
    ref, _ = oracle_for(p)
    # the softmax-weighted |V|: the size of the terms whose rounding is summed
    mag, _ = oracle_for(p, k=oracle.widen_bf16(p.k), v=np.abs(oracle.widen_bf16(p.v)))
    out, _ = run_prefill(p)
    g = out.double().cpu().numpy()
    assert np.all(np.isfinite(g))
    err = np.abs(g - ref)
    assert (err <= 2e-3 + 1e-4 * mag).all(), f"{where} {layout}: max err {err.max():.3e}"
    assert np.abs(ref[0]).max() > 2.0 ** 10, "the scaled rows must reach the first slice's output"


@pytest.mark.parametrize("odt", [torch.bfloat16, torch.float16])
def test_prefill_low_precision_outputs(odt):
    p = CASES["runs_tma_causal"]()
    out, _ = run_prefill(p, out_dtype=odt)
    ref, _ = oracle_for(p)
    assert_parity(out, ref, str(odt), out_dtype=odt)


def test_prefill_empty_slice_and_poisoned_unlisted_rows():
    p = synth.prefill_bf16(seed=21, n_seq=2, seq_rows=600, pool_rows=2048, n_query=100, run=128, Hq=8, Hkv=2)
    used = np.zeros(p.R, bool)
    used[p.kv_rows[p.kv_rows >= 0]] = True
    p.k[~used] = 0x7FC0
    p.v[~used] = 0x7FC0
    out, lse = run_prefill(p)
    ref, ref_lse = oracle_for(p)
    assert_parity(out, ref, "poisoned")
    p.kv_rows[1] = -1
    out, lse = run_prefill(p)
    assert torch.all(out[1] == 0) and torch.all(torch.isinf(lse[1]))


def test_prefill_agrees_with_decode_on_small_query_counts():
    p = synth.random_problem(22, S=3, Nq=2, Hq=8, Hkv=2, D=128, R=3000, L=2500, causal=True)
    a, _ = run_prefill(p)
    q, k, v = dev_bits(p.q, "bf16"), dev_bits(p.k, "bf16"), dev_bits(p.v, "bf16")
    b, _ = far.fa_rows_decode(q, k, v, torch.from_numpy(p.kv_rows).cuda(), p.scale, causal=True)
    assert_parity(a, b.double().cpu().numpy(), "prefill vs decode")


@pytest.mark.slow
def test_workload_prefill_full_size_sampled_rows():
    """The full chunk (4 x 2,048 query rows over 99,936-row lists) in the
    bench's launch configuration.  Slice 0: one query row in every 128-row
    query tile (with 32/8 heads a tile holds 32 positions, two tiles per CTA),
    at a different offset in each tile; every slice: its first and last rows."""
    p = synth.prefill_bf16()
    out, lse = run_prefill(p)
    G = p.Hq // p.Hkv
    pt = 128 // G
    per_tile = [t * pt + (7 * t) % pt for t in range((p.Nq + pt - 1) // pt)]
    rows0 = sorted(set(per_tile) | {0, p.Nq - 1})
    assert len(rows0) >= p.Nq // pt
    checks = [([0], rows0)] + [([s], [0, p.Nq - 1]) for s in range(1, p.S)]
    for sl, rows in checks:
        ref, ref_lse = oracle_for(p, query_rows=rows, slices=sl)
        assert_parity(out[sl][:, rows], ref, f"prefill full slice {sl}")
        assert_lse(lse[sl][:, rows], ref_lse, f"prefill full slice {sl}")
