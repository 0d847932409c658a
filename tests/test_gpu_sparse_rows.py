"""The sparse row-list builder (sinks + top-k by score + recent) against the
oracle's, entry for entry, and the list it builds fed to decode."""
import numpy as np
import pytest
import torch

import oracle
import synth
import row_indexed_flash_gb300 as far

from helpers import assert_parity, dev_bits, oracle_for

pytestmark = pytest.mark.gpu


def _scores(seed, S, n, ties=False, nan_frac=0.0, signed_zeros=False):
    g = synth.rng(seed)
    if ties:
        sc = g.integers(-3, 4, size=(S, n)).astype(np.float32)
    else:
        sc = g.standard_normal((S, n)).astype(np.float32)
    if signed_zeros:
        # mostly zeros of both signs, so the k-th largest score is a zero
        sc = np.where(g.random((S, n)) < 0.9, np.float32(0.0), sc)
        sc = np.where((sc == 0) & (g.random((S, n)) < 0.5), np.float32(-0.0), sc)
    if nan_frac:
        sc[g.random((S, n)) < nan_frac] = np.nan
    return sc


@pytest.mark.parametrize("ws", ["auto", None])
@pytest.mark.parametrize("case", [
    dict(S=3, n=1000, sinks=4, recent=16, k=37, ties=True),
    dict(S=2, n=5000, sinks=0, recent=0, k=100),
    dict(S=4, n=3000, sinks=4, recent=64, k=200, nan_frac=0.1),
    dict(S=2, n=700, sinks=8, recent=8, k=0),
    dict(S=2, n=50, sinks=8, recent=8, k=100),                       # fewer middle positions than k
    dict(S=5, n=2000, sinks=4, recent=32, k=64, ties=True, n_len=True),
    dict(S=1, n=1, sinks=4, recent=4, k=4),
    dict(S=3, n=4099, sinks=3, recent=5, k=77, ties=True),           # rows not 16-byte aligned
    dict(S=1, n=70001, sinks=5, recent=7, k=1000, nan_frac=0.01),
    dict(S=3, n=3000, sinks=4, recent=16, k=500, signed_zeros=True),      # the k-th score is a +-0 tie
    dict(S=2, n=20000, sinks=1, recent=1, k=4000, signed_zeros=True, ties=True),
])
def test_sparse_rows_match_oracle(case, ws):
    S, n = case["S"], case["n"]
    sc = _scores(100 + S + n, S, n, case.get("ties", False), case.get("nan_frac", 0.0),
                 case.get("signed_zeros", False))
    if case.get("signed_zeros"):
        # the case must actually mix signs among the zeros it selects from
        assert (np.signbit(sc) & (sc == 0)).any() and (~np.signbit(sc) & (sc == 0)).any()
    n_len = None
    if case.get("n_len"):
        n_len = synth.rng(5).integers(0, n + 1, size=S).astype(np.int32)
    L = case["sinks"] + case["recent"] + case["k"] + 3   # some padding
    want = oracle.select_rows(sc, case["sinks"], case["recent"], case["k"], L, n_len=n_len)
    got = far.fa_kv_sparse_rows(torch.from_numpy(sc).cuda(), case["sinks"], case["recent"], case["k"], L,
                                n_len=None if n_len is None else torch.from_numpy(n_len).cuda(), workspace=ws)
    assert np.array_equal(got.cpu().numpy(), want)


def test_sparse_rows_with_a_row_map():
    S, n = 2, 4000
    sc = _scores(7, S, n, ties=True)
    row_map = np.stack([synth.rng(8 + s).permutation(1 << 16)[:n] for s in range(S)]).astype(np.int32)
    want = oracle.select_rows(sc, 4, 64, 128, 196, row_map=row_map)
    got = far.fa_kv_sparse_rows(torch.from_numpy(sc).cuda(), 4, 64, 128, 196, row_map=torch.from_numpy(row_map).cuda())
    assert np.array_equal(got.cpu().numpy(), want)


def test_sparse_rows_at_the_sparse_workload_size_then_decode():
    # 262,144 positions, 4 sinks, 512 recent, 1,532 by score: the sparse decode workload's list shape
    p = synth.sparse_bf16()
    sc = _scores(9, 1, p.R)
    want = oracle.select_rows(sc, 4, 512, 1532, 2048)
    rows = far.fa_kv_sparse_rows(torch.from_numpy(sc).cuda(), 4, 512, 1532)
    assert np.array_equal(rows.cpu().numpy(), want)
    assert np.array_equal(far.fa_kv_sparse_rows(torch.from_numpy(sc).cuda(), 4, 512, 1532, workspace=None).cpu().numpy(),
                          want)
    out, _ = far.fa_rows_decode(dev_bits(p.q, "bf16"), dev_bits(p.k, "bf16"), dev_bits(p.v, "bf16"), rows, p.scale)
    ref, _ = oracle_for(p, kv_rows=want)
    assert_parity(out, ref, "built sparse list")


def test_sparse_rows_reject_a_short_list_and_a_short_workspace():
    sc = torch.zeros((1, 100), dtype=torch.float32, device="cuda")
    with pytest.raises(far.FaRowsError):
        far.fa_kv_sparse_rows(sc, 4, 4, 10, list_len=17)
    with pytest.raises(far.FaRowsError):
        far.fa_kv_sparse_rows(sc, 4, 4, 10, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
