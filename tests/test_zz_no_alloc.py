"""fa_rows_decode_static: decode for callers that cannot allocate device memory
(for example code running inside a custom device allocator, or a plugin whose
framework owns every device allocation).  It takes its scratch from a static
device array in the library instead of a caller workspace.

Collected last on purpose, so that a run stopping at the first failure has
already run every other test.  Compares both against fa_rows_decode and
against the fp64 oracle, with the parity tolerance of the other decode tests,
on two calls in a row (the second call sees the array as the first call left
it)."""
import ctypes

import pytest
import torch

import row_indexed_flash_gb300 as far
import synth
from helpers import assert_lse, assert_parity, dev_bits, oracle_for

pytestmark = pytest.mark.gpu


def _device_problem(p):
    q, k, v = dev_bits(p.q, p.dtype), dev_bits(p.k, p.dtype), dev_bits(p.v, p.dtype)
    return q, k, v, torch.from_numpy(p.kv_rows).cuda()


def test_static_scratch_decode_matches_workspace_decode_on_two_calls():
    p = synth.random_problem(4242, S=4, Nq=1, Hq=32, Hkv=8, D=128, R=40000, L=16000, pad_frac=0.05)
    q, k, v, rows = _device_problem(p)
    ref, ref_lse = far.fa_rows_decode(q, k, v, rows, p.scale, want_lse=True)
    torch.cuda.synchronize()
    o_ref, o_lse = oracle_for(p)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        a, out, lse = far.make_args(q, k, v, rows, p.scale, want_lse=True)
        st = far.lib().fa_rows_decode_static(ctypes.byref(a), stream)
        assert st == 0, far.fa_last_error()
        torch.cuda.synchronize()
        assert_parity(out, ref.double().cpu().numpy(), f"static-scratch call {call}")
        assert_parity(lse, ref_lse.double().cpu().numpy(), f"static-scratch lse {call}")
        assert_parity(out, o_ref, f"static-scratch call {call} against the oracle")
        assert_lse(lse, o_lse, f"static-scratch lse {call} against the oracle")


def test_static_scratch_decode_rejects_plans_larger_than_the_array():
    # D 64 lists of 131,072 entries: at most 2,048 entries per CTA, so at least
    # 64 splits of 4 query vectors for each of 512 (slice, KV head) pairs
    p = synth.random_problem(4243, S=64, Nq=1, Hq=32, Hkv=8, D=64, R=131072, L=131072, pad_frac=0.0)
    q, k, v, rows = _device_problem(p)
    a, out, _ = far.make_args(q, k, v, rows, p.scale)
    need = far.fa_rows_workspace_size(a)
    assert need > 16 << 20
    st = far.lib().fa_rows_decode_static(ctypes.byref(a), torch.cuda.current_stream().cuda_stream)
    assert st == far.FaRowsError(3, "").status
    assert "16777216" in far.fa_last_error()
