"""Bounded pipeline waits and the workspace status word.

Every wait in the tensor-core kernels gives up after a time limit; the kernel
then leaves its pipeline, drains its own copies and MMAs, frees its tensor
memory and sets FA_WS_WAIT_EXPIRED in the workspace's status word.  Here the
limit is lowered to 1 ns (fa_set_wait_limit_ns), so the waits run out on
purpose, with no fault and no trap.  Each case checks that the word is set,
that the decode split counters are back at zero after the aborted call, and
that, with the default limit restored, the next call on the same workspace
clears nothing it should not and matches the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import row_indexed_flash_gb300 as far
import synth
from helpers import assert_lse, assert_parity, dev_bits, oracle_for

pytestmark = pytest.mark.gpu


def _decode_bf16():
    p = synth.random_problem(901, S=2, Nq=1, Hq=8, Hkv=2, D=128, R=20000, L=8192, pad_frac=0.02)
    q, k, v = dev_bits(p.q, "bf16"), dev_bits(p.k, "bf16"), dev_bits(p.v, "bf16")
    rows = torch.from_numpy(p.kv_rows).cuda()

    def call(ws):
        return far.fa_rows_decode(q, k, v, rows, p.scale, want_lse=True, workspace=ws)

    def ref():
        return oracle_for(p)
    return p, call, ref, False


def _decode_int8():
    p = synth.random_problem(902, S=2, Nq=1, Hq=8, Hkv=2, D=128, R=20032, L=8192, pad_frac=0.02)
    q = dev_bits(p.q, "bf16")
    kq, ks = far.fa_kv_quantize_int8(dev_bits(p.k, "bf16"), p.R)
    vq, vs = far.fa_kv_quantize_int8(dev_bits(p.v, "bf16"), p.R)
    rows = torch.from_numpy(p.kv_rows).cuda()

    def call(ws):
        return far.fa_rows_decode(q, kq, vq, rows, p.scale, k_scale=ks, v_scale=vs, want_lse=True, workspace=ws)

    def ref():
        okq, oks = oracle.quantize_int8(oracle.widen_bf16(p.k).astype(np.float32))
        ovq, ovs = oracle.quantize_int8(oracle.widen_bf16(p.v).astype(np.float32))
        return oracle_for(p, k=oracle.dequantize_int8(okq, oks).astype(np.float64),
                          v=oracle.dequantize_int8(ovq, ovs).astype(np.float64))
    return p, call, ref, False


def _prefill_bf16():
    p = synth.prefill_bf16(seed=903, n_seq=2, seq_rows=1500, pool_rows=4096, n_query=300, run=256, Hq=8, Hkv=2)
    q, k, v = dev_bits(p.q, "bf16"), dev_bits(p.k, "bf16"), dev_bits(p.v, "bf16")
    rows = torch.from_numpy(p.kv_rows).cuda()

    def call(ws):
        return far.fa_rows_prefill(q, k, v, rows, p.scale, causal=True, want_lse=True, workspace=ws)

    def ref():
        return oracle_for(p)
    return p, call, ref, True


CASES = {"decode_bf16": _decode_bf16, "decode_int8": _decode_int8, "prefill_bf16": _prefill_bf16}


@pytest.mark.parametrize("name", sorted(CASES))
def test_expired_waits_set_the_status_word_and_leave_the_workspace_usable(name):
    p, call, ref, is_prefill = CASES[name]()
    # zero-filled once; 4 MiB covers these plans (at most 128 splits of 4 x 128 fp32 partials per unit)
    ws = torch.zeros(4 << 20, dtype=torch.uint8, device="cuda")
    units = p.S * p.Hkv
    hit = False
    try:
        far.fa_set_wait_limit_ns(1)
        for _ in range(4):
            call(ws)
            torch.cuda.synchronize()
            word = far.fa_rows_status(ws, clear=True)
            assert word & ~far.FA_WS_WAIT_EXPIRED == 0, hex(word)
            if not is_prefill:
                # every split arrived, aborted or not, and the last arrival reset the counter
                counters = ws[256:256 + 4 * units].view(torch.int32).cpu().numpy()
                assert not counters.any(), counters
            if word & far.FA_WS_WAIT_EXPIRED:
                hit = True
                break
    finally:
        far.fa_set_wait_limit_ns(0)
    assert hit, "no wait ran out with a 1 ns limit"
    assert far.fa_rows_status(ws) == 0      # cleared by the read above
    out, lse = call(ws)
    torch.cuda.synchronize()
    assert far.fa_rows_status(ws) == 0, "a wait ran out with the default limit"
    r, r_lse = ref()
    assert_parity(out, r, f"{name} after an aborted call")
    assert_lse(lse, r_lse, f"{name} after an aborted call")


def test_check_status_raises_on_an_expired_wait_and_clears_the_word():
    p, call, ref, _ = _decode_bf16()
    q, k, v = dev_bits(p.q, "bf16"), dev_bits(p.k, "bf16"), dev_bits(p.v, "bf16")
    rows = torch.from_numpy(p.kv_rows).cuda()
    raised = False
    try:
        far.fa_set_wait_limit_ns(1)
        for _ in range(4):
            try:
                far.fa_rows_decode(q, k, v, rows, p.scale, check_status=True)
            except far.FaRowsError as e:
                assert e.status == 6 and "FA_ERR_WAIT_EXPIRED" in str(e)
                raised = True
                break
    finally:
        far.fa_set_wait_limit_ns(0)
    assert raised
    out, _ = far.fa_rows_decode(q, k, v, rows, p.scale, check_status=True)
    assert_parity(out, ref()[0], "decode after a raised expiry")


def test_prefill_refuses_a_missing_workspace():
    p = synth.random_problem(904, S=1, Nq=16, Hq=8, Hkv=2, D=128, R=512, L=300, causal=True)
    a, _, _ = far.make_args(dev_bits(p.q, "bf16"), dev_bits(p.k, "bf16"), dev_bits(p.v, "bf16"),
                            torch.from_numpy(p.kv_rows).cuda(), p.scale, causal=True)
    import ctypes
    st = far.lib().fa_rows_prefill(ctypes.byref(a), None, 0, torch.cuda.current_stream().cuda_stream)
    assert st == 3 and "status word" in far.fa_last_error()
