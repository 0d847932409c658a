"""INT4 pools (the v100llm article's paged INT4 KV): the device codec against
the oracle's, bit for bit, then decode over the dequantised rows against the
fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import row_indexed_flash_gb300 as far

from helpers import assert_lse, assert_parity, dev_bits, oracle_for

pytestmark = pytest.mark.gpu

CASES = {
    "g4": dict(S=3, Nq=1, Hq=32, Hkv=8, D=128, R=320, L=77),
    "g1_f16": dict(S=2, Nq=1, Hq=8, Hkv=8, D=128, R=256, L=130, dtype="f16"),
    "causal_nq4": dict(S=2, Nq=4, Hq=8, Hkv=2, D=128, R=384, L=150, causal=True),
    "g32": dict(S=1, Nq=1, Hq=32, Hkv=1, D=128, R=256, L=96),
    "kvlen_splits": dict(S=3, Nq=1, Hq=8, Hkv=2, D=128, R=8192, L=5000, kv_len=True),
}


def _quantised(p):
    kq, ks = far.fa_kv_quantize_int4(dev_bits(p.k, p.dtype), p.R)
    vq, vs = far.fa_kv_quantize_int4(dev_bits(p.v, p.dtype), p.R)
    okq, oks = oracle.quantize_int4(oracle.widen(p.k, p.dtype).astype(np.float32))
    ovq, ovs = oracle.quantize_int4(oracle.widen(p.v, p.dtype).astype(np.float32))
    assert np.array_equal(kq.cpu().numpy(), okq) and np.array_equal(vq.cpu().numpy(), ovq)
    assert np.array_equal(ks.cpu().numpy().view(np.uint16), oracle.pack_scales(oks).view(np.uint16))
    assert np.array_equal(vs.cpu().numpy().view(np.uint16), oracle.pack_scales(ovs).view(np.uint16))
    kd = oracle.dequantize_int4(okq, oks).astype(np.float64)
    vd = oracle.dequantize_int4(ovq, ovs).astype(np.float64)
    return (kq, ks, vq, vs), (kd, vd)


def _run(p, pools, **kw):
    kq, ks, vq, vs = pools
    extra = {}
    if p.kv_len is not None:
        extra["kv_len"] = torch.from_numpy(p.kv_len).cuda()
    return far.fa_rows_decode(dev_bits(p.q, p.dtype), kq, vq, torch.from_numpy(p.kv_rows).cuda(), p.scale,
                              k_scale=ks, v_scale=vs, causal=p.causal, want_lse=True, **extra, **kw)


def test_int4_codec_is_bit_exact_and_dequantises_exactly():
    bits = synth.normal_bits(synth.rng(31), (256, 4, 128), "bf16")
    x = dev_bits(bits, "bf16")
    q, s = far.fa_kv_quantize_int4(x, 256)
    oq, os_ = oracle.quantize_int4(oracle.widen_bf16(bits).astype(np.float32))
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), oracle.pack_scales(os_).view(np.uint16))
    deq = far.fa_kv_dequantize_int4(q, s).cpu().numpy()
    assert np.array_equal(deq.view(np.uint32), oracle.dequantize_int4(oq, os_).view(np.uint32))


def test_int4_append_writes_named_rows_only():
    R, H, D, n = 192, 2, 128, 40
    bits = synth.normal_bits(synth.rng(32), (n, H, D), "f16")
    dst = synth.rng(33).permutation(R)[:n].astype(np.int32)
    dst[::7] = -1
    q, s = far.fa_kv_quantize_int4(dev_bits(bits, "f16"), R, dst_rows=torch.from_numpy(dst).cuda())
    oq, os_ = oracle.quantize_int4(oracle.widen_f16(bits).astype(np.float32))
    qn, sn = q.cpu().numpy(), oracle.unpack_scales(s.cpu().numpy().view(np.float16))
    for i, r in enumerate(dst):
        if r >= 0:
            assert np.array_equal(qn[r], oq[i]) and np.array_equal(sn[r], os_[i])
    untouched = np.setdiff1d(np.arange(R), dst[dst >= 0])
    assert not qn[untouched].any()


@pytest.mark.parametrize("name", sorted(CASES))
def test_int4_decode_matches_oracle(name):
    p = synth.random_problem(51 + sorted(CASES).index(name), **CASES[name])
    pools, (kd, vd) = _quantised(p)
    out, lse = _run(p, pools)
    ref, ref_lse = oracle_for(p, k=kd, v=vd)
    assert_parity(out, ref, f"int4 {name}")
    assert_lse(lse, ref_lse)


def test_paged_int4_decode_small():
    p = synth.paged_int8(n_seq=6, lo=100, hi=9000)   # the paged layout; the pool is quantised to INT4 here
    rows_np = oracle.page_table_to_rows(p.page_table, p.seq_len, p.L)
    rows = far.fa_kv_page_table_to_rows(torch.from_numpy(p.page_table).cuda(), torch.from_numpy(p.seq_len).cuda(), p.L)
    kq, ks = far.fa_kv_quantize_int4(dev_bits(p.k, "bf16"), p.R)
    vq, vs = far.fa_kv_quantize_int4(dev_bits(p.v, "bf16"), p.R)
    out, lse = far.fa_rows_decode(dev_bits(p.q, "bf16"), kq, vq, rows, p.scale, k_scale=ks, v_scale=vs, want_lse=True,
                                  kv_len=torch.from_numpy(p.seq_len).cuda(), n_valid_hint=int(p.seq_len.sum()))
    used = np.unique(rows_np[rows_np >= 0])
    okq, oks = oracle.quantize_int4(oracle.widen_bf16(p.k[used]).astype(np.float32))
    ovq, ovs = oracle.quantize_int4(oracle.widen_bf16(p.v[used]).astype(np.float32))
    remap = np.full(p.R, -1, np.int64)
    remap[used] = np.arange(used.size)
    r2 = np.where(rows_np >= 0, remap[np.maximum(rows_np, 0)], -1).astype(np.int32)
    ref, ref_lse = oracle.attend_rows(oracle.widen_bf16(p.q), oracle.dequantize_int4(okq, oks).astype(np.float64),
                                      oracle.dequantize_int4(ovq, ovs).astype(np.float64), r2, p.scale)
    assert_parity(out, ref, "paged int4")
    assert_lse(lse, ref_lse)


def test_int4_is_refused_where_it_is_not_built():
    p = synth.random_problem(60, S=1, Nq=1, Hq=4, Hkv=2, D=64, R=128, L=10)
    kq, ks = far.fa_kv_quantize_int4(dev_bits(p.k, "bf16"), p.R)
    with pytest.raises(far.FaRowsError):
        far.fa_rows_decode(dev_bits(p.q, "bf16"), kq, kq, torch.from_numpy(p.kv_rows).cuda(), p.scale,
                           k_scale=ks, v_scale=ks)
