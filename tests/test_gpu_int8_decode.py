"""INT8 pools through decode: codes and scales made on the device, checked
bit-exactly against the oracle's quantiser, then attention over the
dequantised rows compared with the fp64 oracle.

Covers the tensor-core path (D 128/256, 1..32 query vectors per KV head, f16
and bf16 queries, causal query rows, per-slice lengths, split merges) and the
CUDA-core path it leaves to (D 64, dense masks)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import row_indexed_flash_gb300 as far

from helpers import assert_lse, assert_parity, dev_bits, oracle_for

pytestmark = pytest.mark.gpu

CASES = {
    # name: random_problem kwargs (R a multiple of 64: the scale layout is paged)
    "d128_g4": dict(S=3, Nq=1, Hq=32, Hkv=8, D=128, R=320, L=77),
    "d128_g1_f16": dict(S=2, Nq=1, Hq=8, Hkv=8, D=128, R=256, L=130, dtype="f16"),
    "d256_g8": dict(S=2, Nq=1, Hq=16, Hkv=2, D=256, R=448, L=200),
    "d128_causal_nq4": dict(S=2, Nq=4, Hq=8, Hkv=2, D=128, R=384, L=150, causal=True),
    "d128_g32": dict(S=1, Nq=1, Hq=32, Hkv=1, D=128, R=256, L=96),
    "d128_kvlen_splits": dict(S=3, Nq=1, Hq=8, Hkv=2, D=128, R=8192, L=5000, kv_len=True),
    "d256_f16_causal_nq2": dict(S=2, Nq=2, Hq=16, Hkv=2, D=256, R=512, L=333, causal=True, dtype="f16"),
    "d64_cuda_core": dict(S=2, Nq=1, Hq=8, Hkv=2, D=64, R=256, L=90),
    "d128_dense_mask_cuda_core": dict(S=2, Nq=2, Hq=8, Hkv=2, D=128, R=256, L=70, with_mask=True, neg_inf_frac=0.2),
}


def _quantised(p):
    """Device INT8 pools of p, checked against the oracle's codec, and the
    oracle's dequantised float64 pools."""
    kq, ks = far.fa_kv_quantize_int8(dev_bits(p.k, p.dtype), p.R)
    vq, vs = far.fa_kv_quantize_int8(dev_bits(p.v, p.dtype), p.R)
    okq, oks = oracle.quantize_int8(oracle.widen(p.k, p.dtype).astype(np.float32))
    ovq, ovs = oracle.quantize_int8(oracle.widen(p.v, p.dtype).astype(np.float32))
    assert np.array_equal(kq.cpu().numpy(), okq) and np.array_equal(vq.cpu().numpy(), ovq)
    assert np.array_equal(ks.cpu().numpy().view(np.uint16), oracle.pack_scales(oks).view(np.uint16))
    assert np.array_equal(vs.cpu().numpy().view(np.uint16), oracle.pack_scales(ovs).view(np.uint16))
    kd = oracle.dequantize_int8(okq, oks).astype(np.float64)
    vd = oracle.dequantize_int8(ovq, ovs).astype(np.float64)
    return (kq, ks, vq, vs), (kd, vd)


def _poison_unlisted(p, kq, ks, vq, vs):
    """Saturate the codes and put NaN in the scales of every row no list names."""
    listed = np.zeros(p.R, bool)
    listed[p.kv_rows[p.kv_rows >= 0]] = True
    free = np.nonzero(~listed)[0]
    if free.size == 0:
        return
    idx = torch.from_numpy(free).cuda()
    kq[idx] = 127
    vq[idx] = -127
    nan = torch.tensor(float("nan"), dtype=torch.float16, device="cuda")
    pages, offs = idx // 64, idx % 64
    for h in range(p.Hkv):
        ks[pages, h, offs] = nan
        vs[pages, h, offs] = nan


def _run(p, pools, **kw):
    kq, ks, vq, vs = pools
    q = dev_bits(p.q, p.dtype)
    rows = torch.from_numpy(p.kv_rows).cuda()
    extra = {}
    if p.kv_len is not None:
        extra["kv_len"] = torch.from_numpy(p.kv_len).cuda()
    if p.mask is not None:
        extra["mask"] = torch.from_numpy(p.mask).cuda()
    return far.fa_rows_decode(q, kq, vq, rows, p.scale, k_scale=ks, v_scale=vs, causal=p.causal, want_lse=True,
                              **extra, **kw)


@pytest.mark.parametrize("name", sorted(CASES))
def test_int8_decode_matches_oracle(name):
    p = synth.random_problem(11 + sorted(CASES).index(name), **CASES[name])
    pools, (kd, vd) = _quantised(p)
    _poison_unlisted(p, *pools)
    out, lse = _run(p, pools)
    ref, ref_lse = oracle_for(p, k=kd, v=vd)
    assert_parity(out, ref, f"int8 {name}")
    assert_lse(lse, ref_lse)


def test_int8_decode_low_precision_outputs():
    p = synth.random_problem(41, S=2, Nq=1, Hq=16, Hkv=4, D=128, R=256, L=100)
    pools, (kd, vd) = _quantised(p)
    ref, _ = oracle_for(p, k=kd, v=vd)
    for dt in (torch.bfloat16, torch.float16):
        out, _ = _run(p, pools, out_dtype=dt)
        assert_parity(out, ref, f"int8 out {dt}", out_dtype=dt)


def test_int8_decode_empty_and_all_padding_slices():
    p = synth.random_problem(43, S=3, Nq=1, Hq=8, Hkv=2, D=128, R=256, L=64)
    p.kv_rows[1, :] = -1
    pools, (kd, vd) = _quantised(p)
    out, lse = _run(p, pools)
    ref, ref_lse = oracle_for(p, k=kd, v=vd)
    assert_parity(out, ref, "int8 padding slice")
    assert np.all(out[1].cpu().numpy() == 0.0) and np.all(np.isneginf(lse[1].cpu().numpy()))
    assert_lse(lse, ref_lse)
