"""FP8 E4M3 pools: the device codec against the oracle's, bit for bit, then
decode over the dequantised rows against the fp64 oracle."""
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


def _codes(t):
    return t.view(torch.uint8).cpu().numpy()


def _quantised(p):
    kq, ks = far.fa_kv_quantize_fp8(dev_bits(p.k, p.dtype), p.R)
    vq, vs = far.fa_kv_quantize_fp8(dev_bits(p.v, p.dtype), p.R)
    okq, oks = oracle.quantize_fp8(oracle.widen(p.k, p.dtype).astype(np.float32))
    ovq, ovs = oracle.quantize_fp8(oracle.widen(p.v, p.dtype).astype(np.float32))
    assert np.array_equal(_codes(kq), okq) and np.array_equal(_codes(vq), ovq)
    assert np.array_equal(ks.cpu().numpy().view(np.uint16), oracle.pack_scales(oks).view(np.uint16))
    kd = oracle.dequantize_fp8(okq, oks).astype(np.float64)
    vd = oracle.dequantize_fp8(ovq, ovs).astype(np.float64)
    return (kq, ks, vq, vs), (kd, vd)


def test_fp8_codec_is_bit_exact_including_saturation():
    g = synth.rng(41)
    bits = synth.normal_bits(g, (256, 4, 128), "bf16")
    # a few rows with one huge element (everything else goes subnormal in E4M3)
    wide = oracle.widen_bf16(bits).astype(np.float32)
    wide[::17, 0, 3] = 3.0e4
    bits = synth.f32_to_bf16_bits(wide)
    x = dev_bits(bits, "bf16")
    q, s = far.fa_kv_quantize_fp8(x, 256)
    oq, os_ = oracle.quantize_fp8(oracle.widen_bf16(bits).astype(np.float32))
    assert np.array_equal(_codes(q), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), oracle.pack_scales(os_).view(np.uint16))
    deq = far.fa_kv_dequantize_fp8(q, s).cpu().numpy()
    assert np.array_equal(deq.view(np.uint32), oracle.dequantize_fp8(oq, os_).view(np.uint32))


@pytest.mark.parametrize("name", sorted(CASES))
def test_fp8_decode_matches_oracle(name):
    p = synth.random_problem(71 + sorted(CASES).index(name), **CASES[name])
    (kq, ks, vq, vs), (kd, vd) = _quantised(p)
    extra = {}
    if p.kv_len is not None:
        extra["kv_len"] = torch.from_numpy(p.kv_len).cuda()
    out, lse = far.fa_rows_decode(dev_bits(p.q, p.dtype), kq, vq, torch.from_numpy(p.kv_rows).cuda(), p.scale,
                                  k_scale=ks, v_scale=vs, causal=p.causal, want_lse=True, **extra)
    ref, ref_lse = oracle_for(p, k=kd, v=vd)
    assert_parity(out, ref, f"fp8 {name}")
    assert_lse(lse, ref_lse)
