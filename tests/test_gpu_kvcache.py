"""KV-pool kernels against the oracle: bit-exact page expansion, INT8 codes,
scales and dequantisation, row appends; and INT8 paged decode parity."""
import numpy as np
import pytest
import torch

import oracle
import row_indexed_flash_gb300 as far
import synth
from helpers import assert_lse, assert_parity, dev_bits

pytestmark = pytest.mark.gpu


def test_page_table_expansion_is_bit_exact():
    p = synth.paged_int8(n_seq=9, lo=1, hi=5000)
    pt = torch.from_numpy(p.page_table).cuda()
    sl = torch.from_numpy(p.seq_len).cuda()
    for L in (p.L, p.L + 3, p.L - 1):
        got = far.fa_kv_page_table_to_rows(pt, sl, L)
        want = oracle.page_table_to_rows(p.page_table, p.seq_len, L)
        assert np.array_equal(got.cpu().numpy(), want)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f16", 128), ("bf16", 256), ("bf16", 64), ("f16", 96)])
def test_int8_quantise_and_dequantise_are_bit_exact(dtype, D):
    g = synth.rng(77)
    R, H = 640, 4
    bits = synth.normal_bits(g, (R, H, D), dtype)
    bits[3, 1] = 0                                   # an all-zero (row, head): scale 0
    x = dev_bits(bits, dtype)
    q, s = far.fa_kv_quantize_int8(x, R)
    qo, so = oracle.quantize_int8(oracle.widen(bits, dtype).astype(np.float32))
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), oracle.pack_scales(so).view(np.uint16))
    deq = far.fa_kv_dequantize_int8(q, s).cpu().numpy()
    assert np.array_equal(deq.view(np.uint32), oracle.dequantize_int8(qo, so).view(np.uint32))


_NONFINITE = {"bf16": (0x7FC0, 0xFFC0, 0x7F80, 0xFF80), "f16": (0x7E00, 0xFE00, 0x7C00, 0xFC00)}


@pytest.mark.parametrize("codec,dtype,D", [("int8", "bf16", 128), ("int8", "f16", 96), ("int8", "bf16", 256),
                                           ("int4", "bf16", 128), ("int4", "f16", 64), ("fp8", "bf16", 128),
                                           ("fp8", "f16", 96)])
def test_quantisers_keep_nan_and_saturate_inf_like_the_oracle(codec, dtype, D):
    """The non-finite reading: a (row, head) holding a NaN gets scale 0x7E00
    and NaN codes (0, or 0x7f for E4M3); an Inf element gives scale 65504 and
    saturates.  Codes and scales bit-exact, dequantised values equal (NaN
    where the oracle has NaN)."""
    g = synth.rng(80)
    R, H = 128, 4
    bits = synth.normal_bits(g, (R, H, D), dtype)
    qnan, nnan, pinf, ninf = _NONFINITE[dtype]
    bits[1, 0, 5] = qnan                 # one NaN
    bits[2, 3, D - 1] = nnan             # a negative NaN at the last element
    bits[3, 2, 0] = pinf                 # +Inf at the first element
    bits[4, 1, 7] = ninf                 # -Inf
    bits[5, 0, 9], bits[5, 0, 10] = pinf, ninf       # both infinities
    bits[6, 2, 3], bits[6, 2, 4] = pinf, qnan        # Inf and NaN: the NaN decides
    bits[7, 3] = qnan                    # every element NaN
    x = dev_bits(bits, dtype)
    xo = oracle.widen(bits, dtype).astype(np.float32)
    quant, deq_gpu, quant_o, deq_o = {
        "int8": (far.fa_kv_quantize_int8, far.fa_kv_dequantize_int8, oracle.quantize_int8, oracle.dequantize_int8),
        "int4": (far.fa_kv_quantize_int4, far.fa_kv_dequantize_int4, oracle.quantize_int4, oracle.dequantize_int4),
        "fp8": (far.fa_kv_quantize_fp8, far.fa_kv_dequantize_fp8, oracle.quantize_fp8, oracle.dequantize_fp8),
    }[codec]
    q, s = quant(x, R)
    qo, so = quant_o(xo)
    got_codes = q.cpu().view(torch.uint8).numpy() if codec == "fp8" else q.cpu().numpy()
    assert np.array_equal(got_codes.view(np.uint8), qo.view(np.uint8))
    assert np.array_equal(s.cpu().numpy().view(np.uint16), oracle.pack_scales(so).view(np.uint16))
    nan_rows = [(1, 0), (2, 3), (6, 2), (7, 3)]
    for r, h in nan_rows:
        assert s.cpu().numpy().view(np.uint16)[r // 64, h, r % 64] == 0x7E00
    dg = deq_gpu(q, s).cpu().numpy()
    do = deq_o(qo, so)
    assert np.array_equal(np.isnan(dg), np.isnan(do))
    fin = ~np.isnan(do)
    assert np.array_equal(dg[fin].view(np.uint32), do[fin].view(np.uint32))


def test_int8_append_scatters_into_named_rows():
    g = synth.rng(78)
    R, H, D, n = 256, 2, 128, 40
    bits = synth.normal_bits(g, (n, H, D), "bf16")
    dst = g.permutation(R)[:n].astype(np.int32)
    dst[7] = -1
    q, s = far.fa_kv_quantize_int8(dev_bits(bits, "bf16"), R, dst_rows=torch.from_numpy(dst).cuda())
    pool0 = np.zeros((R, H, D), np.int8)
    sc0 = np.zeros((R // 64, H, 64), np.float16)
    qo, so = oracle.append_rows(pool0, oracle.widen_bf16(bits).astype(np.float32), dst, sc0, fmt="int8")
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), so.view(np.uint16))


@pytest.mark.parametrize("codec", ["int8", "int4", "fp8"])
@pytest.mark.parametrize("dtype,D,H", [("bf16", 64, 8), ("f16", 128, 8), ("bf16", 256, 8), ("bf16", 128, 3)])
def test_append_codecs_over_many_items_and_a_ragged_tail(codec, dtype, D, H):
    """A ubatch large enough that each warp of the staged quantiser strides
    over several of its tiles (the grid holds 4 blocks x 8 warps per SM), with
    a ragged last tile, rows named out of order, skipped (-1) and out of range
    (>= R); with 3 KV heads the warps' item stride is not a multiple of the
    head count, so the stepped (row, head) of an item carries.  Then the same
    ubatch from a source that is not 16-byte aligned (the
    one-warp-per-item path).  Codes and scales bit-exact against the oracle's,
    untouched rows zero."""
    g = synth.rng(81 + D + H)
    n = {64: 21_003, 128: 12_003, 256: 6_007}[D] * (2 if H == 3 else 1)
    R = 64 * ((n + 200) // 64 + 1)
    bits = synth.normal_bits(g, (n, H, D), dtype)
    dst = g.permutation(R)[:n].astype(np.int32)
    dst[::11] = -1
    dst[5::13] = R + 5
    quant, quant_o = {"int8": (far.fa_kv_quantize_int8, oracle.quantize_int8),
                      "int4": (far.fa_kv_quantize_int4, oracle.quantize_int4),
                      "fp8": (far.fa_kv_quantize_fp8, oracle.quantize_fp8)}[codec]
    qo, so = quant_o(oracle.widen(bits, dtype).astype(np.float32))
    live = (dst >= 0) & (dst < R)
    flat = torch.zeros(n * H * D + 8, dtype=torch.int16, device="cuda")
    for offset in (0, 1):
        x = flat[offset:offset + n * H * D].view(n, H, D)
        x.copy_(torch.from_numpy(bits.view(np.int16)).cuda())
        q, s = quant(x.view(torch.bfloat16 if dtype == "bf16" else torch.float16), R,
                     dst_rows=torch.from_numpy(dst).cuda())
        qn = q.cpu().view(torch.uint8).numpy() if codec == "fp8" else q.cpu().numpy()
        sn = oracle.unpack_scales(s.cpu().numpy()).view(np.uint16)
        assert np.array_equal(qn[dst[live]].view(np.uint8), qo[live].view(np.uint8))
        assert np.array_equal(sn[dst[live]], so[live].view(np.uint16))
        untouched = np.setdiff1d(np.arange(R), dst[live])
        assert not qn[untouched].any() and not sn[untouched].any()


def _e4m3_positive_values():
    """The finite positive E4M3 values, ascending (bias 7, 3 mantissa bits,
    largest 448): the grid whose midpoints the FP8 tie case uses."""
    sub = [m * 2.0 ** -9 for m in range(1, 8)]
    norm = [(1 + m / 8) * 2.0 ** e for e in range(-6, 9) for m in range(8)]
    return np.array(sorted(v for v in sub + norm if v <= 448.0))


@pytest.mark.parametrize("codec,dtype", [("int8", "f16"), ("int4", "bf16"), ("fp8", "bf16")])
def test_quantisers_round_exact_ties_to_even(codec, dtype):
    """Rows whose scale is 0.09375 (3 * 2^-5, no exact reciprocal) and whose
    other elements make x / s an exact tie: k + 1/2 for the integer codecs, a
    midpoint of the E4M3 grid for FP8.  The codes must round those ties to
    even, bit-exact against the oracle; for INT8 and INT4 also against the
    closed form (k if k is even, else k + 1, with the element's sign).  A few
    elements are -0 and +0, which E4M3 codes apart."""
    s_val = 0.09375
    top = {"int8": 127, "int4": 7, "fp8": 448}[codec]
    if codec == "fp8":
        grid = _e4m3_positive_values()
        q_tie = ((grid[:-1] + grid[1:]) / 2)[-127:]          # 127 midpoints, up to just below 448
    else:
        q_tie = np.arange(top) + 0.5                         # 0.5 .. top - 0.5
    g = synth.rng(83)
    n, H, D = 64, 2, 128
    vals = np.empty((n, H, D))
    vals[:, :, 0] = top * s_val                              # amax: s = fp16(amax / top) = 0.09375 exactly
    picks = g.integers(0, q_tie.size, size=(n, H, D - 1))
    signs = np.where(g.random((n, H, D - 1)) < 0.5, -1.0, 1.0)
    vals[:, :, 1:] = signs * q_tie[picks] * s_val
    vals[::3, :, 1], vals[::3, :, 2] = -0.0, 0.0              # signed zeros (E4M3 codes them 0x80 and 0x00)
    wide = vals.astype(np.float32)
    assert np.array_equal(wide.astype(np.float64), vals)     # every value is exact in fp32
    bits = synth.f32_to_bf16_bits(wide) if dtype == "bf16" else synth.f32_to_f16_bits(wide)
    assert np.array_equal(oracle.widen(bits, dtype).astype(np.float64), vals)   # and in the input type
    quant, quant_o = {"int8": (far.fa_kv_quantize_int8, oracle.quantize_int8),
                      "int4": (far.fa_kv_quantize_int4, oracle.quantize_int4),
                      "fp8": (far.fa_kv_quantize_fp8, oracle.quantize_fp8)}[codec]
    q, s = quant(dev_bits(bits, dtype), n)
    qo, so = quant_o(oracle.widen(bits, dtype).astype(np.float32))
    assert np.all(so.astype(np.float64) == s_val)
    got = q.cpu().view(torch.uint8).numpy() if codec == "fp8" else q.cpu().numpy()
    assert np.array_equal(got.view(np.uint8), qo.view(np.uint8))
    assert np.array_equal(s.cpu().numpy().view(np.uint16), oracle.pack_scales(so).view(np.uint16))
    if codec != "fp8":
        k = np.floor(q_tie[picks]).astype(np.int64)
        want = (signs * np.where(k % 2 == 0, k, k + 1)).astype(np.int64)
        want[::3, :, :2] = 0
        codes = oracle.dequantize_int8(qo, so) if codec == "int8" else oracle.dequantize_int4(qo, so)
        assert np.array_equal(np.rint(codes[:, :, 1:] / s_val).astype(np.int64), want)


def test_append_16bit_rows():
    g = synth.rng(79)
    R, H, D, n = 300, 8, 128, 50
    pool_bits = synth.normal_bits(g, (R, H, D), "bf16")
    new_bits = synth.normal_bits(g, (n, H, D), "bf16")
    dst = g.permutation(R)[:n].astype(np.int32)
    dst[::9] = -3
    pool = dev_bits(pool_bits, "bf16")
    far.fa_kv_append(dev_bits(new_bits, "bf16"), torch.from_numpy(dst).cuda(), pool)
    want, _ = oracle.append_rows(pool_bits, new_bits, dst)
    assert np.array_equal(pool.cpu().view(torch.int16).numpy().view(np.uint16), want)


def _int8_problem_on_device(p, slices=None):
    """Quantise the bf16 pool on the device and, independently, in the oracle."""
    k = dev_bits(p.k, "bf16")
    v = dev_bits(p.v, "bf16")
    kq, ks = far.fa_kv_quantize_int8(k, p.R)
    vq, vs = far.fa_kv_quantize_int8(v, p.R)
    del k, v
    return kq, ks, vq, vs


def _oracle_int8(p, rows, slices):
    """Oracle attention over dequantised INT8 rows; quantises only the rows used."""
    used = np.unique(rows[slices][rows[slices] >= 0])
    kq, ks = oracle.quantize_int8(oracle.widen_bf16(p.k[used]).astype(np.float32))
    vq, vs = oracle.quantize_int8(oracle.widen_bf16(p.v[used]).astype(np.float32))
    kd = oracle.dequantize_int8(kq, ks).astype(np.float64)
    vd = oracle.dequantize_int8(vq, vs).astype(np.float64)
    remap = np.full(p.R, -1, np.int64)
    remap[used] = np.arange(used.size)
    r2 = np.where(rows[slices] >= 0, remap[np.maximum(rows[slices], 0)], -1).astype(np.int32)
    q = oracle.widen_bf16(p.q[slices])
    return oracle.attend_rows(q, kd, vd, r2, p.scale), (kq, ks, vq, vs, used)


def test_paged_int8_decode_small():
    p = synth.paged_int8(n_seq=6, lo=100, hi=9000)
    rows_np = oracle.page_table_to_rows(p.page_table, p.seq_len, p.L)
    kq, ks, vq, vs = _int8_problem_on_device(p)
    rows = far.fa_kv_page_table_to_rows(torch.from_numpy(p.page_table).cuda(), torch.from_numpy(p.seq_len).cuda(), p.L)
    assert np.array_equal(rows.cpu().numpy(), rows_np)
    q = dev_bits(p.q, "bf16")
    out, lse = far.fa_rows_decode(q, kq, vq, rows, p.scale, k_scale=ks, v_scale=vs, want_lse=True,
                                  kv_len=torch.from_numpy(p.seq_len).cuda(), n_valid_hint=int(p.seq_len.sum()))
    (ref, ref_lse), (okq, oks, _, _, used) = _oracle_int8(p, rows_np, slice(None))
    assert np.array_equal(kq.cpu().numpy()[used], okq)
    assert_parity(out, ref, "paged int8 small")
    assert_lse(lse, ref_lse)


@pytest.mark.slow
def test_workload_paged_int8_full_size_sampled_slices():
    p = synth.paged_int8()
    rows_np = oracle.page_table_to_rows(p.page_table, p.seq_len, p.L)
    kq, ks, vq, vs = _int8_problem_on_device(p)
    rows = far.fa_kv_page_table_to_rows(torch.from_numpy(p.page_table).cuda(), torch.from_numpy(p.seq_len).cuda(), p.L)
    assert np.array_equal(rows.cpu().numpy(), rows_np)
    q = dev_bits(p.q, "bf16")
    out, lse = far.fa_rows_decode(q, kq, vq, rows, p.scale, k_scale=ks, v_scale=vs, want_lse=True,
                                  kv_len=torch.from_numpy(p.seq_len).cuda(), n_valid_hint=int(p.seq_len.sum()))
    torch.cuda.synchronize()
    # the oracle on a sample of slices: the longest, the shortest and four random ones
    order = np.argsort(p.seq_len)
    pick = sorted({int(order[0]), int(order[-1])} | set(synth.rng(5).choice(p.S, 4, replace=False).tolist()))
    (ref, ref_lse), (okq, oks, ovq, ovs, used) = _oracle_int8(p, rows_np, pick)
    assert np.array_equal(kq.cpu().numpy()[used], okq) and np.array_equal(vq.cpu().numpy()[used], ovq)
    assert_parity(out[pick], ref, "paged int8 full")
    assert_lse(lse[pick], ref_lse)
