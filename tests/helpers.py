"""Shared test helpers: moving synthetic problems to the device, running the
oracle on the same input bits, and the parity tolerance.

Tolerance (fp16/bf16 inputs, fp32 accumulation): |gpu - oracle| <= 2e-3 for
every element, and |gpu - oracle| / |oracle| <= 1e-2 where |oracle| >= 0.2
(below that the absolute bound is the tighter one).  A bf16/fp16 output is
additionally allowed half an output ulp of rounding.
"""
import numpy as np
import torch

import oracle

ABS_TOL = 2e-3
REL_TOL = 1e-2


def dev_bits(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16).to(device)


def widen(a, dtype):
    return oracle.widen_bf16(a) if dtype == "bf16" else oracle.widen_f16(a)


def assert_parity(got: torch.Tensor, ref: np.ndarray, what: str = "", out_dtype=torch.float32):
    g = got.float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    slack = 0.0
    if out_dtype == torch.bfloat16:
        slack = np.abs(ref) * 2.0 ** -8
    elif out_dtype == torch.float16:
        slack = np.abs(ref) * 2.0 ** -11
    bad = err > ABS_TOL + slack
    assert not bad.any(), f"{what}: max abs err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    big = np.abs(ref) >= 0.2
    if big.any():
        rel = (err[big] - (slack[big] if np.ndim(slack) else 0.0)) / np.abs(ref[big])
        assert rel.max() <= REL_TOL, f"{what}: max rel err {rel.max():.3e}"
    return float(err.max())


def assert_lse(got: torch.Tensor, ref: np.ndarray, what=""):
    g = got.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(g), fin), f"{what}: lse finiteness differs"
    if fin.any():
        err = np.abs(g[fin] - ref[fin])
        assert err.max() <= ABS_TOL * 2, f"{what}: lse err {err.max():.3e}"


def oracle_for(p, k=None, v=None, kv_rows=None, query_rows=None, slices=None):
    """Oracle on problem p (raw bits unless k/v float64 pools are given)."""
    rows = p.kv_rows if kv_rows is None else kv_rows
    q = widen(p.q, p.dtype)
    mask = None if p.mask is None else p.mask.astype(np.float64)
    kv_len = p.kv_len
    if slices is not None:
        q, rows = q[slices], rows[slices]
        mask = None if mask is None else mask[slices]
        kv_len = None if kv_len is None else kv_len[slices]
    if query_rows is not None:
        q = q[:, query_rows]
    fmt = None if k is not None else p.dtype
    return oracle.attend_rows(q, p.k if k is None else k, p.v if v is None else v, rows, p.scale, mask=mask,
                              causal=p.causal, kv_len=kv_len, query_rows=query_rows, n_query=p.Nq,
                              kv_format=fmt)
