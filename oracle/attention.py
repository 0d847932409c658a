"""fp64 row-indexed attention, and the dense-mask form it replaces.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definitions used by both functions (written out from "llama.cpp 0.9.0
inference boundaries", section 1, and the readings stated beside them):

* slice ``s`` has a list ``kv_rows[s, 0:L]``; ``n_s = kv_len[s]`` when a
  per-slice length is given, else ``L`` (reading: entries at or beyond the
  length are padding, the same as a negative index);
* entry ``j`` is *listed* when ``j < n_s`` and ``kv_rows[s, j] >= 0``
  (negative = padding, mask minus infinity);
* query head ``h`` reads KV head ``h // (Hq // Hkv)`` (reading: consecutive
  query heads share a KV head);
* logit ``l_j = scale * <q, K[kv_rows[s, j], g]> + mask[s, i, j]``, the mask
  being additive and indexed by list position (the pages' "corresponding
  mask");
* causal (reading for a ubatch at the end of a prompt): the slice's ``Nq``
  queries are the last ``Nq`` positions of its ``n_s`` list entries, so query
  ``i`` sees list position ``j`` iff ``j <= n_s - Nq + i``;
* entries whose logit is minus infinity take no part; softmax over the rest;
  a query with no visible entry gets output 0 and log-sum-exp minus infinity
  (reading: the pages are silent on empty rows).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .kvcache import widen


def visible_positions(n_s: int, n_query: int, i: int, causal: bool) -> int:
    """Number of leading list positions that query ``i`` may see (before padding)."""
    if not causal:
        return n_s
    return max(0, min(n_s, n_s - n_query + i + 1))


def _softmax_average(logits: np.ndarray, values: np.ndarray):
    """Two-pass softmax over finite logits, then the weighted average of ``values``.

    Returns (output [D], log-sum-exp) with (0, -inf) when nothing is finite.
    """
    keep = logits > -np.inf
    if not np.any(keep):
        return np.zeros(values.shape[1]), -np.inf
    lk = logits[keep]
    m = np.max(lk)                      # pass 1: the maximum
    w = np.exp(lk - m)                  # pass 2: exponentials and their sum
    z = np.sum(w)
    out = (w @ values[keep]) / z
    return out, m + np.log(z)


def attend_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, kv_rows: np.ndarray, scale: float, *,
                mask: Optional[np.ndarray] = None, causal: bool = False,
                kv_len: Optional[np.ndarray] = None, query_rows: Optional[Sequence[int]] = None,
                n_query: Optional[int] = None, kv_format: Optional[str] = None):
    """Exact attention over each slice's listed pool rows.

    q        float64 [S, nq, Hq, D]   (nq query rows given; see ``query_rows``)
    k, v     float64 [R, Hkv, D]      the unified pool
    kv_rows  int     [S, L]           negative = padding
    mask     float   [S, Nq, L] or None, additive, list-aligned
    kv_len   int     [S] or None
    query_rows  which of the slice's ``n_query`` query rows the nq rows of
                ``q`` are (default 0..nq-1); used for causal visibility and to
                pick the mask row.
    kv_format   None when k, v are float64 already; 'bf16' or 'f16' when they
                are raw 16-bit patterns (widened after the gather, which keeps
                multi-GB pools out of float64).
    Returns (O float64 [S, nq, Hq, D], LSE float64 [S, nq, Hq]), LSE natural log.
    """
    S, nq, Hq, D = q.shape
    R, Hkv, Dk = k.shape
    assert Dk == D and v.shape == k.shape and Hq % Hkv == 0
    G = Hq // Hkv
    L = kv_rows.shape[1]
    if query_rows is None:
        query_rows = list(range(nq))
    if n_query is None:
        n_query = nq
    out = np.zeros((S, nq, Hq, D))
    lse = np.full((S, nq, Hq), -np.inf)
    for s in range(S):
        n_s = L if kv_len is None else int(min(max(int(kv_len[s]), 0), L))
        pos = np.arange(n_s)
        rows = kv_rows[s, :n_s].astype(np.int64)
        listed = rows >= 0
        pos, rows = pos[listed], rows[listed]
        for h in range(Hq):
            g = h // G
            Kg = k[rows, g, :]          # gathered listed rows, [n, D]
            Vg = v[rows, g, :]
            if kv_format is not None:
                Kg, Vg = widen(Kg, kv_format), widen(Vg, kv_format)
            for a, i in enumerate(query_rows):
                logits = scale * (Kg @ q[s, a, h, :])
                if mask is not None:
                    logits = logits + mask[s, i, pos].astype(np.float64)
                if causal:
                    limit = visible_positions(n_s, n_query, i, True)
                    logits = np.where(pos < limit, logits, -np.inf)
                out[s, a, h], lse[s, a, h] = _softmax_average(logits, Vg)
    return out, lse


def attend_dense(q: np.ndarray, k: np.ndarray, v: np.ndarray, kv_rows: np.ndarray, scale: float, *,
                 mask: Optional[np.ndarray] = None, causal: bool = False,
                 kv_len: Optional[np.ndarray] = None):
    """The path the row lists replace: attention over the WHOLE unified pool
    with a dense additive mask that is minus infinity on every pool row the
    slice may not see ("llama.cpp 0.9.0 inference boundaries", section 1).

    Needs distinct listed rows per slice (one mask cell per pool row) and
    finite pool contents.  Same arguments and returns as ``attend_rows``
    (all query rows).
    """
    S, Nq, Hq, D = q.shape
    R, Hkv, _ = k.shape
    G = Hq // Hkv
    L = kv_rows.shape[1]
    out = np.zeros((S, Nq, Hq, D))
    lse = np.full((S, Nq, Hq), -np.inf)
    for s in range(S):
        n_s = L if kv_len is None else int(min(max(int(kv_len[s]), 0), L))
        # dense mask over every pool row: start fully excluded, open the listed cells
        dense = np.full((Nq, R), -np.inf)
        for i in range(Nq):
            upto = n_s if not causal else max(0, n_s - Nq + i + 1)
            for j in range(min(upto, n_s)):
                r = int(kv_rows[s, j])
                if r < 0:
                    continue
                assert dense[i, r] == -np.inf, "dense form needs distinct rows"
                dense[i, r] = 0.0 if mask is None else float(mask[s, i, j])
        for h in range(Hq):
            kg = k[:, h // G, :]
            vg = v[:, h // G, :]
            for i in range(Nq):
                full = scale * (kg @ q[s, i, h, :]) + dense[i]
                ok = full > -np.inf
                if not ok.any():
                    continue
                top = full[ok].max()
                e = np.zeros(R)
                e[ok] = np.exp(full[ok] - top)
                tot = e.sum()
                out[s, i, h] = (e[:, None] * vg).sum(axis=0) / tot
                lse[s, i, h] = top + np.log(tot)
    return out, lse
