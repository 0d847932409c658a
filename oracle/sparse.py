"""Sparse row-list builder of the oracle: sinks + recent + top-k by score.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What it follows: the v100llm article (section 5, sparse prefill) selects the
tokens an attention step reads as anchor + recent + sink, and the
llama.cpp-v100 README's QSA sparse attention reads a selected subset of a
long context; "llama.cpp 0.9.0 inference boundaries" (section 1) is the
consumer: a sorted ``kv_rows`` list per query slice.  The learned indexer
that produces the scores is not part of this library: the caller supplies one
score per position.  Readings (the pages fix none of these):

* positions ``0 .. sinks-1`` (sinks) and ``n-recent .. n-1`` (recent) are
  always listed; from the positions in between, the ``k`` with the largest
  score are listed ("anchors");
* ties in score go to the smaller position; a NaN score ranks below every
  number (it is chosen only when fewer than ``k`` numbers remain);
* when the slice is shorter than ``sinks + recent``, or has no more than
  ``k`` middle positions, every position is listed;
* the list is in increasing position order, padded with -1 to ``list_len``;
  entry = ``row_map[s, pos]`` when a position -> pool-row map is given, else
  the position itself.
"""
from __future__ import annotations

from typing import Optional

import numpy as np


def select_rows(score: np.ndarray, sinks: int, recent: int, k: int, list_len: int,
                n_len: Optional[np.ndarray] = None, row_map: Optional[np.ndarray] = None) -> np.ndarray:
    """score [S, n_max] float; n_len [S] (None: n_max); returns int32 [S, list_len]."""
    score = np.asarray(score)
    S, n_max = score.shape
    out = np.full((S, list_len), -1, dtype=np.int32)
    for s in range(S):
        n = n_max if n_len is None else int(min(max(int(n_len[s]), 0), n_max))
        lo = min(sinks, n)
        hi = max(lo, n - recent)
        middle = list(range(lo, hi))
        if len(middle) > k:
            # rank by (score descending, position ascending); NaN below all numbers
            def rank_key(pos):
                v = float(score[s, pos])
                return (1, 0.0, pos) if v != v else (0, -v, pos)
            chosen = sorted(sorted(middle, key=rank_key)[:k])
        else:
            chosen = middle
        picked = list(range(0, lo)) + chosen + list(range(hi, n))
        if len(picked) > list_len:
            raise ValueError(f"slice {s}: {len(picked)} entries do not fit list_len {list_len}")
        rows = [int(row_map[s, pos]) if row_map is not None else pos for pos in picked]
        out[s, :len(rows)] = rows
    return out
