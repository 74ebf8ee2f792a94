"""Top-k over Lightning-Indexer scores.

[GLM] §2.1: the indexer picks, from all history positions, the 2048 most
relevant to the current query; sparse attention then runs on those positions
only. The selection rule is written out here as a total order, so the result
is unique:
  * position i < ctx_len carries the key (score_i, -i): larger score first,
    and among equal scores the lower position first;
  * -0.0 and +0.0 are the same score; NaN is rejected; +-inf are ordinary;
  * the k positions greatest under that order are returned, sorted by
    ascending position (a canonical order; the pages leave it open).
"""
import numpy as np


def topk_ids(scores: np.ndarray, ctx_len: int, k: int) -> np.ndarray:
    s = np.asarray(scores[:ctx_len], dtype=np.float64) + 0.0   # -0.0 -> +0.0
    if ctx_len < k:
        raise ValueError(f"context {ctx_len} shorter than k={k}")
    if np.isnan(s).any():
        raise ValueError("NaN score")
    pos = np.arange(ctx_len)
    # lexsort sorts by the last key first: descending score, then ascending position
    order = np.lexsort((pos, -s))
    return np.sort(order[:k]).astype(np.int32)
