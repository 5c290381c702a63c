"""CPU oracle for QUOKA per-chunk KV selection plus sparse attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call
this module: only the tests, the package's smoke check and the benchmark's
CPU-baseline / reference legs do.  It is plain numpy in float64, written
stage by stage in the order the pages describe, with no blocking or fusion,
so that each function can be checked against the text by eye.  It shares no
code with the CUDA library.

Sources (page title, section):

* [P1] "QUOKA: Query-Oriented KV Selection For Efficient LLM Prefill"
  (paper summary, hw-hk.tistory.com/367): sections "Transformers and
  Attention", "Chunked prefill", "Attention Sparsity and Sparse Attention",
  "QUOKA Method", "Query Subselection", "Scoring via Cosine Similarity",
  "Aggregation Across Queries and KV Groups", "Chunked Prefill with QUOKA".
* [P2] "QUOKA Explained: Choosing Which KV History Attention Should Read":
  sections "Pick the queries that disagree with the crowd", "Letting those
  queries score the history", "Why take the maximum", "From scores to a
  smaller KV set", "A wrinkle: grouped-query attention", "MEAN and MAX do
  different jobs".

The pages lost every formula and both algorithm boxes in extraction.  The
readings taken where they are silent or garbled:

* causal mask: a chunk query at position c sees chunk keys 0..c (the
  diagonal included);
* softmax scale 1/sqrt(d) unless the caller gives another;
* the mean query is the plain mean of the raw queries of the whole chunk;
* GQA pooling has two modes: ``"mean"`` (the paper's pre-aggregation:
  per-group query selection on the head-averaged cosine, then the mean of
  the normalised query heads, not re-normalised) and ``"max"`` (per-head
  selection, max over every selected row of every head of the group);
* ties in both top-k steps go to the lower index; index sets are returned
  sorted ascending;
* a norm below EPS is clamped to EPS (a zero vector scores 0);
* only the history keys are scored and selected; the chunk's own keys are
  always attended, causally;
* the ablations the pages report (dot product instead of cosine, the mean
  instead of the maximum over the selected queries) change the key score
  only: query subselection stays on the cosine to the mean query, and with
  per-head pooling the maximum over the group's heads stays.

Parity pins for every function live in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-12
GQA_MODES = ("mean", "max")


# --------------------------------------------------------------------------
# Query subselection  [P1 "Query Subselection"; P2 "Pick the queries that
# disagree with the crowd"]
# --------------------------------------------------------------------------

def mean_query(Q: np.ndarray) -> np.ndarray:
    """M_q of every query head: the mean of the chunk's C raw queries.  Q [H_q, C, d] -> [H_q, d]."""
    return Q.sum(axis=1) / Q.shape[1]


def cosine(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """CosSim over the last axis, with each norm clamped at EPS."""
    na = np.maximum(np.sqrt((a * a).sum(axis=-1)), EPS)
    nb = np.maximum(np.sqrt((b * b).sum(axis=-1)), EPS)
    return (a * b).sum(axis=-1) / (na * nb)


def query_cosines(Q: np.ndarray) -> np.ndarray:
    """CosSim(M_q, q) for every chunk query of every head.  -> [H_q, C]."""
    M = mean_query(Q)
    return cosine(Q, M[:, None, :])


def keep_least_similar(cos_row: np.ndarray, n_q: int) -> np.ndarray:
    """Rank the queries by S_q = -CosSim(M_q, q) and keep the top n_q.

    Keeping the largest -cos is keeping the smallest cos.  A stable sort on
    cos puts equal values in index order, so ties go to the lower index.
    Returns the kept positions in ascending order.
    """
    n = min(n_q, cos_row.shape[0])
    order = np.argsort(cos_row, kind="stable")
    return np.sort(order[:n])


def select_queries(Q: np.ndarray, n_q: int, H_kv: int, gqa: str) -> np.ndarray:
    """Query subselection for one chunk.

    ``gqa="max"``: one set per query head, from that head's cosines -> [H_q, n].
    ``gqa="mean"``: one set per KV group, from the cosines averaged over the
    group's query heads, so that the group's heads share the token set that
    pre-aggregation averages over -> [H_kv, n].
    """
    cos = query_cosines(Q)
    if gqa == "max":
        return np.stack([keep_least_similar(cos[h], n_q) for h in range(cos.shape[0])])
    if gqa == "mean":
        G = Q.shape[0] // H_kv
        u = cos.reshape(H_kv, G, -1).mean(axis=1)
        return np.stack([keep_least_similar(u[g], n_q) for g in range(H_kv)])
    raise ValueError(gqa)


# --------------------------------------------------------------------------
# Scoring via cosine similarity and aggregation  [P1 "Scoring via Cosine
# Similarity", "Aggregation Across Queries and KV Groups"; P2 "Letting those
# queries score the history", "Why take the maximum", "A wrinkle:
# grouped-query attention", "MEAN and MAX do different jobs"]
# --------------------------------------------------------------------------

def normalize_rows(X: np.ndarray) -> np.ndarray:
    """Scale every row to unit length (norm clamped at EPS)."""
    return X / np.maximum(np.sqrt((X * X).sum(axis=-1, keepdims=True)), EPS)


SCORE_FNS = ("cos", "dot")
QUERY_AGGS = ("max", "mean")


def _query_rows(X: np.ndarray, score_fn: str) -> np.ndarray:
    """A query (or key) row as the score function sees it: unit length for
    the cosine, as it is for the plain dot product (the ablation of
    [P1 "Scoring via Cosine Similarity"])."""
    if score_fn == "cos":
        return normalize_rows(X)
    if score_fn == "dot":
        return X
    raise ValueError(score_fn)


def scoring_queries(Q: np.ndarray, q_idx: np.ndarray, H_kv: int, gqa: str, score_fn: str = "cos") -> list:
    """The rows each KV group scores its history with, one array [R, d] per group.

    ``"max"``: the selected query of every head of the group (R = G * n),
    normalised for the cosine.  ``"mean"``: pre-aggregation, the mean over
    the group's heads of the (normalised) queries at each selected token
    (R = n); the mean is not re-normalised, so its dot with a unit key is
    exactly the mean of the per-head cosines.
    """
    H_q = Q.shape[0]
    G = H_q // H_kv
    out = []
    for g in range(H_kv):
        heads = range(g * G, (g + 1) * G)
        if gqa == "max":
            out.append(np.concatenate([_query_rows(Q[h, q_idx[h]], score_fn) for h in heads], axis=0))
        elif gqa == "mean":
            out.append(sum(_query_rows(Q[h, q_idx[g]], score_fn) for h in heads) / G)
        else:
            raise ValueError(gqa)
    return out


def max_over_queries(S: np.ndarray) -> np.ndarray:
    """Query-axis aggregation: one score per key, the maximum over the rows of S [R, T]."""
    return S.max(axis=0)


def mean_over_queries(S: np.ndarray) -> np.ndarray:
    """The averaging alternative that [P2 "Why take the maximum"] sets against
    the maximum (and [P1 "Aggregation Across Queries and KV Groups"] ablates):
    one score per key, the mean over the rows of S [R, T]."""
    return S.sum(axis=0) / S.shape[0]


def score_keys(Q: np.ndarray, K_hist: np.ndarray, q_idx: np.ndarray, gqa: str, score_fn: str = "cos",
               query_agg: str = "max") -> np.ndarray:
    """Aggregated score of every history key of every KV group -> [H_kv, T].

    Per scoring row r and key t the score function gives r . k_t / |k_t|
    (cosine: the rows are unit too) or r . k_t (dot).  The query axis, the
    selected tokens, is aggregated by ``query_agg``; the GQA axis as the
    pooling mode says: ``"mean"`` already pre-aggregated the heads into the
    rows, ``"max"`` aggregates each head's tokens, then takes the maximum
    over the group's heads.  With ``query_agg="max"`` the latter is the
    maximum over every row of every head of the group.
    """
    if query_agg not in QUERY_AGGS:
        raise ValueError(query_agg)
    agg = max_over_queries if query_agg == "max" else mean_over_queries
    H_kv, T = K_hist.shape[0], K_hist.shape[1]
    rows = scoring_queries(Q, q_idx, H_kv, gqa, score_fn)
    out = np.zeros((H_kv, T))
    for g in range(H_kv):
        if T == 0:
            continue
        S = rows[g] @ _query_rows(K_hist[g], score_fn).T     # score of every row with every key
        if gqa == "max":
            n = q_idx.shape[1]
            G = rows[g].shape[0] // n
            per_head = np.stack([agg(S[k * n:(k + 1) * n]) for k in range(G)])   # one row per head
            out[g] = per_head.max(axis=0)
        else:
            out[g] = agg(S)
    return out


# --------------------------------------------------------------------------
# Top-B history keys  [P2 "From scores to a smaller KV set"; P1 "Chunked
# Prefill with QUOKA"]
# --------------------------------------------------------------------------

def top_b(score_row: np.ndarray, B: int) -> np.ndarray:
    """The min(B, T) keys with the largest score; ties to the lower index; ascending."""
    n = min(B, score_row.shape[0])
    order = np.argsort(-score_row, kind="stable")
    return np.sort(order[:n])


def select_keys(scores: np.ndarray, B: int) -> np.ndarray:
    """Top-B per KV head -> [H_kv, min(B, T)] int64."""
    return np.stack([top_b(scores[g], B) for g in range(scores.shape[0])]).astype(np.int64)


def gather(X_hist: np.ndarray, sel: np.ndarray) -> np.ndarray:
    """Rows of the history at the selected positions (the value comes with its key)."""
    return np.stack([X_hist[g, sel[g]] for g in range(X_hist.shape[0])])


# --------------------------------------------------------------------------
# Attention over the reduced set  [P1 "Transformers and Attention",
# "Chunked prefill", "QUOKA Method"; P2 "MEAN and MAX do different jobs":
# the original query heads attend]
# --------------------------------------------------------------------------

def attend(Q: np.ndarray, K_sel: np.ndarray, V_sel: np.ndarray, K_chunk: np.ndarray,
           V_chunk: np.ndarray, scale: float | None = None):
    """softmax([Q K_sel^T | Q K_chunk^T + M] * scale) [V_sel; V_chunk] for every query head.

    Q [H_q, C, d]; K_sel/V_sel [H_kv, n, d]; K_chunk/V_chunk [H_kv, C, d].
    M is 0 where chunk key j <= query c and -inf elsewhere.  Returns
    (O [H_q, C, d], lse [H_q, C]) with lse the natural log of the softmax
    denominator of the scaled logits.
    """
    H_q, C, d = Q.shape
    H_kv = K_chunk.shape[0]
    G = H_q // H_kv
    s = (1.0 / np.sqrt(d)) if scale is None else scale
    n = K_sel.shape[1]
    mask = np.zeros((C, n + C))
    mask[:, n:] = np.where(np.arange(C)[None, :] <= np.arange(C)[:, None], 0.0, -np.inf)
    O = np.zeros((H_q, C, d))
    lse = np.zeros((H_q, C))
    for h in range(H_q):
        g = h // G
        Kp = np.concatenate([K_sel[g], K_chunk[g]], axis=0)
        Vp = np.concatenate([V_sel[g], V_chunk[g]], axis=0)
        logits = (Q[h] @ Kp.T) * s + mask
        m = logits.max(axis=1, keepdims=True)
        e = np.exp(logits - m)
        den = e.sum(axis=1, keepdims=True)
        O[h] = (e / den) @ Vp
        lse[h] = (m + np.log(den))[:, 0]
    return O, lse


# --------------------------------------------------------------------------
# One chunk end to end  [P1 "QUOKA Method", "Chunked Prefill with QUOKA"]
# --------------------------------------------------------------------------

def chunk_attend(Q, K_hist, V_hist, K_chunk, V_chunk, n_q: int, B: int, gqa: str,
                 scale: float | None = None, score_fn: str = "cos", query_agg: str = "max") -> dict:
    """Select queries, score the history, keep the top-B keys, attend.

    With no history (T = 0) the chunk attends causally to itself only; with
    B >= T every history key is kept and selection is skipped.
    """
    H_kv, T = K_hist.shape[0], K_hist.shape[1]
    out = {"q_idx": None, "scores": None}
    if T == 0 or B >= T:
        sel = np.tile(np.arange(T, dtype=np.int64), (H_kv, 1))
    else:
        q_idx = select_queries(Q, n_q, H_kv, gqa)
        scores = score_keys(Q, K_hist, q_idx, gqa, score_fn, query_agg)
        sel = select_keys(scores, B)
        out.update(q_idx=q_idx, scores=scores)
    O, lse = attend(Q, gather(K_hist, sel), gather(V_hist, sel), K_chunk, V_chunk, scale)
    out.update(sel=sel, O=O, lse=lse)
    return out


def dense_attend(Q, K_hist, V_hist, K_chunk, V_chunk, scale: float | None = None):
    """Full chunked-prefill attention: every history key plus the causal chunk."""
    return attend(Q, K_hist, V_hist, K_chunk, V_chunk, scale)
