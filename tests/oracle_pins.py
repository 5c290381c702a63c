"""Pins that tie the CPU oracle to something other than itself.

Every pin takes the oracle module as an argument and raises AssertionError
when the oracle disagrees with the pages' worked examples, a library routine,
a brute-force enumeration or an invariant of the mathematics.  The same pins
are run against deliberately broken copies of the oracle
(tests/test_oracle_mutants.py) to show that each plausible mistake is caught.
"""
from __future__ import annotations

import itertools
import json
import math
from pathlib import Path

import numpy as np
import scipy.spatial.distance as ssd
import scipy.special as ssp
import torch

GOLDEN = Path(__file__).parent / "golden"


def _golden(name):
    return json.loads((GOLDEN / name).read_text())


def _rng(seed):
    return np.random.default_rng([seed, 99])


# ---------------------------------------------------------------- worked examples

def pin_toy_query_selection(o):
    """Similarities .96 .94 .91 .35 .18 with N_q = 2 keep q4 and q5 (the least similar)."""
    g = _golden("toy_query_selection.json")
    kept = o.keep_least_similar(np.array(g["cos_to_mean"]), g["N_q"])
    assert list(kept) == g["kept_zero_based"], kept


def pin_toy_max_aggregation(o):
    """The 3x4 table aggregates to .90 .85 .95 .20 by the maximum (the mean of K1 would be .40)."""
    g = _golden("toy_max_aggregation.json")
    S = np.array(g["scores"])
    agg = o.max_over_queries(S)
    assert np.allclose(agg, g["max_per_key"], atol=1e-12), agg
    assert not np.isclose(agg[0], g["mean_of_K1"])


def pin_toy_topk(o):
    """Scores .90 .85 .95 .20 .12 .08 with a budget of 3 keep K1, K2, K3."""
    g = _golden("toy_topk.json")
    kept = o.top_b(np.array(g["scores"]), g["B"])
    assert list(kept) == g["kept_zero_based"], kept


# ---------------------------------------------------------------- library routines / brute force

def pin_cosine_vs_scipy(o):
    """CosSim(M_q, q) against scipy's cosine distance, M_q recomputed with np.mean."""
    r = _rng(1)
    Q = r.standard_normal((3, 9, 7)) + 0.5
    cos = o.query_cosines(Q)
    for h in range(3):
        M = np.mean(Q[h], axis=0)
        for c in range(9):
            ref = 1.0 - ssd.cosine(Q[h, c], M)
            assert abs(cos[h, c] - ref) < 1e-12, (h, c, cos[h, c], ref)


def _brute_select(cos_row, n):
    """Rank by (cos ascending, index ascending) with Python's sort; keep n."""
    order = sorted(range(len(cos_row)), key=lambda i: (cos_row[i], i))
    return sorted(order[:n])


def pin_select_queries_brute(o):
    """Per-head and per-group selection against a brute-force sort, with planted ties."""
    r = _rng(2)
    H_q, H_kv, C, d = 4, 2, 12, 5
    Q = r.standard_normal((H_q, C, d))
    Q[:, 7] = Q[:, 3]                # a copy of query 3: an exact cosine tie
    for n in (1, 3, 5, 12, 20):
        got = o.select_queries(Q, n, H_kv, "max")
        for h in range(H_q):
            M = Q[h].mean(axis=0)
            cos = [1.0 - ssd.cosine(Q[h, c], M) for c in range(C)]
            assert list(got[h]) == _brute_select(cos, min(n, C)), (n, h)
        got = o.select_queries(Q, n, H_kv, "mean")
        for g in range(H_kv):
            u = []
            for c in range(C):
                vals = []
                for h in (2 * g, 2 * g + 1):
                    M = Q[h].mean(axis=0)
                    vals.append(1.0 - ssd.cosine(Q[h, c], M))
                u.append(math.fsum(vals) / 2)
            assert list(got[g]) == _brute_select(u, min(n, C)), (n, g)


def _brute_scores(Q, K, q_idx, gqa, G):
    """Explicit loops: every selected query of every head against every key, then aggregate."""
    H_kv, T = K.shape[0], K.shape[1]
    out = np.zeros((H_kv, T))
    for g in range(H_kv):
        heads = list(range(g * G, (g + 1) * G))
        for t in range(T):
            if gqa == "max":
                vals = [1.0 - ssd.cosine(Q[h, i], K[g, t]) for h in heads for i in q_idx[h]]
                out[g, t] = max(vals)
            else:
                # per-head scoring followed by the average over the group's heads
                per_token = [math.fsum(1.0 - ssd.cosine(Q[h, i], K[g, t]) for h in heads) / G
                             for i in q_idx[g]]
                out[g, t] = max(per_token)
    return out


def pin_score_keys_brute(o):
    """Cosine scores with MAX over queries (and heads, or MEAN over heads) by explicit loops."""
    r = _rng(3)
    H_q, H_kv, C, T, d = 6, 2, 10, 17, 8
    Q = r.standard_normal((H_q, C, d))
    K = r.standard_normal((H_kv, T, d)) * r.uniform(0.1, 5.0, (H_kv, T, 1))
    for gqa in ("max", "mean"):
        q_idx = o.select_queries(Q, 4, H_kv, gqa)
        got = o.score_keys(Q, K, q_idx, gqa)
        ref = _brute_scores(Q, K, q_idx, gqa, H_q // H_kv)
        assert np.max(np.abs(got - ref)) < 1e-12, gqa


def pin_preaggregation_identity(o):
    """(Q1 K^T + Q2 K^T)/2 == ((Q1 + Q2)/2) K^T: mean-mode scores equal head-averaged cosines."""
    r = _rng(4)
    H_q, H_kv, C, T, d = 8, 2, 16, 40, 12
    Q = r.standard_normal((H_q, C, d)) * r.uniform(0.5, 3.0, (H_q, C, 1))
    K = r.standard_normal((H_kv, T, d))
    q_idx = o.select_queries(Q, 5, H_kv, "mean")
    got = o.score_keys(Q, K, q_idx, "mean")
    G = H_q // H_kv
    for g in range(H_kv):
        per_head = np.stack([
            np.array([[1.0 - ssd.cosine(Q[h, i], K[g, t]) for t in range(T)] for i in q_idx[g]])
            for h in range(g * G, (g + 1) * G)])
        ref = per_head.mean(axis=0).max(axis=0)
        assert np.max(np.abs(got[g] - ref)) < 1e-12


def _brute_topb(scores, B):
    """Rank counting: key t is kept iff fewer than B keys beat it (higher score, or equal and lower index)."""
    T = len(scores)
    kept = []
    for t in range(T):
        beaten_by = sum(1 for u in range(T)
                        if scores[u] > scores[t] or (scores[u] == scores[t] and u < t))
        if beaten_by < B:
            kept.append(t)
    return kept


def pin_topb_brute(o):
    """Top-B with planted ties against rank counting and against exhaustive subset search."""
    r = _rng(5)
    for trial in range(40):
        T = int(r.integers(1, 9))
        s = r.integers(-2, 3, T) * 0.25            # few distinct values -> frequent ties
        for B in range(1, T + 2):
            got = list(o.top_b(s, B))
            assert got == _brute_topb(s, B), (s, B, got)
            n = min(B, T)
            # exhaustive: the kept set has the largest score sum; among those the smallest indices
            best = max(itertools.combinations(range(T), n),
                       key=lambda S: (round(sum(s[i] for i in S), 9), [-i for i in S]))
            assert got == list(best), (s, B, got, best)


def pin_topb_nested_and_equivariant(o):
    """Kept sets grow by inclusion as B grows; permuting the history permutes the kept set."""
    r = _rng(6)
    s = r.standard_normal(50)
    prev = set()
    for B in range(1, 52):
        cur = set(o.top_b(s, B).tolist())
        assert prev <= cur and len(cur) == min(B, 50)
        prev = cur
    perm = r.permutation(50)
    for B in (1, 7, 30):
        a = set(perm[o.top_b(s[perm], B)].tolist())
        assert a == set(o.top_b(s, B).tolist())


def _sdpa(Q, K, V, mask_bool, scale):
    """torch's scaled_dot_product_attention in float64 on the CPU (mask True = attend)."""
    q = torch.from_numpy(Q)[None]
    k = torch.from_numpy(K)[None]
    v = torch.from_numpy(V)[None]
    m = torch.from_numpy(mask_bool)
    return torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m, scale=scale)[0].numpy()


def pin_attend_vs_sdpa(o):
    """Attention over [selected | causal chunk] against torch SDPA with an explicit boolean mask.

    GQA is expanded the library way (repeat_interleave over heads) rather than by h // G.
    """
    r = _rng(7)
    H_q, H_kv, C, n, d = 6, 3, 9, 13, 8
    Q = r.standard_normal((H_q, C, d))
    Ks, Vs = r.standard_normal((H_kv, n, d)), r.standard_normal((H_kv, n, d))
    Kc, Vc = r.standard_normal((H_kv, C, d)), r.standard_normal((H_kv, C, d))
    O, lse = o.attend(Q, Ks, Vs, Kc, Vc)
    G = H_q // H_kv
    Kall = np.repeat(np.concatenate([Ks, Kc], axis=1), G, axis=0)
    Vall = np.repeat(np.concatenate([Vs, Vc], axis=1), G, axis=0)
    mask = np.concatenate([np.ones((C, n), bool), np.tril(np.ones((C, C), bool))], axis=1)
    ref = _sdpa(Q, Kall, Vall, mask, 1.0 / math.sqrt(d))
    assert np.max(np.abs(O - ref)) < 1e-12
    logits = np.einsum("hcd,hjd->hcj", Q, Kall) / math.sqrt(d)
    logits = np.where(mask[None], logits, -np.inf)
    assert np.max(np.abs(lse - ssp.logsumexp(logits, axis=2))) < 1e-12


def pin_attend_invariants(o):
    """V == 1 gives O == 1; with no history the chunk is plain causal attention (SDPA is_causal)."""
    r = _rng(8)
    H, C, n, d = 2, 7, 5, 4
    Q = r.standard_normal((H, C, d)) * 3
    Ks, Kc = r.standard_normal((H, n, d)), r.standard_normal((H, C, d))
    O, _ = o.attend(Q, Ks, np.ones((H, n, d)), Kc, np.ones((H, C, d)))
    assert np.max(np.abs(O - 1.0)) < 1e-12
    Vc = r.standard_normal((H, C, d))
    O, _ = o.attend(Q, np.zeros((H, 0, d)), np.zeros((H, 0, d)), Kc, Vc, scale=0.3)
    q, k, v = (torch.from_numpy(x)[None] for x in (Q, Kc, Vc))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=0.3)[0].numpy()
    assert np.max(np.abs(O - ref)) < 1e-12


def pin_chunk_dense_when_budget_covers(o):
    """B >= T keeps every history key: the chunk equals dense chunked-prefill attention (SDPA)."""
    r = _rng(9)
    H_q, H_kv, C, T, d = 4, 2, 6, 11, 8
    Q = r.standard_normal((H_q, C, d))
    Kh, Vh = r.standard_normal((H_kv, T, d)), r.standard_normal((H_kv, T, d))
    Kc, Vc = r.standard_normal((H_kv, C, d)), r.standard_normal((H_kv, C, d))
    for B in (T, T + 5):
        res = o.chunk_attend(Q, Kh, Vh, Kc, Vc, 2, B, "max")
        G = H_q // H_kv
        Kall = np.repeat(np.concatenate([Kh, Kc], axis=1), G, axis=0)
        Vall = np.repeat(np.concatenate([Vh, Vc], axis=1), G, axis=0)
        mask = np.concatenate([np.ones((C, T), bool), np.tril(np.ones((C, C), bool))], axis=1)
        ref = _sdpa(Q, Kall, Vall, mask, 1.0 / math.sqrt(d))
        assert np.max(np.abs(res["O"] - ref)) < 1e-12


def pin_chunk_uses_selected_history(o):
    """With B < T the chunk attends exactly to the kept keys (SDPA over a masked full history)."""
    r = _rng(10)
    H_q, H_kv, C, T, d = 4, 2, 8, 30, 8
    Q = r.standard_normal((H_q, C, d))
    Kh, Vh = r.standard_normal((H_kv, T, d)), r.standard_normal((H_kv, T, d))
    Kc, Vc = r.standard_normal((H_kv, C, d)), r.standard_normal((H_kv, C, d))
    for gqa in ("max", "mean"):
        res = o.chunk_attend(Q, Kh, Vh, Kc, Vc, 3, 7, gqa)
        G = H_q // H_kv
        for h in range(H_q):
            g = h // G
            keep = np.zeros(T, bool)
            keep[res["sel"][g]] = True
            mask = np.concatenate([np.tile(keep, (C, 1)), np.tril(np.ones((C, C), bool))], axis=1)
            ref = _sdpa(Q[h:h + 1], np.concatenate([Kh[g], Kc[g]])[None],
                        np.concatenate([Vh[g], Vc[g]])[None], mask, 1.0 / math.sqrt(d))
            assert np.max(np.abs(res["O"][h] - ref[0])) < 1e-12


def pin_scale_invariance(o):
    """Cosine selection and scoring do not change when Q rows or K rows are scaled by c > 0."""
    r = _rng(11)
    H_q, H_kv, C, T, d = 4, 2, 12, 25, 6
    Q = r.standard_normal((H_q, C, d)) + 1.0
    K = r.standard_normal((H_kv, T, d))
    for gqa in ("max", "mean"):
        i0 = o.select_queries(Q, 4, H_kv, gqa)
        s0 = o.score_keys(Q, K, i0, gqa)
        i1 = o.select_queries(Q * 7.5, 4, H_kv, gqa)
        assert (i0 == i1).all()
        s1 = o.score_keys(Q * 7.5, K * r.uniform(0.2, 9.0, (H_kv, T, 1)), i0, gqa)
        assert np.max(np.abs(s0 - s1)) < 1e-12
        assert s0.max() <= 1 + 1e-12 and s0.min() >= -1 - 1e-12


def pin_selection_keeps_least_similar(o):
    """Every kept query is no more similar to the mean than any dropped one; N_q >= C keeps all."""
    r = _rng(12)
    Q = r.standard_normal((3, 20, 5)) + 0.7
    idx = o.select_queries(Q, 6, 3, "max")
    for h in range(3):
        M = Q[h].mean(axis=0)
        cos = np.array([1.0 - ssd.cosine(q, M) for q in Q[h]])
        kept = set(idx[h].tolist())
        dropped = [c for c in range(20) if c not in kept]
        assert max(cos[list(kept)]) <= min(cos[dropped]) + 1e-15
    assert (o.select_queries(Q, 50, 3, "max") == np.arange(20)).all()


def pin_needle_recovered(o):
    """A history key that copies a selected query (plus small noise) is kept by the top-B."""
    r = _rng(13)
    H_q, H_kv, C, T, d = 4, 2, 32, 200, 16
    Q = r.standard_normal((H_q, C, d)) + 2.0 * r.standard_normal((H_q, 1, d))
    K = r.standard_normal((H_kv, T, d))
    q_idx = o.select_queries(Q, 4, H_kv, "max")
    G = H_q // H_kv
    planted = []
    for g in range(H_kv):
        h = g * G + 1
        c = int(q_idx[h][0])
        t = int(r.integers(T))
        K[g, t] = Q[h, c] + 0.01 * r.standard_normal(d)
        planted.append((g, t))
    scores = o.score_keys(Q, K, q_idx, "max")
    sel = o.select_keys(scores, 8)
    for g, t in planted:
        assert t in set(sel[g].tolist()), (g, t)
        assert scores[g, t] > 0.99


# ---------------------------------------------------------------- the ablation variants of the key score

def pin_toy_mean_aggregation(o):
    """Averaging the toy table's K1 column gives the .40 the page prints; a mean never exceeds the maximum."""
    g = _golden("toy_max_aggregation.json")
    S = np.array(g["scores"])
    mean = o.mean_over_queries(S)
    assert abs(mean[0] - g["mean_of_K1"]) < 1e-12, mean
    assert np.all(mean <= o.max_over_queries(S) + 1e-15)
    same = np.tile(S[:1], (5, 1))                 # identical rows: mean and maximum agree
    assert np.allclose(o.mean_over_queries(same), o.max_over_queries(same), atol=1e-15)


def _sim(a, b, score_fn):
    return 1.0 - ssd.cosine(a, b) if score_fn == "cos" else float(np.dot(a, b))


def _brute_scores_variant(Q, K, q_idx, gqa, G, score_fn, query_agg):
    """Explicit loops: per (row, key) similarity, the query axis by max or mean, the GQA axis by the mode."""
    H_kv, T = K.shape[0], K.shape[1]
    agg = max if query_agg == "max" else (lambda v: math.fsum(v) / len(v))
    out = np.zeros((H_kv, T))
    for g in range(H_kv):
        heads = range(g * G, (g + 1) * G)
        for t in range(T):
            if gqa == "max":
                out[g, t] = max(agg([_sim(Q[h, i], K[g, t], score_fn) for i in q_idx[h]]) for h in heads)
            else:
                per_token = [math.fsum(_sim(Q[h, i], K[g, t], score_fn) for h in heads) / G for i in q_idx[g]]
                out[g, t] = agg(per_token)
    return out


def pin_score_variants_brute(o):
    """Cosine or dot, max or mean over the selected queries, both pooling modes, by explicit loops."""
    r = _rng(11)
    H_q, H_kv, C, T, d = 6, 2, 12, 15, 8
    Q = r.standard_normal((H_q, C, d)) * r.uniform(0.2, 4.0, (H_q, C, 1))
    K = r.standard_normal((H_kv, T, d)) * r.uniform(0.1, 5.0, (H_kv, T, 1))
    for gqa in ("max", "mean"):
        q_idx = o.select_queries(Q, 4, H_kv, gqa)
        for score_fn in ("cos", "dot"):
            for query_agg in ("max", "mean"):
                got = o.score_keys(Q, K, q_idx, gqa, score_fn, query_agg)
                ref = _brute_scores_variant(Q, K, q_idx, gqa, H_q // H_kv, score_fn, query_agg)
                assert np.max(np.abs(got - ref)) < 1e-10 * max(1.0, np.abs(ref).max()), (gqa, score_fn, query_agg)


def pin_dot_scales_cos_does_not(o):
    """The dot score is positively homogeneous in the keys and queries; on unit vectors it is the cosine."""
    r = _rng(12)
    H_q, H_kv, C, T, d = 4, 2, 9, 20, 6
    Q = r.standard_normal((H_q, C, d))
    K = r.standard_normal((H_kv, T, d))
    for gqa in ("max", "mean"):
        q_idx = o.select_queries(Q, 3, H_kv, gqa)
        for query_agg in ("max", "mean"):
            s = o.score_keys(Q, K, q_idx, gqa, "dot", query_agg)
            assert np.allclose(o.score_keys(Q, 3.0 * K, q_idx, gqa, "dot", query_agg), 3.0 * s, rtol=1e-12)
            assert np.allclose(o.score_keys(2.0 * Q, K, q_idx, gqa, "dot", query_agg), 2.0 * s, rtol=1e-12)
            Qu = Q / np.linalg.norm(Q, axis=-1, keepdims=True)
            Ku = K / np.linalg.norm(K, axis=-1, keepdims=True)
            assert np.allclose(o.score_keys(Qu, Ku, q_idx, gqa, "dot", query_agg),
                               o.score_keys(Q, K, q_idx, gqa, "cos", query_agg), atol=1e-12)


def pin_query_mean_with_one_query(o):
    """With one selected query per set there is nothing to aggregate: mean and maximum agree."""
    r = _rng(13)
    H_q, H_kv, C, T, d = 4, 2, 7, 11, 5
    Q = r.standard_normal((H_q, C, d))
    K = r.standard_normal((H_kv, T, d))
    for gqa in ("max", "mean"):
        q_idx = o.select_queries(Q, 1, H_kv, gqa)
        for score_fn in ("cos", "dot"):
            assert np.allclose(o.score_keys(Q, K, q_idx, gqa, score_fn, "mean"),
                               o.score_keys(Q, K, q_idx, gqa, score_fn, "max"), atol=1e-14)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
