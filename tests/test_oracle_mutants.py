"""Each plausible mistake, planted in a copy of the CPU oracle, must make at least one pin fail."""
import types
from pathlib import Path

import pytest

from tests import oracle_pins

SRC = (Path(__file__).resolve().parent.parent / "oracle" / "quoka_oracle.py").read_text()

# (name, text in the oracle, planted replacement)
MUTANTS = [
    ("keeps_most_similar_queries", 'order = np.argsort(cos_row, kind="stable")',
     'order = np.argsort(-cos_row, kind="stable")'),
    ("cosine_drops_second_norm", "return (a * b).sum(axis=-1) / (na * nb)",
     "return (a * b).sum(axis=-1) / na"),
    ("group_selection_uses_first_head", "u = cos.reshape(H_kv, G, -1).mean(axis=1)",
     "u = cos.reshape(H_kv, G, -1)[:, 0]"),
    ("mean_over_queries_instead_of_max", "return S.max(axis=0)", "return S.mean(axis=0)"),
    ("keys_not_normalised", "S = rows[g] @ _query_rows(K_hist[g], score_fn).T", "S = rows[g] @ K_hist[g].T"),
    ("queries_not_normalised",
     "out.append(np.concatenate([_query_rows(Q[h, q_idx[h]], score_fn) for h in heads], axis=0))",
     "out.append(np.concatenate([Q[h, q_idx[h]] for h in heads], axis=0))"),
    ("preaggregate_renormalised", "out.append(sum(_query_rows(Q[h, q_idx[g]], score_fn) for h in heads) / G)",
     "out.append(normalize_rows(sum(_query_rows(Q[h, q_idx[g]], score_fn) for h in heads) / G))"),
    ("dot_still_normalises", 'if score_fn == "dot":\n        return X', 'if score_fn == "dot":\n        return normalize_rows(X)'),
    ("query_mean_is_max", "return S.sum(axis=0) / S.shape[0]", "return S.max(axis=0)"),
    ("query_mean_divides_by_keys", "return S.sum(axis=0) / S.shape[0]", "return S.sum(axis=0) / S.shape[1]"),
    ("query_mean_over_all_heads_rows", "per_head = np.stack([agg(S[k * n:(k + 1) * n]) for k in range(G)])",
     "per_head = agg(S)[None, :]"),
    ("heads_averaged_in_max_mode", "out[g] = per_head.max(axis=0)", "out[g] = per_head.mean(axis=0)"),
    ("topb_keeps_smallest", 'order = np.argsort(-score_row, kind="stable")',
     'order = np.argsort(score_row, kind="stable")'),
    ("topb_ties_to_higher_index", 'order = np.argsort(-score_row, kind="stable")',
     'order = (len(score_row) - 1 - np.argsort(-score_row[::-1], kind="stable"))'),
    ("mask_drops_diagonal", "np.arange(C)[None, :] <= np.arange(C)[:, None]",
     "np.arange(C)[None, :] < np.arange(C)[:, None]"),
    ("mask_transposed", "np.arange(C)[None, :] <= np.arange(C)[:, None]",
     "np.arange(C)[:, None] <= np.arange(C)[None, :]"),
    ("softmax_scale_missing", "logits = (Q[h] @ Kp.T) * s + mask", "logits = (Q[h] @ Kp.T) + mask"),
    ("gqa_head_map_modulo", "        g = h // G\n        Kp", "        g = h % H_kv\n        Kp"),
    ("lse_without_max", "lse[h] = (m + np.log(den))[:, 0]", "lse[h] = np.log(den)[:, 0]"),
    ("values_from_keys", "Vp = np.concatenate([V_sel[g], V_chunk[g]], axis=0)",
     "Vp = np.concatenate([K_sel[g], V_chunk[g]], axis=0)"),
    ("gather_from_head_zero", "return np.stack([X_hist[g, sel[g]] for g in range(X_hist.shape[0])])",
     "return np.stack([X_hist[0, sel[g]] for g in range(X_hist.shape[0])])"),
    ("history_not_selected", "O, lse = attend(Q, gather(K_hist, sel), gather(V_hist, sel), K_chunk, V_chunk, scale)",
     "O, lse = attend(Q, K_hist, V_hist, K_chunk, V_chunk, scale)"),
]


def _mutant_module(old, new):
    assert SRC.count(old) == 1, f"mutation anchor not unique: {old!r}"
    mod = types.ModuleType("quoka_oracle_mutant")
    exec(compile(SRC.replace(old, new), "quoka_oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    mod = _mutant_module(old, new)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mod)
        except Exception:            # an AssertionError, or a crash caused by the mistake
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake {name}"
