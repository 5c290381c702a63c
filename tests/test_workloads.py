"""The seeded input generator: determinism, shapes, and the structure each recipe promises."""
import numpy as np
import torch

from oracle import quoka_oracle as qo
from sparse_attention_chunked_gb300 import workloads as wl


def test_tiny_config_deterministic_and_shaped():
    cfg = wl.TINY_MHA_FP32
    a, b = wl.make_chunk(cfg, 0), wl.make_chunk(cfg, 0)
    assert torch.equal(a.Q, b.Q) and torch.equal(a.K_hist, b.K_hist)
    assert a.Q.shape == (4, 128, 64) and a.K_hist.shape == (4, 1024, 64)
    assert a.K_chunk.shape == (4, 128, 64) and a.Q.dtype == torch.float32
    assert a.outliers.shape == (4, 4) and len(a.needles) == 32
    c = wl.make_chunk(cfg, 1)
    assert not torch.equal(a.Q, c.Q)


def test_needles_copy_outlier_queries():
    cfg = wl.TINY_MHA_FP32
    x = wl.make_chunk(cfg, 0)
    Q, K = x.Q.double().numpy(), x.K_hist.double().numpy()
    for g, t, h, c in x.needles:
        assert qo.cosine(K[g, t], Q[h, c]) > 0.99


def test_massive_act_structure():
    cfg, x = wl.small_chunk(H_q=8, H_kv=2, d=128, C=200, T=500, dtype="bf16", recipe="massive_act")
    assert x.Q.dtype == torch.bfloat16
    Q = x.Q.double().numpy()
    n_out = round(0.05 * 200)
    assert x.outliers.shape == (8, n_out)
    cos = qo.query_cosines(Q)
    out = x.outliers[0]
    normal = np.setdiff1d(np.arange(200), out)
    # the shared direction makes ordinary queries far more similar to the mean than outliers
    assert cos[:, normal].mean() > cos[:, out].mean() + 0.2
    K = x.K_hist.double().numpy()
    assert len(x.needles) == 2 * 32
    # a few channels carry a large constant bias
    mean_abs = np.abs(K.mean(axis=1))
    assert (mean_abs > 0.5).sum(axis=1).max() <= 4


def test_oracle_recovers_needles_of_selected_queries():
    """Needles whose source query was selected are kept under GQA max pooling.

    Under mean pooling a needle copies one head of the group, so its score is
    diluted by the other heads: there it only has to beat the median key.
    """
    cfg, x = wl.small_chunk(H_q=8, H_kv=2, d=64, C=200, T=600, N_q=8, B=48, dtype="fp32",
                            recipe="massive_act")
    Q, K = x.Q.double().numpy(), x.K_hist.double().numpy()
    for gqa in ("max", "mean"):
        q_idx = qo.select_queries(Q, cfg.N_q, cfg.H_kv, gqa)
        scores = qo.score_keys(Q, K, q_idx, gqa)
        sel = qo.select_keys(scores, cfg.B)
        checked = 0
        for g, t, h, c in x.needles:
            row = q_idx[h] if gqa == "max" else q_idx[g]
            if c in set(row.tolist()):
                if gqa == "max":
                    assert t in set(sel[g].tolist())
                else:
                    assert scores[g, t] > np.median(scores[g])
                checked += 1
        assert checked > 0


def test_ragged_lengths_log_uniform_in_range():
    Ts = wl.ragged_history_lengths(wl.RAGGED_8x_BF16, 0)
    assert len(Ts) == 8 and all(4096 <= T <= 65536 for T in Ts)
    assert Ts == wl.ragged_history_lengths(wl.RAGGED_8x_BF16, 0)
