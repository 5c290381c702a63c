"""Device-side failure detection without a GPU fault: a bounded wait that can never
complete must record QUOKA_ERR_TIMEOUT and return, leaving the context usable."""
import pytest
import torch

from sparse_attention_chunked_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives(quoka):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert quoka.quoka_get_last_device_error(ws) == 0
    quoka.quoka_selftest_expire_wait(ws, 20_000_000)      # ~10 ms of SM cycles
    assert quoka.quoka_get_last_device_error(ws) == 6     # QUOKA_ERR_TIMEOUT, and the word is cleared
    assert quoka.quoka_get_last_device_error(ws) == 0
    # the context still runs real work
    cfg, x = wl.small_chunk(H_q=4, H_kv=2, d=128, C=64, T=200, N_q=4, B=32, dtype="bf16")
    O, _, _ = quoka.chunk_attend(x.Q.cuda(), x.K_hist.cuda(), x.V_hist.cuda(), x.K_chunk.cuda(), x.V_chunk.cuda(),
                                 cfg.N_q, cfg.B, gqa="max")
    torch.cuda.synchronize()
    assert torch.isfinite(O.float()).all()
