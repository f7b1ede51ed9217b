"""The bounded-wait failure path, exercised without any GPU fault: a wait that
nothing satisfies gives up, the status word is read on the host as
KDA_ERR_TIMEOUT, it is cleared by the read, and the context stays usable."""
import pytest
import torch

import linear_attention_sequence_gb300 as kda
from linear_attention_sequence_gb300 import synth

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    assert kda.kda_get_last_device_error() == 0
    kda.kda_selftest_timeout()
    assert kda.kda_get_last_device_error() == 4          # KDA_ERR_TIMEOUT
    assert kda.kda_get_last_device_error() == 0          # cleared by the read
    inp = synth.random_inputs(64, 2, 128, dtype=torch.bfloat16, seed=1, device="cuda")
    out, fin = kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"])
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
    assert kda.kda_get_last_device_error() == 0


def test_normal_runs_leave_no_status():
    inp = synth.random_inputs(300, 3, 128, dtype=torch.bfloat16, seed=2, device="cuda")
    for v in (kda.PREFILL_DEFAULT, kda.PREFILL_FP32):
        kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], variant=v)
    assert kda.kda_get_last_device_error() == 0
