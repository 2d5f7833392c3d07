"""A wait that runs out inside a kernel reports ATTN_ERR_TIMEOUT through the status word and
leaves the CUDA context usable (no trap, no fault: the wait has a short limit)."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from parity import check_rows

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_and_context_survives():
    import torch

    import exact_io_aware_09_gb300 as attn

    assert attn.attn_poll_status() == 0
    attn.attn_selftest_timeout(20000)          # 20 ms on a barrier nothing arrives at
    assert attn.attn_poll_status() == -6
    assert attn.attn_poll_status() == 0        # polling clears the word
    cfg = syn.PrefillConfig("after", 1, 2, 2, 200, 200, 64, "bf16", True, 9)
    q, k, v = cfg.host_inputs()
    qt, kt, vt = (syn.bits_to_tensor(x, cfg.dtype, "cuda") for x in (q, k, v))
    o, lse = attn.attn_fwd(qt, kt, vt, causal=True, scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    orf, lrf = oracle.attention_rows(q, k, v, cfg.dtype, 1, 2, 2, 200, 200, 64, True, cfg.scale)
    check_rows(o.float().cpu().numpy().reshape(-1, 64), lse.cpu().numpy().reshape(-1), orf, lrf,
               "after a timed-out wait")
    torch.cuda.synchronize()
