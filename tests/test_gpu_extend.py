"""skv_extend (a new turn of an agent session) against the oracle, and the
reason it exists: a grown session keeps its device buffer warm (GPU)."""
import numpy as np
import pytest
import torch

import oracle as orc
import skv_workload as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from skv_pair import Pair
    from sparse_attention_kv_skv_gb300 import SkvError

AGENTIC_SMALL = wl.Workload("agentic_small", B=6, L=3, ctx=2850, k=256, S=512, steps=24, fresh=0.2,
                            dist=wl.DIST_RECENCY, window=150, p_window=0.7, turn_every=4, turn_tokens=150)


def _run(w, republish=False):
    p = Pair(w)
    try:
        for s in range(w.steps):
            p.step(s, republish=republish)
            if s % 8 == 7:
                p.compare_state()
        p.compare_state()
        p.compare_hot_rows(range(w.B))
        assert p.ctx.get_device_error() == 0
        return p.total_misses
    finally:
        p.close()


def test_agent_sessions_extended_each_turn_match_oracle():
    _run(AGENTIC_SMALL)


def test_extend_keeps_the_buffer_warm():
    """The same Top-k sequence misses far less when each turn extends the
    session than when the grown session is published again (cold buffer)."""
    warm = _run(AGENTIC_SMALL, republish=False)
    cold = _run(AGENTIC_SMALL, republish=True)
    turns = AGENTIC_SMALL.steps // AGENTIC_SMALL.turn_every - 1
    w = AGENTIC_SMALL
    assert cold - warm >= turns * w.B * w.L * (w.k - w.n_fresh) * 0.5, (warm, cold)


def test_extend_errors():
    w = wl.Workload("ext_err", B=2, L=2, ctx=20, k=2, S=4, steps=2, turn_every=1, turn_tokens=5)
    p = Pair(w)   # max_context = 20 + 2 * 5 = 30
    try:
        rows = torch.zeros((w.L, 11, wl.ROW_BYTES), dtype=torch.uint8, device="cuda")
        with pytest.raises(SkvError, match="BAD_REQUEST"):
            p.ctx.extend(2, rows, 1)
        with pytest.raises(SkvError, match="CONTEXT_FULL"):
            p.ctx.extend(0, rows, 31)
        p.ctx.extend(0, rows[:, :0], 0)                      # no-op
        p.ctx.extend(0, rows, 11)                            # 20 + 11 > 30: rejected on the device
        assert p.orc.extend(0, rows.cpu().numpy()) == orc.E_CONTEXT_FULL
        assert p.ctx.get_device_error() == p.orc.get_error() == orc.E_CONTEXT_FULL
        p.ctx.extend(0, rows[:, :10].contiguous(), 10)       # exactly fills the region
        assert p.orc.extend(0, rows[:, :10].cpu().numpy()) == 0
        assert p.ctx.export_state(0)["len"] == 30 == p.orc.export(0)["len"]
        assert p.ctx.get_device_error() == 0
    finally:
        p.close()
