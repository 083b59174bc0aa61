"""One-layer assemble calls (skv_assemble_layer) against the oracle's
one-layer calls, bit-exact (GPU)."""
import numpy as np
import pytest
import torch

import oracle as orc
import skv_workload as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from skv_pair import Pair
    from sparse_attention_kv_skv_gb300 import SkvError


def _layer_call(p, layer, topk_layer, slots_d, hits_d, misses_d, topk_d):
    topk_d.copy_(torch.from_numpy(np.ascontiguousarray(topk_layer)))
    p.ctx.assemble_layer(layer, p.req_dev, topk_d, slots_d, hits_d, misses_d)
    e, slots, hits, misses = p.orc.assemble_layer(layer, p.req_ids, topk_layer)
    assert e == 0
    assert np.array_equal(slots_d.cpu().numpy(), slots), layer
    assert np.array_equal(hits_d.cpu().numpy(), hits) and np.array_equal(misses_d.cpu().numpy(), misses)


@pytest.mark.parametrize("order", ["ascending", "varying"])
def test_layer_by_layer_steps_match_oracle(order):
    w = wl.Workload("layers", B=5, L=4, ctx=6000, k=300, S=640, steps=10, fresh=0.3, order=wl.ORDER_SHUFFLED,
                    n_pad=11)
    p = Pair(w, req_perm=[3, 0, 4, 1, 2])
    try:
        topk_d = torch.empty((w.B, w.k), dtype=torch.int32, device="cuda")
        slots_d = torch.empty_like(topk_d)
        hits_d = torch.empty(w.B, dtype=torch.int32, device="cuda")
        misses_d = torch.empty_like(hits_d)
        rng = np.random.default_rng(3)
        for s in range(w.steps):
            topk = p.gen.step(s, p.lens)
            layers = list(range(w.L)) if order == "ascending" else list(rng.permutation(w.L))
            for l in layers:
                _layer_call(p, int(l), topk[:, l, :], slots_d, hits_d, misses_d, topk_d)
            if s % 3 == 2:
                p.compare_state()
        assert p.ctx.clock() == p.orc.now == w.steps * w.L
        p.compare_state()
        p.compare_hot_rows(range(w.B))
    finally:
        p.close()


def test_layer_calls_mixed_with_full_steps_and_captured_in_a_graph():
    w = wl.Workload("mixed", B=3, L=3, ctx=4000, k=256, S=512, steps=9, fresh=0.3)
    p = Pair(w)
    try:
        topk_d = torch.empty((w.L, w.B, w.k), dtype=torch.int32, device="cuda")
        slots_d = torch.empty_like(topk_d)
        hits_d = torch.empty((w.L, w.B), dtype=torch.int32, device="cuda")
        misses_d = torch.empty_like(hits_d)

        def layered(step_topk):
            topk_d.copy_(torch.from_numpy(np.ascontiguousarray(step_topk.transpose(1, 0, 2))))

        # one graph = the L layer calls of a step, in order
        p.step(0)
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side), torch.cuda.graph(g, stream=side):
            for l in range(w.L):
                p.ctx.assemble_layer(l, p.req_dev, topk_d[l], slots_d[l], hits_d[l], misses_d[l])
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        p.compare_state()
        for s in range(1, w.steps):
            if s % 2:   # a full step
                p.step(s)
                continue
            topk = p.gen.step(s, p.lens)
            layered(topk)
            g.replay()
            for l in range(w.L):
                e, slots, hits, misses = p.orc.assemble_layer(l, p.req_ids, topk[:, l, :])
                assert e == 0
                assert np.array_equal(slots_d[l].cpu().numpy(), slots), (s, l)
                assert np.array_equal(hits_d[l].cpu().numpy(), hits)
                assert np.array_equal(misses_d[l].cpu().numpy(), misses)
        p.compare_state()
        p.compare_hot_rows(range(w.B))
    finally:
        p.close()


def test_layer_call_errors():
    w = wl.Workload("lerr", B=2, L=2, ctx=50, k=4, S=6, steps=2)
    p = Pair(w)
    try:
        t = torch.tensor([[1, 2, 3, 4], [5, 6, 7, 8]], dtype=torch.int32, device="cuda")
        out = torch.empty_like(t)
        hm = torch.empty(2, dtype=torch.int32, device="cuda")
        for bad in (-1, 2):
            with pytest.raises(SkvError, match="INVALID_ARG"):
                p.ctx.assemble_layer(bad, p.req_dev, t, out, hm, hm)
        p.ctx.assemble_layer(1, p.req_dev, t, out, hm, hm)
        assert p.orc.assemble_layer(1, p.req_ids, t.cpu().numpy())[0] == 0
        bad_rows = torch.tensor([[1, 2, 3, 4], [5, 6, 7, 50]], dtype=torch.int32, device="cuda")
        p.ctx.assemble_layer(0, p.req_dev, bad_rows, out, hm, hm)
        e, *_ = p.orc.assemble_layer(0, p.req_ids, bad_rows.cpu().numpy())
        assert e == orc.E_BAD_INDEX
        assert (out == -1).all() and (hm == -1).all()
        assert p.ctx.get_device_error() == p.orc.get_error() == orc.E_BAD_INDEX
        p.compare_state()
    finally:
        p.close()
