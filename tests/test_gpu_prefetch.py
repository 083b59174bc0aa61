"""skv_prefetch / skv_prefetch_recent against the oracle (GPU).

A prefetch is an assemble of candidate tokens whose slot tensor is not
handed out, so everything it changes is compared bit-exactly: hit and miss
counts, clocks, maps, last-use stamps, LRU order and hot-buffer bytes.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import skv_workload as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from skv_pair import Pair


def _counts(w, layer):
    shape = (w.B, w.L) if layer < 0 else (w.B,)
    return (torch.full(shape, -7, dtype=torch.int32, device="cuda"),
            torch.full(shape, -7, dtype=torch.int32, device="cuda"))


def _check_counts(hits, misses, want_hits, want_misses, what):
    assert np.array_equal(hits.cpu().numpy(), want_hits), f"{what}: hits differ"
    assert np.array_equal(misses.cpu().numpy(), want_misses), f"{what}: misses differ"


def test_recency_prefetch_between_steps():
    """Recency-biased Top-k with appends: before every step, a window prefetch
    (every layer, or one layer, windows of 0 to k tokens, read after the last
    write back), then the step itself."""
    w = wl.Workload("pf_recency", B=6, L=3, ctx=3000, k=256, S=512, steps=7, fresh=0.4, dist=wl.DIST_RECENCY,
                    window=512, appends=True, max_requests=8)
    p = Pair(w, req_perm=[3, 1, 5, 0, 7, 4])
    try:
        windows = [256, 100, 0, 256, 37, 200, 256]
        for s in range(w.steps):
            layer = -1 if s % 2 == 0 else s % w.L
            hits, misses = _counts(w, layer)
            p.ctx.prefetch_recent(p.req_dev, windows[s], layer=layer, hits=hits, misses=misses)
            e, oh, om = p.orc.prefetch_recent(p.req_ids, windows[s], layer=layer)
            assert e == 0
            _check_counts(hits, misses, oh, om, f"prefetch before step {s}")
            p.compare_state(hot=s % 3 == 0)
            p.step(s)
        p.compare_state()
        assert p.ctx.get_device_error() == 0
    finally:
        p.close()


def test_candidate_prefetch_captured_and_rejected():
    """Caller-given candidates (shuffled, padded, partly resident), eagerly and
    replayed from a CUDA graph together with the step; a candidate beyond a
    request's length rejects the whole prefetch and changes nothing."""
    w = wl.Workload("pf_cand", B=4, L=2, ctx=2000, k=128, S=300, steps=5, fresh=0.3)
    p = Pair(w)
    rng = np.random.default_rng(17)
    cand_dev = torch.empty((w.B, w.L, w.k), dtype=torch.int32, device="cuda")
    hits, misses = _counts(w, -1)

    def draw():
        c = np.full((w.B, w.L, w.k), -1, dtype=np.int32)
        for b in range(w.B):
            for l in range(w.L):
                n = int(rng.integers(0, w.k + 1))
                c[b, l, :n] = rng.choice(p.lens[b], size=n, replace=False)
                rng.shuffle(c[b, l])
        return c

    try:
        p.step(0)
        for s in range(1, 3):  # eager
            c = draw()
            cand_dev.copy_(torch.from_numpy(c))
            p.ctx.prefetch(p.req_dev, cand_dev, hits=hits, misses=misses)
            e, oh, om = p.orc.prefetch(p.req_ids, c)
            assert e == 0
            _check_counts(hits, misses, oh, om, f"prefetch {s}")
            p.step(s)
        p.compare_state()
        # one layer, no counts asked for
        c1 = draw()[:, 1, :].copy()
        cand1 = torch.from_numpy(c1).cuda()
        p.ctx.prefetch(p.req_dev, cand1, layer=1)
        assert p.orc.prefetch(p.req_ids, c1, layer=1)[0] == 0
        p.compare_state()
        # replayed: prefetch of the static candidate buffer, then the step
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                p.ctx.prefetch(p.req_dev, cand_dev, hits=hits, misses=misses)
                p.ctx.assemble(p.req_dev, p.topk_dev, p.slots_dev, p.hits_dev, p.misses_dev)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        for s in range(3, w.steps):
            c = draw()
            topk = p.gen.step(s, p.lens)
            cand_dev.copy_(torch.from_numpy(c))
            p.topk_dev.copy_(torch.from_numpy(topk))
            graph.replay()
            e, oh, om = p.orc.prefetch(p.req_ids, c)
            assert e == 0
            _check_counts(hits, misses, oh, om, f"replayed prefetch {s}")
            e, slots, sh, sm = p.orc.assemble(p.req_ids, topk)
            assert e == 0 and np.array_equal(p.slots_dev.cpu().numpy(), slots)
            _check_counts(p.hits_dev, p.misses_dev, sh, sm, f"replayed step {s}")
        p.compare_state()
        # rejected whole
        bad = draw()
        bad[2, 1, 0] = p.lens[2]
        cand_dev.copy_(torch.from_numpy(bad))
        p.ctx.prefetch(p.req_dev, cand_dev, hits=hits, misses=misses)
        e, oh, om = p.orc.prefetch(p.req_ids, bad)
        assert e == orc.E_BAD_INDEX
        assert (hits.cpu().numpy() == -1).all() and (misses.cpu().numpy() == -1).all()
        assert p.ctx.get_device_error() == e and p.orc.get_error() == e
        p.compare_state()
    finally:
        p.close()


def test_recency_prefetch_keeps_the_window_resident():
    """With the recency window prefetched before every step, no step misses a
    token of the window (its misses are all older picks), and the steps miss
    fewer rows in total than the same steps without the prefetch."""
    w = wl.Workload("pf_effect", B=4, L=2, ctx=4096, k=512, S=1024, steps=6, fresh=0.4, dist=wl.DIST_RECENCY,
                    window=512, p_window=0.7)
    with_pf, without = Pair(w), Pair(w)
    try:
        for s in range(w.steps):
            if s > 0:
                with_pf.ctx.prefetch_recent(with_pf.req_dev, w.window)
                assert with_pf.orc.prefetch_recent(with_pf.req_ids, w.window)[0] == 0
            topk, _, _, misses = with_pf.step(s)
            without.step(s)
            if s > 0:
                older = ((topk >= 0) & (topk < w.ctx - w.window)).sum(axis=2)
                assert (misses <= older).all(), f"step {s}: a window token missed"
        with_pf.compare_state()
        assert with_pf.total_misses < without.total_misses
        assert with_pf.ctx.get_device_error() == 0 and without.ctx.get_device_error() == 0
    finally:
        with_pf.close()
        without.close()


def test_prefetch_argument_checks():
    """Host-side checks: a layer outside [-1, L), a window outside [0, k], a
    missing candidate tensor -- rejected before anything is enqueued."""
    from sparse_attention_kv_skv_gb300 import skv
    w = wl.Workload("pf_args", B=2, L=2, ctx=300, k=16, S=32, steps=1)
    p = Pair(w)
    try:
        clock = p.ctx.clock()
        cand = torch.full((w.B, w.L, w.k), -1, dtype=torch.int32, device="cuda")
        req = p.req_dev.data_ptr()
        assert skv.skv_prefetch_recent(p.ctx.h, req, w.B, w.L, 4, None, None, None) == skv.SKV_ERR_INVALID_ARG
        assert skv.skv_prefetch_recent(p.ctx.h, req, w.B, -2, 4, None, None, None) == skv.SKV_ERR_INVALID_ARG
        assert skv.skv_prefetch_recent(p.ctx.h, req, w.B, -1, w.k + 1, None, None, None) == skv.SKV_ERR_INVALID_ARG
        assert skv.skv_prefetch_recent(p.ctx.h, req, w.B, -1, -1, None, None, None) == skv.SKV_ERR_INVALID_ARG
        assert skv.skv_prefetch_recent(p.ctx.h, req, w.B + 1, -1, 4, None, None, None) == skv.SKV_ERR_INVALID_ARG
        assert skv.skv_prefetch(p.ctx.h, req, w.B, -1, None, None, None, None) == skv.SKV_ERR_INVALID_ARG
        assert skv.skv_prefetch(p.ctx.h, req, w.B, w.L, cand.data_ptr(), None, None, None) == skv.SKV_ERR_INVALID_ARG
        assert skv.skv_prefetch(p.ctx.h, req, 0, -1, cand.data_ptr(), None, None, None) == skv.SKV_OK  # B = 0: no-op
        assert skv.skv_prefetch_recent(p.ctx.h, req, w.B, -1, 0, None, None, None) == skv.SKV_OK  # empty window
        torch.cuda.synchronize()
        assert p.ctx.clock() == clock + 1  # only the empty-window prefetch ran (an all -1 call still ticks)
        assert p.orc.prefetch_recent(p.req_ids, 0)[0] == 0
        p.compare_state()
        assert p.ctx.get_device_error() == 0
    finally:
        p.close()
