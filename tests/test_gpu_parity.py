"""CUDA library vs CPU oracle, bit-exact, on seeded workloads (GPU)."""
import numpy as np
import pytest
import torch

import skv_workload as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from skv_pair import Pair


def run(w, steps=None, state_every=4, req_perm=None, lifecycle=None):
    p = Pair(w, req_perm=req_perm)
    try:
        p.check_pool_rows()
        n = w.steps if steps is None else steps
        for s in range(n):
            if lifecycle is not None and s == lifecycle:
                p.lifecycle(1)
            p.step(s)
            if state_every and (s % state_every == state_every - 1 or s == n - 1):
                p.compare_state()
        p.compare_hot_rows(range(p.R))
        return p.total_misses
    finally:
        p.close()


def test_tiny_config_all_steps():
    """The tiny configuration (4 requests, 1 layer, 4096-token context, k=256,
    512 slots, 20% fresh, sorted rows), all 64 steps, full state each 4 steps."""
    misses = run(wl.WORKLOADS["c1_tiny"])
    assert misses > 4 * 256  # cold step plus steady-state misses happened


RAGGED = [
    # several CTAs' worth of units, ragged k and S (not multiples of 32 / 4 / the block)
    wl.Workload("ragged_shuffled_pad", B=5, L=3, ctx=5000, k=300, S=701, steps=12, fresh=0.3,
                order=wl.ORDER_SHUFFLED, n_pad=17),
    wl.Workload("ragged_sorted_pad", B=3, L=2, ctx=3000, k=257, S=300, steps=12, fresh=0.4, n_pad=9),
    wl.Workload("s_equals_k", B=4, L=2, ctx=2000, k=128, S=128, steps=10, fresh=0.5),
    wl.Workload("k_one", B=6, L=2, ctx=50, k=1, S=3, steps=20, fresh=1.0),
    wl.Workload("tiny_S_small_k", B=2, L=1, ctx=40, k=5, S=7, steps=30, fresh=0.6, order=wl.ORDER_SHUFFLED),
    wl.Workload("recency", B=4, L=2, ctx=9000, k=1000, S=1500, steps=10, fresh=0.4, dist=wl.DIST_RECENCY),
    wl.Workload("zipf", B=3, L=2, ctx=20000, k=512, S=1024, steps=10, fresh=0.2, dist=wl.DIST_ZIPF),
    wl.Workload("append", B=4, L=3, ctx=600, k=64, S=100, steps=16, fresh=0.3, appends=True),
    wl.Workload("max_k_max_S", B=2, L=1, ctx=40000, k=4096, S=16384, steps=6, fresh=0.3, order=wl.ORDER_SHUFFLED),
    wl.Workload("max_k_tight", B=2, L=1, ctx=20000, k=4096, S=4096, steps=6, fresh=0.5),
]


@pytest.mark.parametrize("w", RAGGED, ids=lambda w: w.name)
def test_ragged_and_edge_workloads(w):
    run(w)


@pytest.mark.parametrize("B,L,S", [(38, 4, 320), (50, 6, 320), (60, 9, 320), (38, 4, 4096), (50, 6, 4096)],
                         ids=["152_units", "300_units", "540_units", "152_units_S4096", "300_units_S4096"])
def test_launch_regimes_by_unit_count(B, L, S):
    """The fused kernel's three launch regimes: at most one unit per SM (one
    CTA to an SM with more loads in flight, the kernel starting while
    validation runs), more units than SMs but all resident at once, and more
    than fit at once (units in waves) -- each bit-exact against the oracle,
    with state compared at the end.  In every regime a few warps write the LRU
    order and the maps while the others gather; with S = 4096 the victim
    selection reads the LRU order 16 bytes at a time and the new order is built
    from whole bitmap words (S = 320 takes the one-slot-at-a-time paths)."""
    # with S = 4096, k = 2048 and 60 % fresh tokens a step fill the hot buffer by the third step
    k, steps, fresh = (192, 4, 0.3) if S < 1024 else (2048, 5, 0.6)
    w = wl.Workload(f"regime_{B * L}_{S}", B=B, L=L, ctx=max(2500, 2 * S), k=k, S=S, steps=steps, fresh=fresh,
                    order=wl.ORDER_SHUFFLED, n_pad=5)
    p = Pair(w)
    try:
        for s in range(w.steps):
            p.step(s)
        p.compare_state(reqs=[0, B // 2, B - 1])
        assert p.ctx.get_device_error() == 0
        if S >= 1024:
            assert p.total_misses > B * L * S  # more rows moved than slots: the later steps evicted
    finally:
        p.close()


def test_request_ids_permuted_and_sparse():
    """R > B: the batch uses a permuted subset of the published requests."""
    w = wl.Workload("perm", B=4, L=2, ctx=3000, k=200, S=400, steps=10, fresh=0.3, max_requests=7)
    run(w, req_perm=[5, 2, 6, 0])


def test_release_and_republish_mid_run():
    w = wl.Workload("life", B=3, L=2, ctx=4000, k=256, S=512, steps=12, fresh=0.2)
    run(w, lifecycle=6)


def test_empty_batch_is_a_no_op():
    w = wl.Workload("empty", B=2, L=1, ctx=500, k=16, S=32, steps=3)
    p = Pair(w)
    try:
        p.step(0)
        clock = p.ctx.clock()
        e = torch.empty(0, dtype=torch.int32, device="cuda")
        p.ctx.assemble(e, e, e, e, e, B=0)
        p.ctx.write_back(e, e, n=0)
        assert p.ctx.clock() == clock
        p.step(1)
        p.compare_state()
    finally:
        p.close()


def test_graph_capture_replays_the_step():
    """The whole step captured once in a CUDA graph and replayed with new
    inputs copied into its static input buffer matches the oracle."""
    w = wl.Workload("graph", B=4, L=2, ctx=6000, k=512, S=1024, steps=10, fresh=0.3, order=wl.ORDER_SHUFFLED)
    p = Pair(w)
    try:
        p.step(0)  # warm-up (also compiles nothing: kernels are prebuilt)
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                p.ctx.assemble(p.req_dev, p.topk_dev, p.slots_dev, p.hits_dev, p.misses_dev)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        # capture did not run anything: the state still matches the oracle
        p.compare_state()
        for step in range(1, w.steps):
            topk = p.gen.step(step, p.lens)
            p.topk_dev.copy_(torch.from_numpy(topk))
            g.replay()
            e, slots, hits, misses = p.orc.assemble(p.req_ids, topk)
            assert e == 0
            assert np.array_equal(p.slots_dev.cpu().numpy(), slots)
            assert np.array_equal(p.hits_dev.cpu().numpy(), hits)
            assert np.array_equal(p.misses_dev.cpu().numpy(), misses)
        p.compare_state()
    finally:
        p.close()


@pytest.mark.parametrize("outputs", ["pageable", "pinned", "mixed"])
def test_host_buffer_entry_point(outputs):
    """skv_assemble_host (host-memory inputs and outputs) matches the oracle,
    whether its outputs are pageable (staged and copied back), pinned (written
    by the kernels straight into host memory) or some of each."""
    w = wl.Workload("host", B=3, L=2, ctx=3000, k=300, S=512, steps=8, fresh=0.3)
    p = Pair(w)

    def out(shape, pinned):
        if not pinned:
            return np.full(shape, -7, np.int32)
        return torch.full(shape, -7, dtype=torch.int32).pin_memory()

    try:
        for s in range(w.steps):
            topk = p.gen.step(s, p.lens)
            req = np.array(p.req_ids, dtype=np.int32)
            slots = out(topk.shape, outputs != "pageable")
            hits = out((w.B, w.L), outputs == "pinned")
            misses = out((w.B, w.L), outputs != "pageable")
            p.ctx.assemble_host(req, topk, slots, hits, misses)
            slots, hits, misses = (np.asarray(x) if isinstance(x, np.ndarray) else x.numpy()
                                   for x in (slots, hits, misses))
            e, o_slots, o_hits, o_misses = p.orc.assemble(p.req_ids, topk)
            assert e == 0
            assert np.array_equal(slots, o_slots) and np.array_equal(hits, o_hits)
            assert np.array_equal(misses, o_misses)
        p.compare_state()
    finally:
        p.close()


def test_publish_with_rows_from_host_and_device():
    from sparse_attention_kv_skv_gb300 import Config, Context
    L, T_max, k, S = 2, 64, 4, 8
    rb = wl.ROW_BYTES
    with Context(Config(max_requests=3, num_layers=L, max_context=T_max, topk=k, hot_slots=S, max_batch=2,
                        row_bytes=rb)) as ctx:
        host_rows = np.stack([wl.fill_rows(1, 0, l, 0, 40) for l in range(L)])       # [L][T][rb]
        dev_rows = torch.from_numpy(np.stack([wl.fill_rows(1, 1, l, 0, 50) for l in range(L)])).cuda()
        r0 = ctx.publish(40, rows=host_rows)
        r1 = ctx.publish(50, rows=dev_rows)
        torch.cuda.synchronize()
        import ctypes
        base = ctx.pool_rows()
        view = np.frombuffer((ctypes.c_uint8 * (3 * L * T_max * rb)).from_address(base),
                             dtype=np.uint8).reshape(3, L, T_max, rb)
        assert (r0, r1) == (0, 1)
        assert np.array_equal(view[0, :, :40], host_rows)
        assert np.array_equal(view[1, :, :50], dev_rows.cpu().numpy())
        st = ctx.export_state(1)
        assert st["len"] == 50 and st["active"] == 1 and (st["slot2tok"] == -1).all()
        assert ctx.stats()["calls"] == 0
