"""Device-detected errors: the CUDA library rejects exactly what the oracle
rejects, with the same bits, -1 outputs and no state change (GPU)."""
import numpy as np
import pytest
import torch

import oracle as orc
import skv_workload as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from skv_pair import Pair
    from sparse_attention_kv_skv_gb300 import SkvError


def _assemble_both(p, req, topk):
    B = len(req)
    req_dev = torch.tensor(req, dtype=torch.int32, device="cuda")
    topk = np.asarray(topk, dtype=np.int32).reshape(B, p.w.L, p.w.k)
    t_dev = torch.from_numpy(topk).cuda()
    slots = torch.full_like(t_dev, 7)
    hits = torch.full((B, p.w.L), 7, dtype=torch.int32, device="cuda")
    misses = torch.full_like(hits, 7)
    p.ctx.assemble(req_dev, t_dev, slots, hits, misses, B=B)
    e, o_slots, o_hits, o_misses = p.orc.assemble(req, topk)
    assert np.array_equal(slots.cpu().numpy(), o_slots)
    assert np.array_equal(hits.cpu().numpy(), o_hits)
    assert np.array_equal(misses.cpu().numpy(), o_misses)
    return e


def test_bad_inputs_rejected_like_the_oracle():
    w = wl.Workload("err", B=2, L=2, ctx=50, k=4, S=6, steps=2, max_requests=3)
    p = Pair(w)
    try:
        good = [[[1, 2, 3, 4], [5, 6, 7, 8]], [[9, 10, 11, 12], [1, 3, 5, 7]]]
        assert _assemble_both(p, [0, 1], good) == 0
        # request 2 is published by Pair (R = 3); release it to make it inactive
        p.ctx.release(2)
        assert p.orc.release(2) == 0
        cases = [
            ([0, 1], [[[1, 2, 3, 50], [5, 6, 7, 8]], [[9, 10, 11, 12], [1, 3, 5, 7]]], orc.E_BAD_INDEX),
            ([0, 1], [[[1, 2, 3, -2], [5, 6, 7, 8]], [[9, 10, 11, 12], [1, 3, 5, 7]]], orc.E_BAD_INDEX),
            ([0, 1], [[[1, 2, 3, 4], [5, 6, 7, 8]], [[9, 10, 11, 12], [1, 3, 5, 5]]], orc.E_DUPLICATE),
            ([0, 1], [[[1, 2, 3, 4], [5, 6, 7, 8]], [[9, 9, 11, 60], [1, 3, 5, 7]]],
             orc.E_DUPLICATE | orc.E_BAD_INDEX),
            ([0, 0], good, orc.E_BAD_REQUEST),
            ([0, 2], good, orc.E_BAD_REQUEST),
            ([0, 3], good, orc.E_BAD_REQUEST),
            ([-1, 1], good, orc.E_BAD_REQUEST),
            ([1, 0], [[[-1, -1, -1, -1], [5, -1, 7, 8]], [[9, 10, 11, 12], [2, -3, 5, 7]]], orc.E_BAD_INDEX),
        ]
        for req, rows, bits in cases:
            e = _assemble_both(p, req, rows)
            assert e == bits, (req, rows, e)
            assert p.ctx.get_device_error() == bits
            assert p.orc.get_error() == bits
            assert p.ctx.get_device_error() == 0
            p.compare_state(reqs=[0, 1])
        # sticky: a valid call after an error is a no-op until the word is read
        assert _assemble_both(p, [0, 1], cases[0][1]) == orc.E_BAD_INDEX
        assert _assemble_both(p, [0, 1], good) == orc.E_BAD_INDEX
        p.compare_state(reqs=[0, 1])
        assert p.ctx.get_device_error() == orc.E_BAD_INDEX and p.orc.get_error() == orc.E_BAD_INDEX
        # padding only, repeated -1s
        assert _assemble_both(p, [0, 1], [[[-1, 2, -1, 4], [5, -1, 7, 8]], [[9, 10, -1, -1], [-1] * 4]]) == 0
        p.compare_state(reqs=[0, 1])
    finally:
        p.close()


def test_write_back_errors_and_context_full():
    w = wl.Workload("wb", B=2, L=2, ctx=10, k=2, S=4, steps=2, appends=True, max_requests=3)
    p = Pair(w)   # max_context = ctx + steps = 12
    try:
        rows = torch.zeros((2, w.L, wl.ROW_BYTES), dtype=torch.uint8, device="cuda")
        rows_np = np.zeros((2, w.L, wl.ROW_BYTES), np.uint8)

        def wb(req):
            n = len(req)
            p.ctx.write_back(torch.tensor(req, dtype=torch.int32, device="cuda"), rows[:n], n=n)
            e = p.orc.write_back(req, rows_np[:n])
            g = p.ctx.get_device_error()
            assert g == e == p.orc.get_error(), (req, g, e)
            return e

        assert wb([0, 0]) == orc.E_BAD_REQUEST
        assert wb([0, 5]) == orc.E_BAD_REQUEST
        assert wb([1, 0]) == 0
        assert wb([1]) == 0
        assert wb([1, 0]) == orc.E_CONTEXT_FULL
        p.compare_state(reqs=[0, 1, 2], hot=False)
        assert p.ctx.export_state(0)["len"] == 11 and p.ctx.export_state(1)["len"] == 12
    finally:
        p.close()


def test_host_checked_errors():
    from sparse_attention_kv_skv_gb300 import Config, Context
    with Context(Config(max_requests=2, num_layers=1, max_context=8, topk=2, hot_slots=2, max_batch=2)) as ctx:
        with pytest.raises(SkvError, match="CONTEXT_FULL"):
            ctx.publish(9)
        assert ctx.publish(8) == 0 and ctx.publish(3) == 1
        with pytest.raises(SkvError, match="NO_FREE_REQUEST"):
            ctx.publish(1)
        with pytest.raises(SkvError, match="BAD_REQUEST"):
            ctx.release(2)
        ctx.release(1)
        with pytest.raises(SkvError, match="BAD_REQUEST"):
            ctx.release(1)
        e = torch.zeros(8, dtype=torch.int32, device="cuda")
        with pytest.raises(SkvError, match="INVALID_ARG"):
            ctx.assemble(e, e, e, e, e, B=3)       # B > max_batch
        with pytest.raises(SkvError, match="INVALID_ARG"):
            ctx.assemble(e, e, e, e, e, B=-1)
        with pytest.raises(SkvError, match="INVALID_ARG"):
            ctx.write_back(e, e, n=3)
        with pytest.raises(SkvError, match="INVALID_ARG"):
            ctx.assemble(None, e, e, e, e, B=1)
        assert ctx.get_device_error() == 0


def _rss_bytes() -> int:
    for line in open("/proc/self/status"):
        if line.startswith("VmRSS:"):
            return int(line.split()[1]) * 1024
    return 0


def test_allocation_failure_at_create_frees_everything(monkeypatch):
    """Each of skv_create's 17 allocations made to fail in turn (a host-side
    fake of the failing call, SKV_TEST_FAIL_ALLOC): the create returns
    SKV_ERR_OOM, nothing is left behind (device memory and resident host
    memory as before, over repeated attempts), and a later create succeeds."""
    from sparse_attention_kv_skv_gb300 import Config, Context, skv
    cfg = Config(max_requests=8, num_layers=2, max_context=32768, topk=256, hot_slots=4096, max_batch=8)
    monkeypatch.delenv("SKV_TEST_FAIL_ALLOC", raising=False)
    Context(cfg).close()  # the first create of the process loads code; measure after it
    torch.cuda.synchronize()
    free0, rss0 = torch.cuda.mem_get_info()[0], _rss_bytes()
    for rounds in range(2):
        for n in range(1, 18):
            monkeypatch.setenv("SKV_TEST_FAIL_ALLOC", str(n))
            with pytest.raises(SkvError) as e:
                Context(cfg)
            assert e.value.status == skv.SKV_ERR_OOM, (n, e.value)
            assert b"out of memory" in skv.skv_last_cuda_error(), n
    torch.cuda.synchronize()
    free1, rss1 = torch.cuda.mem_get_info()[0], _rss_bytes()
    assert free1 == free0, f"device memory leaked: {free0 - free1} bytes"
    # the pool alone is 8 x 2 x 32768 rows x 1152 B = 604 MB; 34 leaked pools would be 20 GB
    assert rss1 - rss0 < 256 << 20, f"host memory grew by {(rss1 - rss0) >> 20} MiB"
    monkeypatch.setenv("SKV_TEST_FAIL_ALLOC", "18")  # past the last allocation: nothing fails
    with Context(cfg) as ctx:
        assert ctx.publish(100) == 0 and ctx.clock() == 0
    monkeypatch.delenv("SKV_TEST_FAIL_ALLOC")
