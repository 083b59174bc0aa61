"""skv_assemble_noalloc -- the assemble step for callers that cannot allocate
device memory at call time (engines that reserve nearly all HBM up front,
code running inside someone else's stream capture) -- gives the same results
as skv_assemble and as the CPU oracle: eagerly, replayed from a captured CUDA
graph, and with two contexts taking turns on the one static work list.  Its
first call on a device allocates nothing (checked in a fresh process).  This
file is collected last so that a failure here cannot hide other tests'
results.  (GPU)"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import skv_workload as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from sparse_attention_kv_skv_gb300 import Config, Context, SkvError
    from skv_pair import Pair

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _context(w):
    rb = wl.ROW_BYTES
    T_max = w.max_context
    ctx = Context(Config(max_requests=w.B, num_layers=w.L, max_context=T_max, topk=w.k, hot_slots=w.S,
                         max_batch=w.B, row_bytes=rb))
    pool = ctx.pool_rows()
    for r in range(w.B):
        assert ctx.publish(w.ctx) == r
    torch.cuda.synchronize()
    for r in range(w.B):
        wl.fill_request(pool + r * w.L * T_max * rb, w.L, T_max, w.ctx, w.base_seed, w.req_key(r))
    return ctx


def test_noalloc_matches_assemble_on_two_calls_in_a_row():
    w = wl.Workload("noalloc", B=6, L=4, ctx=20000, k=2048, S=4096, steps=2, fresh=0.3, order=wl.ORDER_SHUFFLED)
    ref, var = _context(w), _context(w)
    try:
        gen = wl.TopkStream(w)
        req = torch.arange(w.B, dtype=torch.int32, device="cuda")
        outs = {}
        for s in range(2):
            topk = torch.from_numpy(gen.step(s, [w.ctx] * w.B)).cuda()
            for name, ctx in (("ref", ref), ("var", var)):
                slots = torch.full_like(topk, -7)
                hits = torch.full((w.B, w.L), -7, dtype=torch.int32, device="cuda")
                misses = torch.full_like(hits, -7)
                if name == "ref":
                    ctx.assemble(req, topk, slots, hits, misses)
                else:
                    ctx.assemble_noalloc(req, topk, slots, hits, misses)
                outs[name] = (slots.cpu().numpy(), hits.cpu().numpy(), misses.cpu().numpy())
            for a, b in zip(outs["ref"], outs["var"]):
                assert np.array_equal(a, b), f"call {s}: outputs differ"
            assert outs["var"][2].sum() > 0   # rows were gathered
        assert ref.clock() == var.clock() == 2
        assert ref.get_device_error() == 0 and var.get_device_error() == 0
        for r in range(w.B):
            a, b = ref.export_state(r), var.export_state(r)
            for key in ("slot2tok", "ts", "lru", "tok2slot"):
                assert np.array_equal(a[key], b[key]), (r, key)
            assert np.array_equal(ref.export_hot(r), var.export_hot(r)), r
        gen.close()
    finally:
        ref.close()
        var.close()


def test_noalloc_rejects_calls_beyond_its_capacity():
    # B*L*k = 20 * 16 * 4096 = 1310720 > 2^20 entries; small rows keep this cheap
    with Context(Config(max_requests=20, num_layers=16, max_context=4096, topk=4096, hot_slots=4096,
                        max_batch=20, row_bytes=16)) as ctx:
        req = torch.arange(20, dtype=torch.int32, device="cuda")
        topk = torch.full((20, 16, 4096), -1, dtype=torch.int32, device="cuda")
        slots = torch.empty_like(topk)
        hm = torch.empty((20, 16), dtype=torch.int32, device="cuda")
        with pytest.raises(SkvError, match="INVALID_ARG"):
            ctx.assemble_noalloc(req, topk, slots, hm, hm)
        from sparse_attention_kv_skv_gb300 import skv
        assert b"exceeds the static work-list capacity" in skv.skv_last_cuda_error()
        # 16 requests fit exactly (16 * 16 * 4096 = 2^20)
        for r in range(16):
            ctx.publish(10)
        ctx.assemble_noalloc(req[:16], topk[:16], slots[:16], hm[:16], hm[:16], B=16)
        assert ctx.get_device_error() == 0 and ctx.clock() == 1


def test_noalloc_matches_the_oracle():
    """Ragged shapes, padded and shuffled rows, a permuted request subset:
    slots and counts every step, maps, LRU order and hot rows at the end."""
    w = wl.Workload("noalloc_orc", B=5, L=3, ctx=5000, k=300, S=701, steps=8, fresh=0.3,
                    order=wl.ORDER_SHUFFLED, n_pad=17, max_requests=7)
    p = Pair(w, req_perm=[6, 1, 4, 0, 3], entry="assemble_noalloc")
    try:
        for s in range(w.steps):
            p.step(s)
        p.compare_state()
        p.compare_hot_rows(range(p.R))
        assert p.ctx.get_device_error() == 0
    finally:
        p.close()


def test_noalloc_replays_from_a_captured_graph():
    """One eager call, then the call captured once and replayed with each
    step's new Top-k rows in the same input buffer; the oracle decides."""
    w = wl.Workload("noalloc_graph", B=4, L=2, ctx=6000, k=512, S=1024, steps=6, fresh=0.3)
    p = Pair(w, entry="assemble_noalloc")
    try:
        p.step(0)
        p.capture()
        for s in range(1, w.steps):
            p.step(s)
        p.compare_state()
        assert p.ctx.get_device_error() == 0
    finally:
        p.close()


def test_two_contexts_take_turns_on_the_static_work_list():
    """Two contexts of different shapes call the entry point one after the
    other on one stream; each matches its own oracle."""
    wa = wl.Workload("noalloc_a", B=3, L=2, ctx=4000, k=256, S=512, steps=5, fresh=0.4)
    wb = wl.Workload("noalloc_b", B=2, L=3, ctx=3000, k=200, S=333, steps=5, fresh=0.5, order=wl.ORDER_SHUFFLED)
    a = Pair(wa, entry="assemble_noalloc")
    b = Pair(wb, entry="assemble_noalloc")
    try:
        for s in range(5):
            a.step(s)
            b.step(s)
        a.compare_state()
        b.compare_state()
        assert a.ctx.get_device_error() == 0 and b.ctx.get_device_error() == 0
    finally:
        a.close()
        b.close()


FIRST_CALL = r"""
import sys
sys.path.insert(0, sys.argv[1])
import torch
from sparse_attention_kv_skv_gb300 import Config, Context
ctx = Context(Config(max_requests=4, num_layers=2, max_context=4096, topk=256, hot_slots=512, max_batch=4))
for r in range(4):
    ctx.publish(1000)
req = torch.arange(4, dtype=torch.int32, device="cuda")
topk = torch.arange(256, dtype=torch.int32, device="cuda").repeat(4, 2, 1).contiguous()
slots = torch.empty_like(topk)
hits = torch.empty((4, 2), dtype=torch.int32, device="cuda")
misses = torch.empty_like(hits)
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
ctx.assemble_noalloc(req, topk, slots, hits, misses)
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
assert ctx.get_device_error() == 0 and int(misses.sum()) == 4 * 2 * 256
ctx.close()
print("FREE", free0, free1)
"""


def test_first_call_in_a_fresh_process_allocates_nothing():
    """skv_create brings the static array into existence on the context's
    device, so the free device memory is the same before and after the first
    skv_assemble_noalloc call of a process."""
    r = subprocess.run([sys.executable, "-c", FIRST_CALL, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [x for x in r.stdout.splitlines() if x.startswith("FREE")][-1]
    free0, free1 = map(int, line.split()[1:])
    assert free0 == free1, f"free device memory changed by {free0 - free1} bytes at the first call"
