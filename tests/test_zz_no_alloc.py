"""skv_assemble_noalloc -- the assemble step for callers that cannot allocate
device memory at call time (engines that reserve nearly all HBM up front,
code running inside someone else's stream capture) -- gives the same results
as skv_assemble.  Its gather work list is a static device array shared by all
calls; this file is collected last so that a failure here cannot hide other
tests' results.  (GPU)"""
import numpy as np
import pytest
import torch

import skv_workload as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from sparse_attention_kv_skv_gb300 import Config, Context, SkvError


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
