"""skv_attend (tensor-core sparse MLA attention over assembled slots) against
the fp64 attention oracle evaluated on the CPU oracle's own hot buffer (GPU).

Tolerance, from the arithmetic: q and the key rows are bf16, their products
are exact in fp32 and summed in fp32; the half of each score summed on the
other CTA of the pair crosses over as the upper 24 bits of its fp32 (relative
error <= 2^-16: under 5e-4 for the partials of these inputs, |partial| < 30,
so under 2e-4 in the exponent at scale 0.35); the probabilities P enter the second product rounded to bf16 (relative error
<= 2^-9), so |error of out| <= 2^-9 * max|V| = 2e-3 with |V| <= 1; the output
is rounded to bf16 (another 2^-9 |out|).  The test allows 6e-3 + 6e-3 |out|
(x3 margin) and 5e-3 on lse.
"""
import numpy as np
import pytest
import torch

import skv_workload as wl
from oracle import attention as att

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from skv_pair import Pair

ATOL, RTOL, LSE_ATOL = 6e-3, 6e-3, 5e-3


def _queries(w, units):
    """[units][128][576] bf16 for the given (b, l) list."""
    return np.stack([wl.fill_q(w.base_seed, b, l) for b, l in units]).view(np.uint16)


def _check_units(p, units, slots, q, out, lse, scale):
    hot_cache = {}
    for n, (b, l) in enumerate(units):
        r = p.req_ids[b]
        if r not in hot_cache:
            hot_cache[r] = p.orc.export_hot(r)
        row = slots[n]
        valid = row >= 0
        keys = np.zeros((row.size, 576))
        keys[valid] = att.bf16_rows_to_f64(hot_cache[r][l][row[valid]])
        want, want_lse = att.attend(att.bf16_rows_to_f64(q[n].view(np.uint8)), keys, valid, scale)
        got = att.bf16_rows_to_f64(out[n].view(np.uint8))
        err = np.abs(got - want) - (ATOL + RTOL * np.abs(want))
        assert err.max() <= 0, f"unit {(b, l)}: out off by {np.abs(got - want).max()}"
        both_inf = np.isneginf(want_lse) & np.isneginf(lse[n])
        diff = np.abs(np.where(both_inf, 0.0, lse[n] - want_lse))
        assert np.all(diff <= LSE_ATOL), f"unit {(b, l)}: lse"


@pytest.mark.parametrize("scale,sms", [(1.0 / 24.0, 0), (0.35, 0), (0.35, 4)])
def test_attention_over_assembled_slots(scale, sms):
    """sms = 4: two clusters walk the six units, three each (cross-unit pipeline)."""
    w = wl.Workload("attn", B=3, L=2, ctx=3000, k=300, S=512, steps=3, fresh=0.3, order=wl.ORDER_SHUFFLED,
                    n_pad=7)
    p = Pair(w, req_perm=[2, 0, 1])
    try:
        for s in range(w.steps):
            p.step(s)
        units = [(b, l) for b in range(w.B) for l in range(w.L)]
        q = _queries(w, units)
        q_d = torch.from_numpy(q).cuda()
        out_d = torch.full((len(units), 128, 512), 0x7FC0, dtype=torch.int16, device="cuda")
        lse_d = torch.full((len(units), 128), float("nan"), device="cuda")
        p.ctx.set_attend_sms(sms)
        p.ctx.attend(p.req_dev, q_d, p.slots_dev, out_d, lse_d, sm_scale=scale)
        slots = p.slots_dev.cpu().numpy().reshape(len(units), w.k)
        _check_units(p, units, slots, q, out_d.cpu().numpy().view(np.uint16), lse_d.cpu().numpy(), scale)
        assert p.ctx.get_device_error() == 0
    finally:
        p.close()


def test_attention_one_layer_and_fully_masked_units():
    w = wl.Workload("attn1", B=4, L=3, ctx=2500, k=256, S=400, steps=2, fresh=0.3)
    p = Pair(w)
    try:
        for s in range(w.steps):
            p.step(s)
        layer = 1
        # one batch entry selects nothing in this layer: all -1
        topk = p.gen.step(w.steps, p.lens)[:, layer, :].copy()
        topk[2, :] = -1
        t_d = torch.from_numpy(topk).cuda()
        slots_d = torch.empty_like(t_d)
        hm = torch.empty(w.B, dtype=torch.int32, device="cuda")
        p.ctx.assemble_layer(layer, p.req_dev, t_d, slots_d, hm, hm.clone())
        e, o_slots, _, _ = p.orc.assemble_layer(layer, p.req_ids, topk)
        assert e == 0 and np.array_equal(slots_d.cpu().numpy(), o_slots)
        units = [(b, layer) for b in range(w.B)]
        q = _queries(w, units)
        out_d = torch.empty((w.B, 128, 512), dtype=torch.int16, device="cuda")
        lse_d = torch.empty((w.B, 128), device="cuda")
        p.ctx.attend(p.req_dev, torch.from_numpy(q).cuda(), slots_d, out_d, lse_d, layer=layer, sm_scale=0.2)
        out = out_d.cpu().numpy().view(np.uint16)
        lse = lse_d.cpu().numpy()
        _check_units(p, units, o_slots, q, out, lse, 0.2)
        assert not out[2].any() and np.all(np.isneginf(lse[2]))
    finally:
        p.close()


@pytest.mark.parametrize("k,S,ctx", [(20, 64, 700), (40, 64, 700), (4096, 4096, 6000)])
def test_attention_short_topk_and_non_request(k, S, ctx):
    """One and two key blocks (the pipeline never fills) and the largest Top-k
    (k = 4096: 64 blocks), plus an entry whose request id is not a request:
    zero output and lse = -inf for it."""
    w = wl.Workload(f"attn_k{k}", B=3, L=2, ctx=ctx, k=k, S=S, steps=2, fresh=0.5)
    p = Pair(w)
    try:
        for s in range(w.steps):
            p.step(s)
        units = [(b, l) for b in range(w.B) for l in range(w.L)]
        q = _queries(w, units)
        req = p.req_dev.clone()
        req[1] = -1
        out_d = torch.full((len(units), 128, 512), 0x7FC0, dtype=torch.int16, device="cuda")
        lse_d = torch.full((len(units), 128), float("nan"), device="cuda")
        p.ctx.attend(req, torch.from_numpy(q).cuda(), p.slots_dev, out_d, lse_d, sm_scale=0.3)
        out = out_d.cpu().numpy().view(np.uint16)
        lse = lse_d.cpu().numpy()
        slots = p.slots_dev.cpu().numpy().reshape(len(units), w.k)
        keep = [n for n, (b, _) in enumerate(units) if b != 1]
        _check_units(p, [units[n] for n in keep], slots[keep], q[keep], out[keep], lse[keep], 0.3)
        for n, (b, _) in enumerate(units):
            if b == 1:
                assert not out[n].any() and np.all(np.isneginf(lse[n]))
        assert p.ctx.get_device_error() == 0
    finally:
        p.close()


@pytest.mark.fullsize
def test_attention_full_size_sampled():
    """The bench's launch configuration: the 192 x 8 target workload (k = 2048,
    S = 4096) after a cold and two steady steps, one call over all 1536 units;
    a spread of units is checked against the definition on the oracle's hot
    buffer."""
    w = wl.WORKLOADS["target_16k_b192_f20"]
    p = Pair(w)
    try:
        for s in range(3):
            p.step(s)
        units = [(b, l) for b in range(w.B) for l in range(w.L)]
        q = _queries(w, units)
        out_d = torch.full((len(units), 128, 512), 0x7FC0, dtype=torch.int16, device="cuda")
        lse_d = torch.full((len(units), 128), float("nan"), device="cuda")
        scale = 1.0 / 576 ** 0.5
        p.ctx.attend(p.req_dev, torch.from_numpy(q).cuda(), p.slots_dev, out_d, lse_d, sm_scale=scale)
        torch.cuda.synchronize()
        assert p.ctx.get_device_error() == 0
        pick = [n for n, (b, l) in enumerate(units)
                if (b, l) in {(0, 0), (0, 7), (1, 3), (63, 5), (95, 4), (127, 1), (190, 6), (191, 7)}]
        slots = p.slots_dev.cpu().numpy().reshape(len(units), w.k)[pick]
        out = out_d.cpu().numpy().view(np.uint16)[pick]
        lse = lse_d.cpu().numpy()[pick]
        _check_units(p, [units[n] for n in pick], slots, q[pick], out, lse, scale)
        assert np.isfinite(lse_d.cpu().numpy()).all()  # every unit of the call produced a result
    finally:
        p.close()


def test_attention_beside_layer_assembly_on_another_stream():
    """Layer l's attention (limited to 8 SMs: four clusters walking 16 units each) runs on
    its own stream while layer l + 1 is assembled on another, as a pipelined decode step
    does; every unit is checked against the definition, and no wait may give up."""
    w = wl.Workload("attn_pipe", B=64, L=3, ctx=3000, k=320, S=512, steps=3, fresh=0.3)
    p = Pair(w)
    side = torch.cuda.Stream()
    try:
        for s in range(w.steps - 1):
            p.step(s)
        topk = p.gen.step(w.steps - 1, p.lens)
        rows = [torch.from_numpy(np.ascontiguousarray(topk[:, l, :])).cuda() for l in range(w.L)]
        slots_l = [torch.empty((w.B, w.k), dtype=torch.int32, device="cuda") for _ in range(w.L)]
        hm = torch.empty((w.L, w.B), dtype=torch.int32, device="cuda")
        q = np.stack([_queries(w, [(b, l) for b in range(w.B)]) for l in range(w.L)])
        q_d = torch.from_numpy(q).cuda()
        out_d = torch.empty((w.L, w.B, 128, 512), dtype=torch.int16, device="cuda")
        lse_d = torch.empty((w.L, w.B, 128), device="cuda")
        p.ctx.set_attend_sms(8)
        main = torch.cuda.current_stream()
        done = [torch.cuda.Event() for _ in range(w.L)]
        for l in range(w.L):
            p.ctx.assemble_layer(l, p.req_dev, rows[l], slots_l[l], hm[l], hm[l].clone(), stream=main.cuda_stream)
            done[l].record(main)
            side.wait_event(done[l])
            p.ctx.attend(p.req_dev, q_d[l], slots_l[l], out_d[l], lse_d[l], layer=l, sm_scale=0.3,
                         stream=side.cuda_stream)
        torch.cuda.synchronize()
        assert p.ctx.get_device_error() == 0
        for l in range(w.L):
            e, o_slots, _, _ = p.orc.assemble_layer(l, p.req_ids, topk[:, l, :].copy())
            assert e == 0 and np.array_equal(slots_l[l].cpu().numpy(), o_slots)
            _check_units(p, [(b, l) for b in range(w.B)], o_slots, q[l], out_d[l].cpu().numpy().view(np.uint16),
                         lse_d[l].cpu().numpy(), 0.3)
    finally:
        p.close()
