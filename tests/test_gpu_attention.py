"""skv_attend (tensor-core sparse MLA attention over assembled slots) against
the fp64 attention oracle evaluated on the CPU oracle's own hot buffer (GPU).

Every tolerance is derived from the kernel's arithmetic, per unit and head,
from the unit's own q and keys (``bounds``):

  score error.  q and the key rows are bf16, so every product q_d k_d is exact
  in fp32.  A score is summed in two halves (dims [0, 288) on one CTA of the
  pair, [288, 576) on the other), each over 18 tensor-core steps of 16
  products with fp32 accumulation, and the halves are added in fp32: taking
  each step's rounding as at most 2^-22 of the magnitude it sums (generous for
  fp32's 2^-24), the error is at most 19 * 2^-22 * A with A = sum_d |q_d k_d|.
  One of the two halves crosses the pair as the upper 24 bits of its fp32
  (round to nearest: relative error at most 2^-16 of that partial P).  So a
  scaled score is off by at most
      ds = scale * (2^-16 * max(|P0|, |P1|) + 19 * 2^-22 * A).
  lse.  lse = log sum_j exp(s_j) moves by at most max_j ds_j when every s_j
  moves by at most ds_j; the rest -- ex2.approx (relative error about 2^-22 a
  term), the fp32 sums of the denominator (at most k/32 + 64 roundings of
  2^-24 along any chain), log2f and the final scaling -- stays below
  1e-5 + (k/32 + 64) * 2^-24.  At scale 0.35 on these inputs that is about
  5e-4; at scale 1/24 about 6e-5, while one dropped key of a flat softmax over
  k keys moves lse by about 1/k.
  out.  P enters the value product rounded to bf16 (relative error at most
  2^-8 each, so at most 2^-8 * max|V| on the normalised output), score errors
  change the normalised weights by at most a factor exp(2 ds), and the output
  is rounded to bf16 (at most 2^-8 |out|):
      |out - want| <= (2^-8 + 2 ds) * max|V| + (2^-8 + 1e-5) |want|.
Planted-key cases put one key whose score is about 8 above the others at a
chosen position (0, 63, 64, 65, k - 1) of a unit's slot list, with a masked
slot among the others, for k on and next to the 64-key block boundary: a key
that is dropped, duplicated or moved to another position breaks them.
"""
import numpy as np
import pytest
import torch

import skv_workload as wl
from attention_check import check_unit
from oracle import attention as att

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from skv_pair import Pair


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
        check_unit(q[n], keys, valid, out[n], lse[n], scale, f"unit {(b, l)}")


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


PLANT_POS = (0, 63, 64, 65, -1)   # -1: the last position, k - 1
PLANT_HEADS = (0, 37, 64, 127)    # heads of different warps and lanes


@pytest.mark.parametrize("k", [63, 64, 65, 127, 128, 129, 2048])
def test_planted_key_at_block_boundaries(k):
    """Unit (b, l) holds k distinct tokens in shuffled order with one -1 slot;
    the token at position PLANT_POS[b] is planted: heads PLANT_HEADS of q are
    its own key row, so its score (scale 0.05 * |key|^2, about 9.6) stands
    about 8 above every other.  The other heads are uniform queries, whose
    nearly flat softmax makes lse move by about 1/k for a key that is dropped.
    Run with every SM and with one cluster walking all ten units in turn."""
    B, L, scale = 5, 2, 0.05
    w = wl.Workload(f"plant_k{k}", B=B, L=L, ctx=max(3000, 2 * k + 100), k=k, S=k + 37, steps=1)
    p = Pair(w)
    try:
        rng = np.random.default_rng(1000 + k)
        topk = np.empty((B, L, k), np.int32)
        plant = {}
        for b in range(B):
            pos = PLANT_POS[b] if 0 <= PLANT_POS[b] < k else k - 1
            for l in range(L):
                row = rng.permutation(w.ctx)[:k].astype(np.int32)
                row[(pos + 1 + int(rng.integers(k - 1))) % k] = -1  # one masked slot, never the planted one
                topk[b, l] = row
                plant[(b, l)] = (pos, int(row[pos]))
        p.ctx.assemble(p.req_dev, torch.from_numpy(topk).cuda(), p.slots_dev, p.hits_dev, p.misses_dev)
        e, o_slots, _, _ = p.orc.assemble(p.req_ids, topk)
        assert e == 0 and np.array_equal(p.slots_dev.cpu().numpy(), o_slots)
        units = [(b, l) for b in range(B) for l in range(L)]
        slots = o_slots.reshape(len(units), k)
        q = _queries(w, units).copy()
        for n, (b, l) in enumerate(units):
            pos, tok = plant[(b, l)]
            assert slots[n, pos] >= 0 and (slots[n] < 0).sum() == 1
            krow = p.pool_view(p.req_ids[b])[l, tok].view(np.uint16)
            for h in PLANT_HEADS:
                q[n, h] = krow
            # the construction does what it says: the planted score leads by more than 6
            hot = p.orc.export_hot(p.req_ids[b])[l]
            keys = att.bf16_rows_to_f64(hot[slots[n][slots[n] >= 0]])
            kp = att.bf16_rows_to_f64(krow.view(np.uint8))
            sc = scale * keys @ kp
            top2 = np.sort(sc)[-2:]
            assert top2[1] == pytest.approx(scale * kp @ kp) and top2[1] - top2[0] > 6
        q_d = torch.from_numpy(q).cuda()
        for sms in (0, 2):
            out_d = torch.full((len(units), 128, 512), 0x7FC0, dtype=torch.int16, device="cuda")
            lse_d = torch.full((len(units), 128), float("nan"), device="cuda")
            p.ctx.set_attend_sms(sms)
            p.ctx.attend(p.req_dev, q_d, p.slots_dev, out_d, lse_d, sm_scale=scale)
            out = out_d.cpu().numpy().view(np.uint16)
            lse = lse_d.cpu().numpy()
            _check_units(p, units, slots, q, out, lse, scale)
            assert p.ctx.get_device_error() == 0
    finally:
        p.close()


def test_attention_wait_that_runs_out_reports_timeout():
    """The kernel's bounded waits, made to run out without endangering the
    GPU: skv_selftest_attend_timeout launches the attention kernel with its key
    loads withheld, so its first wait for keys gives up with nothing in flight.
    The sticky word then carries SKV_DEVERR_TIMEOUT, and the context stays
    usable: a normal call over the same slots is right afterwards, and the
    assembly goes on bit-exact."""
    from sparse_attention_kv_skv_gb300 import skv
    w = wl.Workload("attn_timeout", B=2, L=2, ctx=2000, k=128, S=256, steps=3, fresh=0.3)
    p = Pair(w)
    try:
        p.step(0)
        units = [(b, l) for b in range(w.B) for l in range(w.L)]
        q = _queries(w, units)
        q_d = torch.from_numpy(q).cuda()
        out_d = torch.empty((len(units), 128, 512), dtype=torch.int16, device="cuda")
        lse_d = torch.empty((len(units), 128), device="cuda")
        p.ctx.selftest_attend_timeout(p.req_dev, q_d, p.slots_dev, out_d)
        torch.cuda.synchronize()
        assert p.ctx.get_device_error() == skv.SKV_DEVERR_TIMEOUT
        assert p.ctx.get_device_error() == 0  # read and cleared
        p.ctx.attend(p.req_dev, q_d, p.slots_dev, out_d, lse_d, sm_scale=0.2)
        slots = p.slots_dev.cpu().numpy().reshape(len(units), w.k)
        _check_units(p, units, slots, q, out_d.cpu().numpy().view(np.uint16), lse_d.cpu().numpy(), 0.2)
        assert p.ctx.get_device_error() == 0
        p.step(1)
        p.step(2)
        p.compare_state()
    finally:
        p.close()
