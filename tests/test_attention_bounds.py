"""The attention parity bounds (tests/attention_check.py) on the CPU: they
admit the kernel's documented roundings, emulated here (24-bit exchange of
one partial score, fp32 sums, P and the output rounded to bf16), and they
reject planted mistakes that a kernel could make -- a dropped key, a key
taken from the neighbouring position across a 64-key block boundary, a
masked slot read as a zero key.  (CPU)"""
import numpy as np
import pytest

import skv_workload as wl
from attention_check import check_unit
from oracle import attention as att


def to_bf16_bits(x) -> np.ndarray:
    """float -> bf16 bits, round to nearest even (via fp32)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def upper24(x32: np.ndarray) -> np.ndarray:
    """The upper 24 bits of an fp32, rounded to nearest (how a partial score crosses the CTA pair)."""
    b = x32.view(np.uint32).astype(np.uint64)
    return (((b + 0x80) >> 8) << 8).astype(np.uint32).view(np.float32)


def unit_inputs(k: int, seed: int = 3, planted: int | None = None, scale: float = 1 / 24):
    keys_bits = wl.fill_rows(seed, 7, 0, 0, k)                 # [k][1152] bf16 bytes
    keys = att.bf16_rows_to_f64(keys_bits)
    q = wl.fill_q(seed, 0, 0).view(np.uint16).copy()         # [128][576] bf16 bits
    if planted is not None:
        for h in (0, 37, 64, 127):
            q[h] = keys_bits[planted].view(np.uint16)
    return q, keys, np.ones(k, bool), scale


def emulate_kernel(q_bits, keys, valid, scale):
    """The kernel's arithmetic as the bounds model it: per key two fp32 half
    scores, one of them rounded to 24 bits, summed in fp32; p = 2^(s - m) in
    fp32; the value product with P rounded to bf16; the output rounded to bf16."""
    q = att.bf16_rows_to_f64(q_bits.view(np.uint8)).astype(np.float32)
    kv = keys[valid].astype(np.float32)
    p0 = (q[:, :288] @ kv[:, :288].T).astype(np.float32)
    p1 = (q[:, 288:] @ kv[:, 288:].T).astype(np.float32)
    s = (p0 + upper24(p1)).astype(np.float32)
    sl2 = np.float32(scale * 1.4426950408889634)
    m = (s.max(axis=1, keepdims=True) * sl2).astype(np.float32)
    p = np.exp2((s * sl2 - m).astype(np.float32)).astype(np.float32)
    l = p.sum(axis=1, dtype=np.float32)
    pb = att.bf16_rows_to_f64(to_bf16_bits(p).view(np.uint8).reshape(p.shape[0], -1))
    out = (pb @ kv[:, :512].astype(np.float64)) / l[:, None]
    lse = ((m[:, 0] + np.log2(l)) * np.float32(np.log(2))).astype(np.float32)
    return to_bf16_bits(out), lse


@pytest.mark.parametrize("k,scale,planted", [(300, 1 / 24, None), (300, 0.35, None), (129, 0.05, 64),
                                             (2048, 0.05, 2047)])
def test_the_kernel_roundings_stay_inside_the_bounds(k, scale, planted):
    q, keys, valid, scale = unit_inputs(k, planted=planted, scale=scale)
    out, lse = emulate_kernel(q, keys, valid, scale)
    check_unit(q, keys, valid, out, lse, scale, "emulated kernel")


def _wrong(q, keys, valid_used, scale):
    """A kernel that computed over the wrong keys, with exact arithmetic, then
    rounded its output to bf16."""
    want, lse = att.attend(att.bf16_rows_to_f64(q.view(np.uint8)), keys, valid_used, scale)
    return to_bf16_bits(want), lse.astype(np.float32)


def test_a_dropped_key_of_a_flat_softmax_fails():
    q, keys, valid, scale = unit_inputs(300, scale=1 / 24)
    used = valid.copy()
    used[123] = False
    out, lse = _wrong(q, keys, used, scale)
    with pytest.raises(AssertionError):
        check_unit(q, keys, valid, out, lse, scale, "dropped key")
    # lse alone would catch it too: one key of a flat softmax over 300 is ~1/300 of the sum
    from attention_check import bounds
    qf = att.bf16_rows_to_f64(q.view(np.uint8))
    assert np.abs(lse - att.attend(qf, keys, valid, scale)[1]).min() > 10 * bounds(qf, keys, valid, scale)[0].max()


@pytest.mark.parametrize("k", [65, 128, 2048])
def test_a_key_taken_across_the_block_boundary_fails(k):
    """Position 64's key replaced by position 63's (an off-by-one at the first
    block boundary), with the planted key at 64."""
    q, keys, valid, scale = unit_inputs(k, planted=64, scale=0.05)
    moved = keys.copy()
    moved[64] = keys[63]
    want_out, want_lse = _wrong(q, moved, valid, scale)
    with pytest.raises(AssertionError):
        check_unit(q, keys, valid, want_out, want_lse, scale, "moved key")


def test_a_masked_slot_read_as_a_zero_key_fails():
    """A -1 slot must drop out of the softmax; read as a zero row it would add
    exp(0) to the denominator."""
    q, keys, valid, scale = unit_inputs(300, scale=1 / 24)
    valid[77] = False
    zeroed = keys.copy()
    zeroed[77] = 0.0
    out, lse = _wrong(q, zeroed, np.ones(300, bool), scale)
    with pytest.raises(AssertionError, match="lse"):
        check_unit(q, keys, valid, out, lse, scale, "masked slot")
