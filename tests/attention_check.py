"""The derived parity bounds of the tensor-core attention (skv_attend)
against its float64 definition, per unit and head; the derivation is in
tests/test_gpu_attention.py's docstring.  Shared by the GPU parity tests and
the CPU tests that plant mistakes to show the bounds catch them."""
import numpy as np

from oracle import attention as att

U_BF16 = 2.0 ** -8        # unit roundoff of bf16 (7 fraction bits, round to nearest even)
X24 = 2.0 ** -16          # a partial score sent as the upper 24 bits of its fp32
ACC = 19 * 2.0 ** -22     # fp32 accumulation: 18 MMA steps per half plus the sum of the halves
MISC = 1e-5               # ex2.approx, log2f, the 1/l scaling


def bounds(q, keys, valid, scale):
    """Per head: the derived bound on lse, and the absolute and relative bounds
    on out.  q [H][576], keys [k][576] float64, valid [k] bool."""
    kv = keys[valid]
    H = q.shape[0]
    if kv.shape[0] == 0:
        return np.zeros(H), np.zeros((H, 1)), np.zeros((H, 1))
    p0 = q[:, :288] @ kv[:, :288].T
    p1 = q[:, 288:] @ kv[:, 288:].T
    a = np.abs(q) @ np.abs(kv).T
    ds = (scale * (X24 * np.maximum(np.abs(p0), np.abs(p1)) + ACC * a)).max(axis=1)
    lse_tol = ds + MISC + (kv.shape[0] / 32 + 64) * 2.0 ** -24
    vmax = np.abs(kv[:, :att.V_DIM]).max()
    return lse_tol, ((U_BF16 + 2 * ds) * vmax)[:, None] + 1e-7, np.full((H, 1), U_BF16 + MISC)


def check_unit(q_bits, keys, valid, out_bits, lse, scale, what):
    """Element-wise check of one unit's out (bf16 bits [H][512]) and lse [H]
    against the definition on q (bf16 bits [H][576]) and the keys."""
    qf = att.bf16_rows_to_f64(q_bits.view(np.uint8))
    want, want_lse = att.attend(qf, keys, valid, scale)
    lse_tol, atol, rtol = bounds(qf, keys, valid, scale)
    got = att.bf16_rows_to_f64(out_bits.view(np.uint8))
    excess = np.abs(got - want) - (atol + rtol * np.abs(want))
    assert excess.max() <= 0, f"{what}: out off by {np.abs(got - want).max()} (worst excess {excess.max()})"
    both_inf = np.isneginf(want_lse) & np.isneginf(lse)
    with np.errstate(invalid="ignore"):
        diff = np.where(both_inf, 0.0, np.abs(lse - want_lse))
    assert np.all(diff <= lse_tol), f"{what}: lse off by {diff.max()} (bound {lse_tol[np.argmax(diff - lse_tol)]})"
