"""Sparse MLA decode attention written out as its definition -- TEST
INFRASTRUCTURE ONLY (only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline use it; the product never does).

DSA's "select, then compute" ("SGLang и Tair представили иерархичную Sparse
Attention ...", paragraph 2): attention of each head over the selected tokens
only.  For one (request, layer) unit, with q [H][576] (a 512-wide latent plus
64 rope dims) and the selected key rows K [k][576], of which `valid` are real
(padding is masked):

    s_hj = scale * sum_d q_hd K_jd            (valid j only)
    out_h = sum_j softmax_j(s_h)_j * K_j[0:512]     (V = the latent part)
    lse_h = log sum_j exp(s_hj)

in float64, with numpy's matmul as a step.  All masked: out = 0, lse = -inf.

Parity status: pinned in tests/test_oracle_attention.py by closed forms
(uniform scores, one key, two keys, a repeated key), invariants (masking, key
order) and a scalar-loop evaluation of the definition on tiny inputs.
"""
from __future__ import annotations

import numpy as np

V_DIM = 512


def bf16_rows_to_f64(rows_u8: np.ndarray) -> np.ndarray:
    """bf16 rows stored as bytes [..., 2*n] -> float64 [..., n] (exact)."""
    u16 = np.ascontiguousarray(rows_u8).view(np.uint16).astype(np.uint32) << 16
    return u16.view(np.float32).astype(np.float64)


def attend(q: np.ndarray, keys: np.ndarray, valid: np.ndarray, scale: float):
    """(out [H][512], lse [H]) for one unit; q [H][576], keys [k][576] floats."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(keys, dtype=np.float64)[np.asarray(valid, dtype=bool)]
    H = q.shape[0]
    if k.shape[0] == 0:
        return np.zeros((H, V_DIM)), np.full(H, -np.inf)
    s = scale * (q @ k.T)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    denom = e.sum(axis=1, keepdims=True)
    out = (e / denom) @ k[:, :V_DIM]
    lse = (m + np.log(denom))[:, 0]
    return out, lse
