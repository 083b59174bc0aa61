"""The attention oracle against closed forms (CPU)."""
import numpy as np

from oracle import attention as att


def _keys(rng, k, d=576):
    return rng.uniform(-1, 1, size=(k, d))


def test_uniform_scores_give_the_mean_of_valid_values():
    rng = np.random.default_rng(0)
    K = _keys(rng, 40)
    valid = rng.random(40) < 0.6
    out, lse = att.attend(np.zeros((3, 576)), K, valid, 0.7)
    assert np.allclose(out, K[valid][:, :512].mean(axis=0), atol=1e-12)
    assert np.allclose(lse, np.log(valid.sum()))


def test_one_valid_key_returns_its_value_part():
    rng = np.random.default_rng(1)
    K = _keys(rng, 9)
    q = rng.uniform(-1, 1, size=(4, 576))
    valid = np.zeros(9, bool)
    valid[5] = True
    out, lse = att.attend(q, K, valid, 0.3)
    assert np.allclose(out, K[5, :512])
    assert np.allclose(lse, 0.3 * q @ K[5])


def test_two_keys_closed_form():
    rng = np.random.default_rng(2)
    K = _keys(rng, 2)
    q = rng.uniform(-1, 1, size=(5, 576))
    scale = 0.05
    s1, s2 = scale * q @ K[0], scale * q @ K[1]
    w1 = 1.0 / (1.0 + np.exp(s2 - s1))
    out, lse = att.attend(q, K, np.ones(2, bool), scale)
    assert np.allclose(out, w1[:, None] * K[0, :512] + (1 - w1)[:, None] * K[1, :512])
    assert np.allclose(lse, np.logaddexp(s1, s2))


def test_masked_keys_and_key_order_do_not_matter():
    rng = np.random.default_rng(3)
    K = _keys(rng, 64)
    q = rng.uniform(-1, 1, size=(6, 576))
    valid = rng.random(64) < 0.5
    out, lse = att.attend(q, K, valid, 0.2)
    junk = K.copy()
    junk[~valid] = 1e3                                   # masked rows may hold anything
    perm = rng.permutation(64)
    out2, lse2 = att.attend(q, junk[perm], valid[perm], 0.2)
    assert np.allclose(out, out2) and np.allclose(lse, lse2)


def test_all_masked_gives_zeros_and_minus_infinity():
    out, lse = att.attend(np.ones((2, 576)), np.ones((3, 576)), np.zeros(3, bool), 1.0)
    assert not out.any() and np.all(np.isneginf(lse))


def test_bf16_decoding_is_exact():
    vals = np.array([1.0, -0.5, 0.15625, -2.0 ** -10], dtype=np.float32)
    u16 = (vals.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(att.bf16_rows_to_f64(u16.view(np.uint8)), vals.astype(np.float64))


def test_against_a_literal_loop_on_tiny_inputs():
    """The definition written out with scalar loops (no matrix product, no max shift)."""
    import math
    rng = np.random.default_rng(4)
    H, k, d = 3, 5, 576
    q = rng.uniform(-1, 1, size=(H, d))
    K = _keys(rng, k, d)
    valid = np.array([True, False, True, True, False])
    scale = 0.09
    out, lse = att.attend(q, K, valid, scale)
    for h in range(H):
        w = {}
        for j in range(k):
            if valid[j]:
                w[j] = math.exp(scale * sum(q[h, t] * K[j, t] for t in range(d)))
        z = sum(w.values())
        for c in range(512):
            assert abs(out[h, c] - sum(w[j] * K[j, c] for j in w) / z) < 1e-12
        assert abs(lse[h] - math.log(z)) < 1e-12


def test_a_repeated_key_weighs_twice():
    """Two copies of one key give the same output as one copy and lse + log 2."""
    rng = np.random.default_rng(5)
    K = _keys(rng, 7)
    q = rng.uniform(-1, 1, size=(4, 576))
    K2 = np.concatenate([K, K[3:4]])
    w_out, w_lse = att.attend(q, K2, np.ones(8, bool), 0.15)
    # with key 3 twice, its weight doubles
    s = 0.15 * q @ K.T
    wts = np.exp(s)
    wts[:, 3] *= 2
    want = (wts / wts.sum(axis=1, keepdims=True)) @ K[:, :512]
    assert np.allclose(w_out, want) and np.allclose(w_lse, np.log(wts.sum(axis=1)))
    only = np.zeros(7, bool)
    only[3] = True
    o1, l1 = att.attend(q, K, only, 0.15)
    o2, l2 = att.attend(q, np.stack([K[3], K[3]]), np.ones(2, bool), 0.15)
    assert np.allclose(o1, o2) and np.allclose(l2, l1 + np.log(2))
