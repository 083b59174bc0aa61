"""The seeded input generators: shapes, distinctness, determinism, mix."""
import numpy as np
import pytest

import skv_workload as wl


def test_splitmix64_published_values():
    # SplitMix64 started at state 0 (Vigna's reference splitmix64.c): the first
    # outputs are the published test values.
    assert wl.splitmix64_at(0, 0) == 0xE220A8397B1DCDAF
    assert wl.splitmix64_at(0, 1) == 0x6E789E6AA1B965F4
    assert wl.splitmix64_at(0, 2) == 0x06C45D188009454F


def test_rows_are_bf16_in_range_and_deterministic():
    a = wl.fill_rows(1, 2, 3, 100, 50)
    b = wl.fill_rows(1, 2, 3, 100, 50)
    assert a.shape == (50, wl.ROW_BYTES) and np.array_equal(a, b)
    # a row depends on (seed, request, layer, token)
    assert not np.array_equal(a[0], wl.fill_rows(1, 2, 3, 101, 1)[0])
    assert not np.array_equal(a[0], wl.fill_rows(1, 2, 4, 100, 1)[0])
    assert not np.array_equal(a[0], wl.fill_rows(1, 3, 3, 100, 1)[0])
    assert not np.array_equal(a[0], wl.fill_rows(2, 2, 3, 100, 1)[0])
    bits = a.view(np.uint16).astype(np.uint32) << 16
    x = bits.view(np.float32)
    # uniform in [-1, 1) before rounding; values just below 1 round up to 1.0
    assert np.all(x >= -1.0) and np.all(x <= 1.0)
    assert abs(float(x.mean())) < 0.02 and 0.55 < float(x.std()) < 0.60   # uniform[-1,1): std 1/sqrt(3)
    # bf16 rounding: value equals the float32 rounded to 8 mantissa bits
    assert np.all((bits & 0xFFFF) == 0)


def test_fill_request_layout_matches_rows():
    L, T_max, T = 3, 40, 33
    buf = np.zeros((L, T_max, wl.ROW_BYTES), dtype=np.uint8)
    wl.fill_request(buf.ctypes.data, L, T_max, T, seed=5, req_key=9, nthreads=3)
    for l in range(L):
        assert np.array_equal(buf[l, :T], wl.fill_rows(5, 9, l, 0, T))
        assert not buf[l, T:].any()


@pytest.mark.parametrize("name", ["c1_tiny"])
def test_topk_keep_and_fresh_fractions(name):
    w = wl.WORKLOADS[name]
    g = wl.TopkStream(w)
    lens = [w.ctx] * w.B
    prev = g.step(0, lens)
    for s in range(1, 8):
        cur = g.step(s, lens)
        for b in range(w.B):
            for l in range(w.L):
                row = cur[b, l]
                assert np.all(np.diff(row) > 0)                  # sorted, distinct
                assert row.min() >= 0 and row.max() < w.ctx
                kept = len(set(row.tolist()) & set(prev[b, l].tolist()))
                # 80% kept; a fresh pick may land on a token dropped this step
                assert w.k - w.n_fresh <= kept <= w.k - w.n_fresh + 8
        prev = cur
    assert w.n_fresh == 51


def test_topk_deterministic_and_thread_independent():
    w = wl.Workload("det", B=5, L=3, ctx=3000, k=64, S=128, steps=4, fresh=0.4, dist=wl.DIST_RECENCY, window=100)
    a, b = wl.TopkStream(w, nthreads=1), wl.TopkStream(w, nthreads=4)
    for s in range(4):
        assert np.array_equal(a.step(s, [w.ctx] * w.B), b.step(s, [w.ctx] * w.B))


def test_topk_padding_and_shuffle():
    w = wl.Workload("pad", B=2, L=2, ctx=500, k=40, S=64, steps=3, fresh=0.25, n_pad=7, order=wl.ORDER_SHUFFLED)
    g = wl.TopkStream(w)
    x = g.step(0, [w.ctx] * w.B)
    for row in x.reshape(-1, w.k):
        assert (row == -1).sum() == 7
        v = row[row >= 0]
        assert len(set(v.tolist())) == v.size == 33
    w2 = wl.Workload("pad2", B=1, L=1, ctx=500, k=40, S=64, steps=3, fresh=0.25, n_pad=7)
    row = wl.TopkStream(w2).step(0, [500])[0, 0]
    v = row[row >= 0]
    assert (row == -1).sum() == 7 and np.all(np.diff(v) > 0)


def test_recency_and_zipf_shapes():
    w = wl.Workload("rec", B=8, L=2, ctx=16384, k=512, S=1024, steps=6, fresh=0.4, dist=wl.DIST_RECENCY,
                    window=2048)
    g = wl.TopkStream(w)
    prev = g.step(0, [w.ctx] * w.B)
    frac = []
    for s in range(1, 6):
        cur = g.step(s, [w.ctx] * w.B)
        for b in range(w.B):
            for l in range(w.L):
                fresh = np.setdiff1d(cur[b, l], prev[b, l])
                frac.append(np.mean(fresh >= w.ctx - 2048))
        prev = cur
    assert 0.4 < np.mean(frac) < 0.8          # biased to the last 2048 positions
    z = wl.Workload("zipf", B=4, L=1, ctx=131072, k=2048, S=4096, steps=3, fresh=0.2, dist=wl.DIST_ZIPF)
    g = wl.TopkStream(z)
    a = g.step(0, [z.ctx] * z.B)
    b2 = g.step(1, [z.ctx] * z.B)
    # heavy head: the selected set covers far fewer 64-token blocks than a
    # uniform set of 2048 tokens would (about 2048 * (1 - 1/e) ~ 1295 blocks)
    for x in (a, b2):
        assert np.unique(x[0, 0] // 64).size < 1000


def test_appending_lengths_are_respected():
    w = wl.Workload("app", B=2, L=1, ctx=100, k=20, S=32, steps=5, fresh=0.5, appends=True)
    g = wl.TopkStream(w)
    for s in range(5):
        x = g.step(s, [w.ctx + s] * w.B)
        assert x.max() < w.ctx + s
