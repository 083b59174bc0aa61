"""Pins for the CPU oracle: checks against facts fixed outside the oracle.

Each ``check_*`` function loads an oracle shared library (the real one, or a
variant with a planted mistake) and raises AssertionError when the oracle
disagrees with:

* ``check_golden``      -- hand-derived worked examples (tests/golden);
* ``check_closed_forms`` -- Top-k sequences whose slots follow in closed form;
* ``check_bruteforce``  -- exhaustive enumeration of tiny Top-k sequences,
  compared with an independent definition of the rule (lru_definition.py);
* ``check_invariants``  -- per-step invariants on seeded random workloads
  (residency and row bytes, miss count as a set difference, occupancy, map
  inverses, clock stamps, LRU order, counts);
* ``check_errors``      -- all-or-nothing rejection of bad calls.
"""
from __future__ import annotations

import itertools
import os

import numpy as np

import oracle as orc
import skv_workload as wl
from lru_definition import DefinitionLRU

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")
RB = 32          # row bytes for the small checks (16 bf16 elements)
ROW_ELEMS = RB // 2


def _ints(s: str):
    return [int(x) for x in s.split(",")] if s else []


def make_pool(R, L, T_max, seed=7, T=None):
    """A pool view [R][L][T_max][RB] filled with generator rows (request key = r)."""
    pool = np.zeros((R, L, T_max, RB), dtype=np.uint8)
    T = T_max if T is None else T
    for r in range(R):
        for l in range(L):
            pool[r, l, :T] = wl.fill_rows(seed, r, l, 0, T, ROW_ELEMS)
    return pool


# ----------------------------------------------------------------------------
# golden walk-through
# ----------------------------------------------------------------------------

def check_golden(lib_path=None, name="lru_walkthrough.txt"):
    o = None
    pool = None
    seed = 7
    appended = {}   # (r, l, t) -> row given to write_back
    lines = open(os.path.join(GOLDEN, name)).read().splitlines()
    for ln, raw in enumerate(lines, 1):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        where = f"{name}:{ln}: {line}"
        lhs, _, rhs = (p.strip() for p in line.partition("->"))
        words = lhs.split()
        cmd = words[0]
        if cmd == "config":
            R, L, T_max, k, S = map(int, words[1:])
            pool = make_pool(R, L, T_max, seed)
            o = orc.Oracle(R, L, T_max, RB, k, S, pool, lib_path=lib_path)
        elif cmd == "publish":
            got = o.publish(int(words[1]))
            assert got == int(rhs), where
        elif cmd == "release":
            got = o.release(int(words[1]))
            assert got == int(rhs), where
        elif cmd == "get_error":
            assert o.get_error() == int(rhs), where
        elif cmd == "write_back":
            req = _ints(words[1].split("=")[1])
            rows = []
            for r in req:
                ln_r = o.export(r, tok2slot=False)["len"] if 0 <= r < o.R else 0
                for l in range(o.L):
                    row = wl.fill_rows(seed + 1, r, l, ln_r, 1, ROW_ELEMS)[0]
                    rows.append(row)
            e = o.write_back(req, np.stack(rows))
            assert e == int(rhs), where
            if e == 0:
                for i, r in enumerate(req):
                    for l in range(o.L):
                        appended[(r, l, o.export(r, tok2slot=False)["len"] - 1)] = rows[i * o.L + l]
        elif cmd == "assemble":
            req = _ints(words[1].split("=")[1])
            rows = [_ints(x) for x in words[2].split("=")[1].split(";")]
            topk = np.array(rows, dtype=np.int32).reshape(len(req), o.L, o.k)
            err, slots, hits, misses = o.assemble(req, topk)
            exp = rhs.split()
            assert err == int(exp[0]), where
            assert slots.reshape(-1).tolist() == _ints(exp[1].split("=")[1]), (where, slots)
            assert hits.reshape(-1).tolist() == _ints(exp[2].split("=")[1]), (where, hits)
            assert misses.reshape(-1).tolist() == _ints(exp[3].split("=")[1]), (where, misses)
            if err == 0:
                # every selected token's slot holds that token's row bytes
                hot = {r: o.export_hot(r) for r in set(req)}
                for b, r in enumerate(req):
                    for l in range(o.L):
                        for i, t in enumerate(topk[b, l]):
                            if t < 0:
                                continue
                            want = appended.get((r, l, int(t)))
                            if want is None:
                                want = pool[r, l, t]
                            assert np.array_equal(hot[r][l, slots[b, l, i]], want), where
        elif cmd == "state":
            r, l = int(words[1]), int(words[2])
            st = o.export(r, tok2slot=True)
            exp = dict(x.split("=") for x in rhs.split())
            assert st["slot2tok"][l].tolist() == _ints(exp["slot2tok"]), (where, st["slot2tok"][l])
            assert st["ts"][l].tolist() == _ints(exp["ts"]), (where, st["ts"][l])
            assert st["lru"][l].tolist() == _ints(exp["lru"]), (where, st["lru"][l])
            assert o.now == int(exp["now"]), where
        else:
            raise ValueError(where)


# ----------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------

def _single_unit(k, S, T, lib_path):
    pool = make_pool(1, 1, T, seed=11)
    o = orc.Oracle(1, 1, T, RB, k, S, pool, lib_path=lib_path)
    assert o.publish(T) == 0
    return o, pool


def check_closed_forms(lib_path=None):
    rng = np.random.default_rng(5)
    # (i) cold first step with a sorted row: out[i] = i, all k miss
    for k, S in [(8, 8), (16, 40), (33, 64)]:
        o, _ = _single_unit(k, S, 200, lib_path)
        row = np.sort(rng.choice(200, size=k, replace=False)).astype(np.int32)
        err, slots, hits, misses = o.assemble([0], row.reshape(1, 1, k))
        assert err == 0 and slots.reshape(-1).tolist() == list(range(k)), "cold step"
        assert hits[0, 0] == 0 and misses[0, 0] == k
        # cold step with the same set shuffled: slot = rank of the token
        o2, _ = _single_unit(k, S, 200, lib_path)
        perm = rng.permutation(k)
        err, slots, _, _ = o2.assemble([0], row[perm].reshape(1, 1, k))
        assert slots.reshape(-1).tolist() == perm.tolist(), "cold step, shuffled"
    # (ii) the same Top-k every step: no miss after the first step, slots fixed
    k, S = 16, 24
    o, _ = _single_unit(k, S, 100, lib_path)
    row = rng.choice(100, size=k, replace=False).astype(np.int32).reshape(1, 1, k)
    _, first, _, _ = o.assemble([0], row)
    for _ in range(5):
        err, slots, hits, misses = o.assemble([0], row)
        assert err == 0 and misses[0, 0] == 0 and hits[0, 0] == k
        assert np.array_equal(slots, first), "repeated Top-k"
    # (iii) pairwise-disjoint rows with S = q*k: the j-th smallest token of
    # step s goes to slot (s mod q)*k + j.  (iv) is q = 1.
    for q in (1, 2, 3):
        k = 8
        S = q * k
        steps = 3 * q + 2
        T = k * steps
        o, _ = _single_unit(k, S, T, lib_path)
        toks = rng.permutation(T).astype(np.int32)
        for s in range(steps):
            chunk = toks[s * k:(s + 1) * k]
            err, slots, hits, misses = o.assemble([0], chunk.reshape(1, 1, k))
            assert err == 0 and misses[0, 0] == k
            rank = np.argsort(np.argsort(chunk))
            assert slots.reshape(-1).tolist() == ((s % q) * k + rank).tolist(), f"disjoint rows q={q} step {s}"
    # (v) sliding window [s, s+k) with S = k: one token leaves and one enters
    # each step; the only non-hit slot is the departed token's, so token t
    # lives in slot t mod k.
    k = 8
    o, _ = _single_unit(k, k, 64, lib_path)
    for s in range(40):
        row = np.arange(s, s + k, dtype=np.int32)
        err, slots, hits, misses = o.assemble([0], row.reshape(1, 1, k))
        assert err == 0
        assert slots.reshape(-1).tolist() == (row % k).tolist(), f"sliding window step {s}"
        assert misses[0, 0] == (k if s == 0 else 1)


# ----------------------------------------------------------------------------
# brute force against the definition
# ----------------------------------------------------------------------------

def _rows(T, k, variant):
    toks = range(T)
    if variant == "sorted":
        return [list(c) for c in itertools.combinations(toks, k)]
    if variant == "ordered":
        return [list(p) for p in itertools.permutations(toks, k)]
    if variant == "padded":
        out = []
        for p in itertools.product([-1] + list(toks), repeat=k):
            v = [t for t in p if t != -1]
            if len(set(v)) == len(v):
                out.append(list(p))
        return out
    raise ValueError(variant)


def check_bruteforce(lib_path=None, T=5, k=2, S_values=(2, 3), steps=3, variant="sorted", limit=None):
    """Every sequence of `steps` rows (from `variant`) over T tokens, one
    request per sequence, all run as one batch."""
    rows = _rows(T, k, variant)
    seqs = list(itertools.product(range(len(rows)), repeat=steps))
    if limit is not None and len(seqs) > limit:
        idx = np.random.default_rng(1).choice(len(seqs), size=limit, replace=False)
        seqs = [seqs[i] for i in sorted(idx)]
    R = len(seqs)
    pool = make_pool(R, 1, T, seed=3)
    for S in S_values:
        o = orc.Oracle(R, 1, T, RB, k, S, pool, lib_path=lib_path)
        for r in range(R):
            assert o.publish(T) == r
        defs = [DefinitionLRU(S) for _ in range(R)]
        for s in range(steps):
            topk = np.array([rows[seq[s]] for seq in seqs], dtype=np.int32).reshape(R, 1, k)
            err, slots, hits, misses = o.assemble(list(range(R)), topk)
            assert err == 0
            for r in range(R):
                out, h, m = defs[r].step(topk[r, 0].tolist())
                assert slots[r, 0].tolist() == out, (S, seqs[r], s, slots[r, 0], out)
                assert (hits[r, 0], misses[r, 0]) == (h, m), (S, seqs[r], s)
        hot_all = None
        for r in range(R):
            st = o.export(r, tok2slot=True)
            d = defs[r]
            assert st["slot2tok"][0].tolist() == d.token, (S, seqs[r])
            assert st["ts"][0].tolist() == d.last, (S, seqs[r])
            assert st["lru"][0].tolist() == d.lru_order(), (S, seqs[r])
            t2s = [-1] * T
            for slot, t in enumerate(d.token):
                if t != -1:
                    t2s[t] = slot
            assert st["tok2slot"][0].tolist() == t2s, (S, seqs[r])
            hot_all = o.export_hot(r)
            for slot, t in enumerate(d.token):
                want = pool[r, 0, t] if t != -1 else np.zeros(RB, np.uint8)
                assert np.array_equal(hot_all[0, slot], want), (S, seqs[r], slot)
        o.close()


# ----------------------------------------------------------------------------
# invariants on seeded random workloads
# ----------------------------------------------------------------------------

def check_invariants(w: wl.Workload, lib_path=None, steps=None):
    """Run workload `w` (small sizes, RB-byte rows) through the oracle and check
    every invariant after every step; returns the rows the steps gathered."""
    R = w.R
    T_max = w.max_context
    seed = w.base_seed
    pool = np.zeros((R, w.L, T_max, RB), dtype=np.uint8)
    lens = [w.ctx] * w.B
    o = orc.Oracle(R, w.L, T_max, RB, w.k, w.S, pool, lib_path=lib_path)
    req_ids = []
    for b in range(w.B):
        r = o.publish(w.ctx)
        assert r == b
        for l in range(w.L):
            pool[r, l, :w.ctx] = wl.fill_rows(seed, w.req_key(b), l, 0, w.ctx, ROW_ELEMS)
        req_ids.append(r)
    gen = wl.TopkStream(w, nthreads=1)
    now = 0
    appended = {}
    gathered = 0
    nsteps = w.steps if steps is None else steps
    for s in range(nsteps):
        before = {r: o.export(r, tok2slot=False) for r in req_ids}
        topk = gen.step(s, lens)
        err, slots, hits, misses = o.assemble(req_ids, topk)
        assert err == 0
        gathered += int(misses.sum())
        now += 1
        assert o.now == now
        for b, r in enumerate(req_ids):
            st = o.export(r, tok2slot=True)
            hot = o.export_hot(r)
            for l in range(w.L):
                row = topk[b, l]
                valid = row[row >= 0]
                res_before = set(before[r]["slot2tok"][l][before[r]["slot2tok"][l] >= 0].tolist())
                # miss count = |Top-k \ resident before|, as a set difference
                assert misses[b, l] == len(set(valid.tolist()) - res_before)
                assert hits[b, l] + misses[b, l] == valid.size
                s2t = st["slot2tok"][l]
                t2s = st["tok2slot"][l]
                occupied = np.flatnonzero(s2t >= 0)
                assert occupied.size <= w.S
                # the two maps are inverse on the resident set
                assert np.array_equal(t2s[s2t[occupied]], occupied)
                assert (t2s >= 0).sum() == occupied.size
                # every Top-k token is resident, in the slot the step reported,
                # stamped with this step's clock
                sl = slots[b, l]
                assert np.array_equal(sl[row < 0], np.full((row < 0).sum(), -1))
                assert np.array_equal(s2t[sl[row >= 0]], valid)
                assert np.all(st["ts"][l][sl[row >= 0]] == now)
                # untouched slots keep their stamp
                untouched = np.setdiff1d(np.arange(w.S), sl[row >= 0])
                assert np.array_equal(st["ts"][l][untouched], before[r]["ts"][l][untouched])
                # LRU list = all slots sorted by (last use, slot)
                order = np.lexsort((np.arange(w.S), st["ts"][l]))
                assert np.array_equal(st["lru"][l], order)
                # residency bytes: a resident slot holds its token's pool row;
                # an empty slot holds zeros
                for slot in range(w.S):
                    t = int(s2t[slot])
                    if t < 0:
                        assert not hot[l, slot].any()
                        continue
                    want = appended.get((r, l, t))
                    if want is None:
                        want = pool[r, l, t]
                    assert np.array_equal(hot[l, slot], want), (s, b, l, slot, t)
                # evicted tokens left the map
                gone = res_before - set(s2t[occupied].tolist())
                assert all(t2s[t] == -1 for t in gone)
        if w.appends:
            rows = np.zeros((len(req_ids), w.L, RB), dtype=np.uint8)
            for b, r in enumerate(req_ids):
                for l in range(w.L):
                    rows[b, l] = wl.fill_rows(seed, w.req_key(b), l, lens[b], 1, ROW_ELEMS)[0]
            assert o.write_back(req_ids, rows) == 0
            for b, r in enumerate(req_ids):
                for l in range(w.L):
                    appended[(r, l, lens[b])] = rows[b, l]
                    assert np.array_equal(o.pool_row(r, l, lens[b]), rows[b, l])
                lens[b] += 1
    o.close()
    gen.close()
    return gathered


# ----------------------------------------------------------------------------
# errors: all-or-nothing
# ----------------------------------------------------------------------------

def check_errors(lib_path=None):
    R, L, T, k, S = 3, 2, 50, 4, 6
    pool = make_pool(R, L, T + 2, seed=9)
    o = orc.Oracle(R, L, T + 2, RB, k, S, pool, lib_path=lib_path)
    assert o.publish(T) == 0 and o.publish(T) == 1
    good = np.array([[[1, 2, 3, 4], [5, 6, 7, 8]], [[9, 10, 11, 12], [1, 3, 5, 7]]], dtype=np.int32)
    assert o.assemble([0, 1], good)[0] == 0

    def snapshot():
        return [(o.export(r)["slot2tok"].copy(), o.export(r)["ts"].copy(), o.export(r)["lru"].copy(),
                 o.export(r)["len"], o.export_hot(r).copy()) for r in range(R)] + [o.now]

    def same(a, b):
        for x, y in zip(a[:-1], b[:-1]):
            for p, q in zip(x, y):
                if not np.array_equal(np.asarray(p), np.asarray(q)):
                    return False
        return a[-1] == b[-1]

    cases = [
        ([0, 1], [[[1, 2, 3, 50], [5, 6, 7, 8]], [[9, 10, 11, 12], [1, 3, 5, 7]]], orc.E_BAD_INDEX),
        ([0, 1], [[[1, 2, 3, -2], [5, 6, 7, 8]], [[9, 10, 11, 12], [1, 3, 5, 7]]], orc.E_BAD_INDEX),
        ([0, 1], [[[1, 2, 3, 4], [5, 6, 7, 8]], [[9, 10, 11, 12], [1, 3, 5, 5]]], orc.E_DUPLICATE),
        ([0, 1], [[[1, 2, 3, 4], [5, 6, 7, 8]], [[9, 9, 11, 60], [1, 3, 5, 7]]], orc.E_DUPLICATE | orc.E_BAD_INDEX),
        ([0, 0], good.tolist(), orc.E_BAD_REQUEST),
        ([0, 2], good.tolist(), orc.E_BAD_REQUEST),        # 2 is not published
        ([0, 3], good.tolist(), orc.E_BAD_REQUEST),        # out of range
        ([-1, 1], good.tolist(), orc.E_BAD_REQUEST),
    ]
    for req, rows, bits in cases:
        before = snapshot()
        err, slots, hits, misses = o.assemble(req, np.array(rows, dtype=np.int32))
        assert err == bits, (req, rows, err, bits)
        assert (slots == -1).all() and (hits == -1).all() and (misses == -1).all()
        assert same(before, snapshot()), (req, rows)
        assert o.get_error() == bits
        assert o.get_error() == 0
    # the error word is sticky: until it is read, a valid call is a no-op that
    # reports it
    before = snapshot()
    assert o.assemble([0, 1], np.array(cases[0][1], dtype=np.int32))[0] == orc.E_BAD_INDEX
    err, slots, hits, misses = o.assemble([0, 1], good)
    assert err == orc.E_BAD_INDEX and (slots == -1).all() and (hits == -1).all()
    assert o.write_back([0], np.zeros((1, L, RB), dtype=np.uint8)) == orc.E_BAD_INDEX
    assert same(before, snapshot())
    assert o.get_error() == orc.E_BAD_INDEX and o.get_error() == 0
    # -1 padding is legal, repeated -1 is not a duplicate
    err, slots, hits, misses = o.assemble([0, 1], np.array([[[-1, 2, -1, 4], [5, -1, 7, 8]],
                                                            [[9, 10, -1, -1], [-1, -1, -1, -1]]], dtype=np.int32))
    assert err == 0 and misses[1, 1] == 0 and hits[1, 1] == 0
    # write_back: bad requests and a full context are rejected whole
    row = np.zeros((1, L, RB), dtype=np.uint8)
    rows2 = np.zeros((2, L, RB), dtype=np.uint8)
    assert o.write_back([2], row) == orc.E_BAD_REQUEST and o.get_error() == orc.E_BAD_REQUEST
    assert o.write_back([0, 0], rows2) == orc.E_BAD_REQUEST and o.get_error() == orc.E_BAD_REQUEST
    assert o.write_back([0], row) == 0 and o.write_back([0], row) == 0
    before = snapshot()
    assert o.write_back([1, 0], rows2) == orc.E_CONTEXT_FULL
    assert same(before, snapshot())
    assert o.get_error() == orc.E_CONTEXT_FULL
    # lifecycle
    assert o.release(2) == -1
    assert o.release(0) == 0 and o.release(0) == -1
    assert o.publish(T + 3) == -2
    assert o.publish(T) == 0 and o.publish(T) == 2 and o.publish(T) == -1
    st = o.export(0)
    assert (st["slot2tok"] == -1).all() and (st["ts"] == 0).all() and st["len"] == T
    assert not o.export_hot(0).any()
    o.close()


# ----------------------------------------------------------------------------
# one-layer steps against full steps
# ----------------------------------------------------------------------------

def check_layer_mode(lib_path=None, steps=6):
    """Assembling layers 0..L-1 one call each must leave every (request, layer)
    exactly as one call over all layers does -- same slots, counts, maps, LRU
    order and bytes -- except that the clock advances once per call, so a slot
    stamped c by the full call (c = step + 1) is stamped (c - 1) * L + l + 1 by
    the layer calls."""
    w = wl.Workload("layers", B=3, L=3, ctx=400, k=24, S=40, steps=steps, fresh=0.4, order=wl.ORDER_SHUFFLED,
                    n_pad=3)
    pool = make_pool(w.B, w.L, w.ctx, seed=21)
    full = orc.Oracle(w.B, w.L, w.ctx, RB, w.k, w.S, pool, lib_path=lib_path)
    per = orc.Oracle(w.B, w.L, w.ctx, RB, w.k, w.S, pool, lib_path=lib_path)
    for _ in range(w.B):
        full.publish(w.ctx)
        per.publish(w.ctx)
    req = [2, 0, 1]
    gen = wl.TopkStream(w, nthreads=1)
    for s in range(steps):
        topk = gen.step(s, [w.ctx] * w.B)
        e, slots, hits, misses = full.assemble(req, topk)
        assert e == 0
        for l in range(w.L):
            e, sl, h, m = per.assemble_layer(l, req, topk[:, l, :])
            assert e == 0
            assert np.array_equal(sl, slots[:, l, :]), (s, l)
            assert np.array_equal(h, hits[:, l]) and np.array_equal(m, misses[:, l]), (s, l)
    assert per.now == steps * w.L and full.now == steps
    for r in range(w.B):
        a, b = full.export(r), per.export(r)
        for key in ("slot2tok", "tok2slot", "lru"):
            assert np.array_equal(a[key], b[key]), (r, key)
        for l in range(w.L):
            ts_a = a["ts"][l].astype(np.int64)
            want = np.where(ts_a > 0, (ts_a - 1) * w.L + l + 1, 0)
            assert np.array_equal(b["ts"][l], want), (r, l)
        assert np.array_equal(full.export_hot(r), per.export_hot(r)), r
    # a bad layer is refused; an error in one layer's call changes nothing
    assert per.assemble_layer(w.L, req, topk[:, 0, :])[0] == -100
    before = [per.export(r) for r in range(w.B)]
    bad = topk[:, 1, :].copy()
    bad[1, 0] = w.ctx
    e, sl, h, m = per.assemble_layer(1, req, bad)
    assert e == orc.E_BAD_INDEX and (sl == -1).all() and (h == -1).all()
    assert per.get_error() == orc.E_BAD_INDEX
    for r in range(w.B):
        after = per.export(r)
        for key in ("slot2tok", "ts", "lru"):
            assert np.array_equal(before[r][key], after[key])
    full.close()
    per.close()
    gen.close()


# ----------------------------------------------------------------------------
# extend = n write backs
# ----------------------------------------------------------------------------

def check_extend(lib_path=None):
    """Extending a request by n rows leaves the pool and the request exactly as
    n single-row write backs do; a full region rejects the whole extension."""
    R, L, T, k, S = 2, 2, 10, 3, 4
    T_max = 16
    pool = make_pool(R, L, T_max, seed=31, T=T)
    a = orc.Oracle(R, L, T_max, RB, k, S, pool, lib_path=lib_path)
    b = orc.Oracle(R, L, T_max, RB, k, S, pool, lib_path=lib_path)
    for o in (a, b):
        assert o.publish(T) == 0 and o.publish(T) == 1
        assert o.assemble([0, 1], np.array([[[1, 2, 3], [4, 5, 6]], [[7, 8, 9], [0, 1, 2]]], np.int32))[0] == 0
    n = 4
    rows = np.stack([wl.fill_rows(77, 1, l, T, n, ROW_ELEMS) for l in range(L)])   # [L][n][RB]
    assert a.extend(1, rows) == 0
    for j in range(n):
        assert b.write_back([1], rows[:, j, :][None]) == 0
    for o in (a, b):
        assert o.export(1)["len"] == T + n and o.export(0)["len"] == T
    for l in range(L):
        for j in range(n):
            assert np.array_equal(a.pool_row(1, l, T + j), rows[l, j])
            assert np.array_equal(b.pool_row(1, l, T + j), rows[l, j])
    for r in range(R):
        ea, eb = a.export(r), b.export(r)
        for key in ("slot2tok", "ts", "lru", "tok2slot"):
            assert np.array_equal(ea[key], eb[key]), key
    # the new tokens are selectable, and miss on first use
    e, slots, hits, misses = a.assemble([1], np.array([[[T, T + 3, 1], [T + 1, 0, 2]]], np.int32))
    assert e == 0 and misses.tolist() == [[3, 1]]   # layer 0 holds {7, 8, 9}; layer 1 holds {0, 1, 2}
    # a region without room for all n rows is rejected whole
    big = np.zeros((L, T_max - (T + n) + 1, RB), np.uint8)
    assert a.extend(1, big) == orc.E_CONTEXT_FULL
    assert a.export(1)["len"] == T + n and a.get_error() == orc.E_CONTEXT_FULL
    assert a.extend(5, rows) == -1 and a.extend(1, rows[:, :0]) == 0
    a.close()
    b.close()


# ----------------------------------------------------------------------------
# prefetch (HiSparse's prefetching, kept by XM-Sparse: "XM-Sparse: Netpreme
# X-Mem ...", section on the SGLang HiSparse integration)
# ----------------------------------------------------------------------------

def check_prefetch(lib_path=None):
    """Hand-derived states after recency-window and explicit prefetches: the
    window's tokens take the least recently used slots like any miss, are
    stamped with the prefetch's own clock tick, and the next assemble that
    selects them hits; a bad candidate rejects the whole prefetch."""
    R, L, T, k, S, T_max = 3, 2, 12, 4, 6, 16
    pool = make_pool(R, L, T_max, seed=41, T=T)
    o = orc.Oracle(R, L, T_max, RB, k, S, pool, lib_path=lib_path)
    assert [o.publish(T), o.publish(T), o.publish(2)] == [0, 1, 2]

    def unit(r, l):
        st = o.export(r, tok2slot=False)
        return st["slot2tok"][l].tolist(), st["ts"][l].tolist()

    # the candidates themselves: the n newest tokens, all of [0, len) when len < n
    assert o.recent_candidates([0, 2], 3).tolist() == [[[9, 10, 11, -1]] * L, [[0, 1, -1, -1]] * L]
    assert o.recent_candidates([1], 4, layer=1).tolist() == [[8, 9, 10, 11]]
    assert o.recent_candidates([5, 2], 0).tolist() == [[[-1] * k] * L] * 2
    # 1. cold units: the j-th newest-window token takes slot j (every slot last used at 0)
    e, hits, misses = o.prefetch_recent([0, 1], 3)
    assert e == 0 and hits.tolist() == [[0, 0], [0, 0]] and misses.tolist() == [[3, 3], [3, 3]] and o.now == 1
    for r in (0, 1):
        for l in range(L):
            assert unit(r, l) == ([9, 10, 11, -1, -1, -1], [1, 1, 1, 0, 0, 0])
            for j, t in enumerate((9, 10, 11)):
                assert np.array_equal(o.export_hot(r)[l][j], pool[r, l, t])
    # 2. an assemble selecting two prefetched tokens hits them; its misses 2 < 5 take
    #    the never-used slots 3, 4 before the prefetched token 9's slot
    e, slots, hits, misses = o.assemble([0], np.array([[[10, 2, 11, 5]] * L], np.int32))
    assert e == 0 and hits.tolist() == [[2, 2]] and misses.tolist() == [[2, 2]] and o.now == 2
    assert slots.tolist() == [[[1, 3, 2, 4]] * L]
    for l in range(L):
        assert unit(0, l) == ([9, 10, 11, 2, 5, -1], [1, 2, 2, 2, 2, 0])
    # 3. one layer of request 1, window of 4: 9, 10, 11 hit (restamped), 8 takes slot 3;
    #    the other layer is untouched
    e, hits, misses = o.prefetch_recent([1], 4, layer=1)
    assert e == 0 and hits.tolist() == [3] and misses.tolist() == [1] and o.now == 3
    assert unit(1, 1) == ([9, 10, 11, 8, -1, -1], [3, 3, 3, 3, 0, 0])
    assert unit(1, 0) == ([9, 10, 11, -1, -1, -1], [1, 1, 1, 0, 0, 0])
    # 4. after a write back the window moves with the length: token 12 misses and takes
    #    the one slot never used (slot 5)
    new = np.stack([wl.fill_rows(43, 0, l, T, 1, ROW_ELEMS)[0] for l in range(L)])[None]
    assert o.write_back([0], new) == 0
    e, hits, misses = o.prefetch_recent([0], 1)
    assert e == 0 and misses.tolist() == [[1, 1]] and o.now == 4
    for l in range(L):
        assert unit(0, l) == ([9, 10, 11, 2, 5, 12], [1, 2, 2, 2, 2, 4])
        assert np.array_equal(o.export_hot(0)[l][5], new[0, l])
    # 5. explicit candidates: -1 padding, any order; a full window evicts by (last use, slot):
    #    misses 0, 1 (ascending) take slot 0 (token 9, used at 1) then slot 1 (10, used at 2)
    e, hits, misses = o.prefetch([0], np.array([[12, 1, -1, 0]], np.int32), layer=0)
    assert e == 0 and hits.tolist() == [1] and misses.tolist() == [2] and o.now == 5
    assert unit(0, 0) == ([0, 1, 11, 2, 5, 12], [5, 5, 2, 2, 2, 5])
    # 6. rejected whole: a token beyond len, an inactive request; nothing changes
    before = [o.export(r) for r in range(R)]
    e, _, _ = o.prefetch([0, 1], np.array([[[3, -1, -1, -1]] * L, [[12, -1, -1, -1]] * L], np.int32))
    assert e == orc.E_BAD_INDEX and o.now == 5
    assert o.get_error() == orc.E_BAD_INDEX and o.get_error() == 0  # read and cleared, as after any error
    assert o.release(2) == 0
    e, _, _ = o.prefetch_recent([2], 2)
    assert e == orc.E_BAD_REQUEST and o.now == 5
    assert o.get_error() == orc.E_BAD_REQUEST
    for r in range(R):
        after = o.export(r)
        for key in ("slot2tok", "ts", "lru", "tok2slot"):
            assert np.array_equal(before[r][key], after[key]) or r == 2, (r, key)
    o.close()
