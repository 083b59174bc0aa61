"""Run one workload through the CUDA library and the CPU oracle side by side.

The library owns the pinned host pool; the workload generator writes the
published rows into it directly (never through library code), and the
oracle reads the same memory as its pool view.  ``check_pool_rows`` verifies
that shared data against the generator before anything is compared.
Appended rows (write back) are written by the library into its pool and by
the oracle into its own store, and compared.

Every comparison is bit-exact: slot indices, counts, error bits, maps,
clocks, LRU order and hot-buffer bytes.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as orc
import skv_workload as wl
from sparse_attention_kv_skv_gb300 import Config, Context

RB = wl.ROW_BYTES


class Pair:
    def __init__(self, w: wl.Workload, req_perm=None, oracle_threads: int = 0, gen_threads: int | None = None,
                 entry: str = "assemble"):
        """entry: the Context method each step calls ("assemble" or "assemble_noalloc")."""
        self.w = w
        self.R = w.R
        self.T_max = w.max_context
        self.threads = oracle_threads or wl.default_threads()
        self.dev = torch.device("cuda", 0)
        self.stream = torch.cuda.current_stream()
        self.ctx = Context(Config(max_requests=self.R, num_layers=w.L, max_context=self.T_max, topk=w.k,
                                  hot_slots=w.S, max_batch=w.B, row_bytes=RB))
        self.pool = self.ctx.pool_rows()
        self.assemble_fn = getattr(self.ctx, entry)
        self.orc = orc.Oracle(self.R, w.L, self.T_max, RB, w.k, w.S, self.pool)
        self.gen = wl.TopkStream(w, nthreads=gen_threads)
        self.generation = {}
        # publish R requests on both sides; the batch uses B of them, in the
        # order given by req_perm (default: 0..B-1)
        for r in range(self.R):
            self._publish_fresh(expect=r)
        self.req_ids = list(range(w.B)) if req_perm is None else list(req_perm)
        assert len(self.req_ids) == w.B
        self.lens = [w.ctx] * w.B
        self.req_dev = torch.tensor(self.req_ids, dtype=torch.int32, device=self.dev)
        self.topk_dev = torch.empty((w.B, w.L, w.k), dtype=torch.int32, device=self.dev)
        self.slots_dev = torch.empty_like(self.topk_dev)
        self.hits_dev = torch.empty((w.B, w.L), dtype=torch.int32, device=self.dev)
        self.misses_dev = torch.empty_like(self.hits_dev)
        self.appended = {}
        self.total_misses = 0

    # ------------------------------------------------------------------ setup
    def req_base(self, r: int) -> int:
        return self.pool + r * self.w.L * self.T_max * RB

    def _publish_fresh(self, expect: int | None = None) -> int:
        w = self.w
        r = self.ctx.publish(w.ctx, rows=None)
        ro = self.orc.publish(w.ctx)
        assert r == ro, (r, ro)
        if expect is not None:
            assert r == expect
        torch.cuda.synchronize()
        gen = self.generation.get(r, -1) + 1
        self.generation[r] = gen
        wl.fill_request(self.req_base(r), w.L, self.T_max, w.ctx, w.base_seed, w.req_key(r, gen))
        return r

    def pool_view(self, r: int) -> np.ndarray:
        """The library's pool region of request r as a numpy array [L][T_max][RB]."""
        import ctypes
        n = self.w.L * self.T_max * RB
        buf = (ctypes.c_uint8 * n).from_address(self.req_base(r))
        return np.frombuffer(buf, dtype=np.uint8).reshape(self.w.L, self.T_max, RB)

    def check_pool_rows(self, samples: int = 64, seed: int = 0) -> None:
        """Published rows in the shared pool equal the generator's rows."""
        rng = np.random.default_rng(seed)
        w = self.w
        for r in range(self.R):
            pv = self.pool_view(r)
            key = w.req_key(r, self.generation[r])
            for _ in range(max(1, samples // self.R)):
                l = int(rng.integers(w.L))
                t = int(rng.integers(w.ctx))
                assert np.array_equal(pv[l, t], wl.fill_rows(w.base_seed, key, l, t, 1)[0]), (r, l, t)

    # ------------------------------------------------------------------ steps
    def capture(self) -> None:
        """From now on each step replays one captured CUDA graph of the step's
        entry point over the static input buffer (as the benchmark times it)."""
        self.graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(self.graph, stream=side):
                self.assemble_fn(self.req_dev, self.topk_dev, self.slots_dev, self.hits_dev, self.misses_dev)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()

    def extend_all(self, n: int, republish: bool = False) -> None:
        """A new turn for every session: n more tokens per request (skv_extend),
        or -- the cold alternative -- release and publish the grown request."""
        w = self.w
        for b, r in enumerate(self.req_ids):
            key = w.req_key(r, self.generation[r])
            if republish:
                self.ctx.release(r)
                assert self.orc.release(r) == 0
                new_len = self.lens[b] + n
                assert self.ctx.publish(new_len) == r and self.orc.publish(new_len) == r
                torch.cuda.synchronize()
                wl.fill_request(self.req_base(r), w.L, self.T_max, new_len, w.base_seed, key)
            else:
                rows = np.stack([wl.fill_rows(w.base_seed, key, l, self.lens[b], n) for l in range(w.L)])
                self.ctx.extend(r, torch.from_numpy(rows).to(self.dev), n)
                assert self.orc.extend(r, rows) == 0
            self.lens[b] += n

    def step(self, s: int, compare: bool = True, republish: bool = False):
        w = self.w
        if w.turn_every and s > 0 and s % w.turn_every == 0:
            self.extend_all(w.turn_tokens, republish=republish)
        topk = self.gen.step(s, self.lens)
        self.topk_dev.copy_(torch.from_numpy(topk))
        if getattr(self, "graph", None) is not None:
            self.graph.replay()
        else:
            self.assemble_fn(self.req_dev, self.topk_dev, self.slots_dev, self.hits_dev, self.misses_dev)
        e, slots, hits, misses = self.orc.assemble(self.req_ids, topk, nthreads=self.threads)
        assert e == 0
        self.total_misses += int(misses.sum())
        if compare:
            g_slots = self.slots_dev.cpu().numpy()
            g_hits = self.hits_dev.cpu().numpy()
            g_misses = self.misses_dev.cpu().numpy()
            if not np.array_equal(g_slots, slots):
                bad = np.argwhere(g_slots != slots)
                raise AssertionError(f"step {s}: {len(bad)} slot mismatches, first at {bad[0].tolist()}: "
                                     f"gpu {g_slots[tuple(bad[0])]} oracle {slots[tuple(bad[0])]}")
            assert np.array_equal(g_hits, hits), f"step {s}: hits differ"
            assert np.array_equal(g_misses, misses), f"step {s}: misses differ"
        if w.appends:
            self.write_back_all()
        return topk, slots, hits, misses

    def write_back_all(self):
        w = self.w
        rows = np.empty((w.B, w.L, RB), dtype=np.uint8)
        for b, r in enumerate(self.req_ids):
            key = w.req_key(r, self.generation[r])
            for l in range(w.L):
                rows[b, l] = wl.fill_rows(w.base_seed, key, l, self.lens[b], 1)[0]
        rows_dev = torch.from_numpy(rows).to(self.dev)
        self.ctx.write_back(self.req_dev, rows_dev)
        assert self.orc.write_back(self.req_ids, rows) == 0
        torch.cuda.synchronize()
        for b, r in enumerate(self.req_ids):
            pv = self.pool_view(r)
            for l in range(w.L):
                self.appended[(r, l, self.lens[b])] = rows[b, l]
                # the library stored the row at the request's old length
                assert np.array_equal(pv[l, self.lens[b]], rows[b, l]), (r, l, self.lens[b])
                assert np.array_equal(self.orc.pool_row(r, l, self.lens[b]), rows[b, l])
            self.lens[b] += 1

    def lifecycle(self, b: int) -> None:
        """Release batch entry b's request and publish a fresh one in its place."""
        r = self.req_ids[b]
        self.ctx.release(r)
        assert self.orc.release(r) == 0
        torch.cuda.synchronize()
        r2 = self._publish_fresh()
        assert r2 == r
        self.lens[b] = self.w.ctx
        self.gen.reset(b)
        for key in [k for k in self.appended if k[0] == r]:
            del self.appended[key]

    # ------------------------------------------------------------------ state
    def compare_state(self, reqs=None, hot: bool = True, tok2slot: bool = True) -> None:
        reqs = range(self.R) if reqs is None else reqs
        assert self.ctx.clock() == self.orc.now
        for r in reqs:
            g = self.ctx.export_state(r, tok2slot=tok2slot)
            o = self.orc.export(r, tok2slot=tok2slot)
            for key in ("slot2tok", "ts", "lru") + (("tok2slot",) if tok2slot else ()):
                if not np.array_equal(g[key], o[key]):
                    bad = np.argwhere(g[key] != o[key])
                    raise AssertionError(f"request {r}: {key} differs at {bad[0].tolist()} "
                                         f"(gpu {g[key][tuple(bad[0])]}, oracle {o[key][tuple(bad[0])]})")
            assert g["len"] == o["len"] and g["active"] == o["active"], r
            if hot:
                gh = self.ctx.export_hot(r)
                oh = self.orc.export_hot(r)
                if not np.array_equal(gh, oh):
                    bad = np.argwhere((gh != oh).any(axis=2))
                    raise AssertionError(f"request {r}: hot rows differ at (layer, slot) {bad[0].tolist()}")

    def compare_hot_rows(self, reqs) -> None:
        """For the given requests, every resident device row equals its
        token's row as the generator defines it, and every empty slot is
        zero."""
        w = self.w
        for r in reqs:
            st = self.orc.export(r, tok2slot=False)
            gh = self.ctx.export_hot(r)
            key = w.req_key(r, self.generation[r])
            for l in range(w.L):
                s2t = st["slot2tok"][l]
                occ = np.flatnonzero(s2t >= 0)
                assert not gh[l][s2t < 0].any(), (r, l)
                toks = s2t[occ]
                # published, extended and written-back rows all follow the
                # generator's formula for (request key, layer, token)
                want = np.empty((occ.size, RB), dtype=np.uint8)
                for j in range(occ.size):
                    want[j] = wl.fill_rows(w.base_seed, key, l, int(toks[j]), 1)[0]
                if not np.array_equal(gh[l][occ], want):
                    bad = np.flatnonzero((gh[l][occ] != want).any(axis=1))
                    raise AssertionError(f"request {r} layer {l}: slot {occ[bad[0]]} (token {toks[bad[0]]}) "
                                         f"holds the wrong row")

    def close(self):
        self.gen.close()
        self.orc.close()
        self.ctx.close()

