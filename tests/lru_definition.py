"""The replacement rule of the device buffer written out as its definition.

This is deliberately NOT the oracle's algorithm: there is no token map, no
linked list and no incremental update.  Each step recomputes, from the raw
per-slot record (token held, step of last use), which tokens are resident, which
Top-k entries miss, and which slots are the least recently used -- by sorting
every candidate slot on (last use, slot index).  It is used on tiny inputs only,
as the brute-force cross-check of the oracle.

Rule (pages: a Top-k LRU buffer on the GPU, "SGLang и Tair представили
иерархичную Sparse Attention ...", paragraph 1; only the sparse difference is
moved, same page, paragraph 3; readings where the pages are silent: ties to the
lowest slot index, misses in ascending token order, hits and fills get the
step's clock).
"""


class DefinitionLRU:
    def __init__(self, S: int):
        self.S = S
        self.token = [-1] * S   # token held by each slot, -1 = empty
        self.last = [0] * S     # clock of the step that last used the slot
        self.now = 0

    def resident(self):
        return {t: s for s, t in enumerate(self.token) if t != -1}

    def lru_order(self):
        return sorted(range(self.S), key=lambda s: (self.last[s], s))

    def step(self, row):
        """Apply one step; returns (out, hits, misses)."""
        self.now += 1
        where = self.resident()
        out = [-1] * len(row)
        used = set()
        for i, t in enumerate(row):
            if t != -1 and t in where:
                out[i] = where[t]
                used.add(where[t])
        hits = len(used)
        need = sorted((t, i) for i, t in enumerate(row) if t != -1 and t not in where)
        candidates = sorted((s for s in range(self.S) if s not in used), key=lambda s: (self.last[s], s))
        assert len(candidates) >= len(need)
        for (t, i), s in zip(need, candidates):
            self.token[s] = t
            out[i] = s
            used.add(s)
        for s in used:
            self.last[s] = self.now
        return out, hits, len(need)
