"""Planted mistakes in the oracle must each be caught by its pins.

Each case copies the oracle source, applies one small edit that models a
plausible implementation mistake (a wrong tie-break, a missing sort, a dropped
map update, a wrong source row, ...), compiles the copy and runs the pins on it
(CPU only).  The test passes when at least one pin fails for every mutant, i.e.
no such mistake could hide behind the current pins.
"""
import concurrent.futures as cf
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest

import oracle as orc

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

MUTANTS = {
    "tie_break_highest_slot": [
        ("for (int32_t s = 0; s < o->S; ++s) u.lru.push_back(s);",
         "for (int32_t s = o->S - 1; s >= 0; --s) u.lru.push_back(s);")],
    "misses_in_row_order": [
        ("std::sort(missing.begin(), missing.end());", "/* no sort */")],
    "misses_descending": [
        ("std::sort(missing.begin(), missing.end());",
         "std::sort(missing.begin(), missing.end(), [](auto a, auto b) { return a > b; });")],
    "hits_evictable_and_not_refreshed": [
        ("u.lru.remove_if([&](int32_t s) { return hit_set.count(s) != 0; });", "/* hits stay */"),
        ("std::vector<int32_t> touched(hit_slots);", "std::vector<int32_t> touched;")],
    "hit_stamp_not_updated": [
        ("u.ts[s] = now;",
         "if (std::find(victims.begin(), victims.end(), s) != victims.end()) u.ts[s] = now;")],
    "evicted_token_kept_in_map": [
        ("if (old >= 0) u.tok2slot.erase(old);", "(void)old;")],
    "wrong_source_row": [
        ("pool_row(o, q, u, r, l, t), o->row_bytes);", "pool_row(o, q, u, r, l, t > 0 ? t - 1 : t), o->row_bytes);")],
    "clock_advances_on_reject": [
        ("        o->err |= e;\n        reject();\n        return e;",
         "        o->err |= e;\n        o->now += 1;\n        reject();\n        return e;")],
    "duplicates_not_checked": [
        ("else if (!row_tokens.insert(t).second) e |= E_DUPLICATE;", "else row_tokens.insert(t);")],
    "touched_not_in_slot_order": [
        ("std::sort(touched.begin(), touched.end());", "/* no sort */")],
    "victims_from_back": [
        ("victims.push_back(u.lru.front());\n        u.lru.pop_front();",
         "victims.push_back(u.lru.back());\n        u.lru.pop_back();")],
    "write_back_no_len_increment": [
        ("        q.len += 1;\n", "")],
    "layer_index_ignored": [
        ("const int32_t l = layer < 0 ? (int32_t)(x % nl) : layer;",
         "const int32_t l = layer < 0 ? (int32_t)(x % nl) : 0;")],
    "layer_call_not_validated": [
        ("for (int64_t j = 0; j < nl; ++j) {\n            std::unordered_set<int32_t> row_tokens;",
         "for (int64_t j = 0; j < (layer < 0 ? nl : 0); ++j) {\n            std::unordered_set<int32_t> row_tokens;")],
    "extend_off_by_one": [
        ("q.units[l].appended[q.len + j] =", "q.units[l].appended[q.len + j + 1] =")],
    "sticky_error_ignored": [
        ("    if (o->err) {\n        reject();\n        return o->err;\n    }", "")],
}


def _build(name, edits, tmp):
    src = open(orc.SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    p = os.path.join(tmp, f"{name}.cpp")
    open(p, "w").write(src)
    return orc.compile_oracle(p, os.path.join(tmp, f"lib{name}.so"))


_CHECKS = """
import sys
import oracle_pins as pins, skv_workload as wl
lib = sys.argv[1]
checks = [
    lambda: pins.check_golden(lib),
    lambda: pins.check_closed_forms(lib),
    lambda: pins.check_errors(lib),
    lambda: pins.check_bruteforce(lib, T=4, k=2, S_values=(2, 3), steps=3, variant="ordered"),
    lambda: pins.check_invariants(wl.Workload("mut_inv", B=2, L=1, ctx=100, k=12, S=20, steps=6, fresh=0.4,
                                              order=wl.ORDER_SHUFFLED), lib),
    lambda: pins.check_layer_mode(lib, steps=3),
    lambda: pins.check_extend(lib),
]
for c in checks:
    try:
        c()
    except (AssertionError, IndexError, KeyError, ValueError):
        sys.exit(1)
sys.exit(0)
"""


def _caught(lib_path):
    """Run every pin on the library in a child process; a failed pin or a crash
    (a mistake can make the oracle throw or read out of bounds) counts as caught."""
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([ROOT, HERE, os.environ.get("PYTHONPATH", "")]))
    p = subprocess.run([sys.executable, "-c", _CHECKS, lib_path], env=env, capture_output=True, timeout=600)
    return p.returncode != 0


def test_every_planted_mistake_is_caught():
    with tempfile.TemporaryDirectory() as tmp:
        with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 2) as ex:
            libs = dict(zip(MUTANTS, ex.map(lambda kv: _build(kv[0], kv[1], tmp), MUTANTS.items())))
        with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 2) as ex:
            caught = dict(zip(libs, ex.map(_caught, libs.values())))
        missed = [name for name, c in caught.items() if not c]
    assert not missed, f"pins did not catch: {missed}"


def test_unmodified_oracle_passes_the_same_checks():
    assert not _caught(orc.build())


PREFETCH_MUTANTS = {
    # the window one token short at its newest end
    "window_misses_newest": lambda self, req, n, layer=-1: _shift_window(self, req, n, layer, end=-1),
    # the window one token too long at its oldest end
    "window_one_older": lambda self, req, n, layer=-1: _shift_window(self, req, n + 1, layer, end=0),
    # the whole context instead of the newest n tokens
    "window_from_start": lambda self, req, n, layer=-1: _shift_window(self, req, n, layer, end=0, from_start=True),
}


def _shift_window(o, req_ids, n, layer, end, from_start=False):
    rows = o.L if layer < 0 else 1
    out = np.full((len(req_ids), rows, o.k), -1, dtype=np.int32)
    for b, r in enumerate(req_ids):
        st = o.export(int(r), tok2slot=False)
        hi = st["len"] + end
        lo = 0 if from_start else max(0, hi - n)
        toks = np.arange(lo, hi, dtype=np.int32)[: o.k]
        out[b, :, :toks.size] = toks
    return out if layer < 0 else out[:, 0, :]


@pytest.mark.parametrize("name", sorted(PREFETCH_MUTANTS))
def test_every_planted_prefetch_window_mistake_is_caught(name, monkeypatch):
    """A wrong recency window in the oracle's prefetch fails the hand-derived prefetch pins."""
    sys.path.insert(0, HERE)
    import oracle_pins as pins
    monkeypatch.setattr(orc.Oracle, "recent_candidates", PREFETCH_MUTANTS[name])
    with pytest.raises(AssertionError):
        pins.check_prefetch()
