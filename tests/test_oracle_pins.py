"""The CPU oracle against facts fixed outside it (see oracle_pins.py)."""
import pytest

import skv_workload as wl
import oracle_pins as pins


def test_golden_walkthrough():
    pins.check_golden()


def test_closed_forms():
    pins.check_closed_forms()


@pytest.mark.parametrize("T,k,S_values,steps,variant", [
    (5, 2, (2, 3, 4), 3, "sorted"),
    (4, 2, (2, 3), 3, "ordered"),
    (3, 2, (2, 3), 3, "padded"),
    (6, 3, (3, 4, 5), 3, "sorted"),
    (4, 1, (1, 2, 3), 5, "sorted"),
])
def test_bruteforce_against_definition(T, k, S_values, steps, variant):
    pins.check_bruteforce(T=T, k=k, S_values=S_values, steps=steps, variant=variant)


SMALL = [
    wl.Workload("inv_uniform", B=3, L=2, ctx=300, k=32, S=48, steps=12, fresh=0.3),
    wl.Workload("inv_tight", B=2, L=1, ctx=120, k=40, S=40, steps=12, fresh=0.5),
    wl.Workload("inv_shuffled_pad", B=2, L=2, ctx=200, k=24, S=37, steps=12, fresh=0.25,
                order=wl.ORDER_SHUFFLED, n_pad=5),
    wl.Workload("inv_sorted_pad", B=2, L=1, ctx=200, k=24, S=30, steps=10, fresh=0.25, n_pad=3),
    wl.Workload("inv_recency", B=2, L=2, ctx=400, k=32, S=64, steps=10, fresh=0.4, dist=wl.DIST_RECENCY,
                window=48),
    wl.Workload("inv_zipf", B=2, L=1, ctx=512, k=32, S=64, steps=10, fresh=0.2, dist=wl.DIST_ZIPF, block=8),
    wl.Workload("inv_append", B=3, L=2, ctx=100, k=20, S=32, steps=10, fresh=0.3, appends=True),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_invariants(w):
    pins.check_invariants(w)


def test_errors_and_lifecycle():
    pins.check_errors()


def test_layer_calls_match_full_steps():
    pins.check_layer_mode()


def test_extend_equals_repeated_write_back():
    pins.check_extend()


def test_prefetch_hand_derived():
    pins.check_prefetch()
