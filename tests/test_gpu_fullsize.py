"""Full-size parity: every evaluation workload at its full shape, stepped
through captured CUDA graphs as the benchmark runs it, against the CPU oracle
run over the same pinned pool (GPU; tens of GB of host memory).

Every step's slot tensor and hit / miss counts are compared in full; at the
end the maps, clocks, LRU order and hot rows of a spread of requests are
compared in full, and every resident row of those requests is checked against
the generator.
"""
import pytest
import torch

import skv_workload as wl

pytestmark = [pytest.mark.gpu, pytest.mark.fullsize]

if torch.cuda.is_available():
    from skv_pair import Pair

# (workload, requests whose full state is compared at the end); every
# workload runs all of its steps (128 or 64), including c5's release and
# re-publish of a request at step 32
CASES = [
    ("target_16k_b192_f20", [0, 1, 63, 127, 190, 191]),
    ("c2_16k_b64_append", [0, 17, 63]),
    ("c3_16k_b192_f40_recency", [0, 95, 191]),
    ("c4_128k_b32_zipf", [0, 13, 31]),
    ("c5_1m_b4_lifecycle", [0, 1, 2, 3]),
]


@pytest.mark.parametrize("name,reqs", CASES, ids=[c[0] for c in CASES])
def test_full_size_workload(name, reqs):
    w = wl.WORKLOADS[name]
    steps = w.steps
    p = Pair(w)
    try:
        p.check_pool_rows(samples=256)
        p.step(0)                       # cold step (eager)
        p.capture()
        for s in range(1, steps):
            if s == w.lifecycle_step:
                p.lifecycle(1)          # release + publish a fresh request in its place
            p.step(s)
        p.compare_state(reqs=reqs)
        p.compare_hot_rows(reqs)
        assert p.ctx.get_device_error() == 0
        st = p.ctx.stats()
        assert st["calls"] == steps and st["misses"] == p.total_misses
    finally:
        p.close()
