"""The host C/C++ code (the CPU oracle and the input generator) under
AddressSanitizer and UndefinedBehaviorSanitizer (CPU only).

Both libraries are rebuilt with -fsanitize=address,undefined into a scratch
directory and the oracle's pins run in a child process that preloads the ASan
runtime; any memory error or undefined behaviour aborts the child.
"""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle as orc
import skv_workload as wl

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SAN = ["-fsanitize=address,undefined", "-fno-sanitize-recover=undefined", "-fno-omit-frame-pointer", "-g", "-O1"]

CHILD = r"""
import sys
sys.path.insert(0, {tests!r})
import oracle_pins as pins
import skv_workload as wl
lib = {lib!r}
pins.check_golden(lib)
pins.check_closed_forms(lib)
pins.check_bruteforce(lib, T=5, k=2, S_values=(2, 3), steps=3, variant="sorted")
pins.check_bruteforce(lib, T=3, k=2, S_values=(2, 3), steps=3, variant="padded")
for w in [wl.Workload("san_uniform", B=2, L=2, ctx=300, k=32, S=48, steps=6, fresh=0.3),
          wl.Workload("san_shuffled", B=2, L=1, ctx=200, k=24, S=37, steps=6, fresh=0.25, order=wl.ORDER_SHUFFLED,
                      n_pad=5),
          wl.Workload("san_recency", B=2, L=1, ctx=400, k=32, S=64, steps=6, fresh=0.4, dist=wl.DIST_RECENCY, window=48),
          wl.Workload("san_zipf", B=2, L=1, ctx=512, k=32, S=64, steps=6, fresh=0.2, dist=wl.DIST_ZIPF, block=8),
          wl.Workload("san_append", B=2, L=2, ctx=100, k=20, S=32, steps=6, fresh=0.3, appends=True)]:
    pins.check_invariants(w, lib)
pins.check_errors(lib)
pins.check_layer_mode(lib)
pins.check_extend(lib)
pins.check_prefetch(lib)
print("sanitized pins ok")
"""


def _runtime(name):
    p = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_oracle_and_generator_under_asan_and_ubsan():
    asan = _runtime("libasan.so")
    if asan is None or _runtime("libubsan.so") is None:
        pytest.skip("the gcc sanitizer runtimes are not installed")
    with tempfile.TemporaryDirectory() as tmp:
        olib = os.path.join(tmp, "libskv_oracle_san.so")
        glib = os.path.join(tmp, "libskv_workload_san.so")
        subprocess.run(["g++", "-std=c++17", "-fPIC", "-shared", "-fopenmp", *SAN, "-o", olib, orc.SRC], check=True)
        subprocess.run(["gcc", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", *SAN, "-o", glib,
                        os.path.join(os.path.dirname(wl.__file__), "skv_workload.c"), "-lm"], check=True)
        env = dict(os.environ, LD_PRELOAD=asan, SKV_WORKLOAD_LIB=glib, OMP_NUM_THREADS="2",
                   ASAN_OPTIONS="detect_leaks=0:abort_on_error=1:allocator_may_return_null=0",
                   UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1",
                   PYTHONPATH=os.pathsep.join([ROOT, HERE, os.environ.get("PYTHONPATH", "")]))
        r = subprocess.run([sys.executable, "-c", CHILD.format(tests=HERE, lib=olib)], env=env, cwd=ROOT,
                           capture_output=True, text=True, timeout=900)
        assert r.returncode == 0 and "sanitized pins ok" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])
        # the instrumentation is live: a copy of the oracle whose gather writes one byte past the
        # destination row aborts the same run with a heap-buffer-overflow report
        src = open(orc.SRC).read()
        row_copy = "std::memcpy(u.hot.data() + (size_t)v * o->row_bytes, pool_row(o, q, u, r, l, t), o->row_bytes);"
        assert src.count(row_copy) == 1
        bad_src = os.path.join(tmp, "oracle_overflow.cpp")
        open(bad_src, "w").write(src.replace(row_copy, row_copy.replace("o->row_bytes);", "o->row_bytes + 1);")))
        bad_lib = os.path.join(tmp, "libskv_oracle_overflow.so")
        subprocess.run(["g++", "-std=c++17", "-fPIC", "-shared", "-fopenmp", *SAN, "-o", bad_lib, bad_src], check=True)
        r = subprocess.run([sys.executable, "-c", CHILD.format(tests=HERE, lib=bad_lib)], env=env, cwd=ROOT,
                           capture_output=True, text=True, timeout=900)
        assert r.returncode != 0 and "AddressSanitizer: heap-buffer-overflow" in r.stderr, r.stderr[-2000:]
