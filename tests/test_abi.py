"""The C ABI library loads and exports every entry point of include/skv.h;
host-side checks that need no GPU (CPU only)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "skv.h")


@pytest.fixture(scope="module")
def lib_path():
    from sparse_attention_kv_skv_gb300 import build
    return build.build()


def declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^SKV_API\s+[\w\s\*]+?\b(skv_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_lifecycle():
    names = declared()
    for n in LIFECYCLE:
        assert n in names


LIFECYCLE = ("skv_create", "skv_destroy", "skv_publish", "skv_write_back", "skv_assemble", "skv_release",
             "skv_get_device_error", "skv_hot_buffer", "skv_export_state")


def doc_comment(name: str) -> str:
    """The comment block right above the declaration of `name`."""
    src = open(HEADER).read()
    m = re.search(r"/\*((?:(?!\*/).)*)\*/\s*SKV_API\s+[\w\s\*]+?\b" + name + r"\s*\(", src, flags=re.S)
    assert m, name
    return m.group(1)


def test_every_lifecycle_declaration_cites_its_source():
    """Each boundary call of the hot path states where it comes from: a page
    section (by the header's tags) or, where the pages are silent, the
    reading the library implements."""
    for n in LIFECYCLE:
        doc = doc_comment(n)
        assert "Source:" in doc, n
        cite = doc.split("Source:", 1)[1]
        assert re.search(r"\[(talk|digest|xm)\]", cite) or "pages are silent" in cite, n
    head = open(HEADER).read().split("#ifndef SKV_H_")[0]
    for tag in ("[talk]", "[digest]", "[xm]"):
        assert tag in head  # every tag is defined in the opening comment


def test_every_declared_symbol_is_exported(lib_path):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert set(declared()) <= exported
    # nothing but the ABI is exported (the static CUDA runtime stays private)
    assert all(s.startswith("skv_") for s in exported), sorted(s for s in exported if not s.startswith("skv_"))


def test_library_loads_and_binding_has_every_entry_point(lib_path):
    lib = ctypes.CDLL(lib_path)
    for n in declared():
        assert hasattr(lib, n)
    from sparse_attention_kv_skv_gb300 import skv
    for n in declared():
        assert hasattr(skv, n), n


def test_config_struct_layout_matches_header():
    from sparse_attention_kv_skv_gb300 import skv
    assert ctypes.sizeof(skv.skv_config) == 40
    assert skv.skv_config.max_context.offset == 8
    assert skv.skv_config.device.offset == 32


def test_host_argument_checks_need_no_gpu(lib_path):
    from sparse_attention_kv_skv_gb300 import skv
    h = ctypes.c_void_p()
    assert skv.skv_create(None, ctypes.byref(h)) == skv.SKV_ERR_INVALID_ARG
    bad = [
        skv.skv_config(0, 1, 10, 1152, 4, 8, 1, 0),       # no requests
        skv.skv_config(1, 1, 10, 1000, 4, 8, 1, 0),       # row bytes not a multiple of 16
        skv.skv_config(1, 1, 10, 1152, 8, 4, 1, 0),       # S < k
        skv.skv_config(1, 1, 10, 1152, 5000, 8000, 1, 0),  # k above the limit
        skv.skv_config(1, 1, 10, 1152, 4, 20000, 1, 0),   # S above the limit
        skv.skv_config(1 << 16, 64, 1 << 20, 1152, 4, 8, 1, 0),  # R*L*T_max >= 2^32
        skv.skv_config(1, 1, 10, 1152, 4, 8, 0, 0),       # max_batch 0
        skv.skv_config(1, 1, 10, 65552, 4, 8, 1, 0),      # rows above 64 KiB
    ]
    for c in bad:
        assert skv.skv_create(ctypes.byref(c), ctypes.byref(h)) == skv.SKV_ERR_INVALID_ARG
    assert skv.skv_destroy(None) == skv.SKV_OK
    assert skv.skv_assemble(None, None, 0, None, None, None, None, None) == skv.SKV_ERR_INVALID_ARG
    assert skv.skv_prefetch(None, None, 1, -1, None, None, None, None) == skv.SKV_ERR_INVALID_ARG
    assert skv.skv_prefetch_recent(None, None, 1, -1, 4, None, None, None) == skv.SKV_ERR_INVALID_ARG
    assert skv.skv_attend(None, None, 1, -1, None, None, None, None, 0.1, None) == skv.SKV_ERR_INVALID_ARG
    assert skv.skv_set_attend_sms(None, 0) == skv.SKV_ERR_INVALID_ARG
    assert skv.skv_status_string(skv.SKV_ERR_CONTEXT_FULL) == b"SKV_ERR_CONTEXT_FULL"
