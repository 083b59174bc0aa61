"""Host NUMA placement of the pool: the node nearest a GPU, read from fake
sysfs trees (CPU; no GPU, no real topology involved)."""
import os

import pytest


@pytest.fixture(scope="module")
def skv():
    from sparse_attention_kv_skv_gb300 import build
    build.build()
    from sparse_attention_kv_skv_gb300 import skv as mod
    return mod


def make_tree(root, nodes, dev="0000:01:00.0", local_cpus=None, numa_node=None):
    """nodes: {id: cpulist or ''}; the device's local_cpulist / numa_node files if given."""
    for n, cpus in nodes.items():
        d = os.path.join(root, "devices", "system", "node", f"node{n}")
        os.makedirs(d, exist_ok=True)
        with open(os.path.join(d, "cpulist"), "w") as f:
            f.write(cpus + "\n")
    d = os.path.join(root, "bus", "pci", "devices", dev)
    os.makedirs(d, exist_ok=True)
    if local_cpus is not None:
        with open(os.path.join(d, "local_cpulist"), "w") as f:
            f.write(local_cpus + "\n")
    if numa_node is not None:
        with open(os.path.join(d, "numa_node"), "w") as f:
            f.write(f"{numa_node}\n")
    return str(root)


def test_two_grace_sockets_device_on_the_second(skv, tmp_path):
    root = make_tree(tmp_path, {0: "0-71", 1: "72-143"}, local_cpus="72-143", numa_node=1)
    assert skv.host_node_for_pci("0000:01:00.0", root) == 1


def test_local_cpus_win_over_a_cpu_less_gpu_memory_node(skv, tmp_path):
    """On a coherent GPU the device's numa_node may be its own (CPU-less) memory node."""
    root = make_tree(tmp_path, {0: "0-71", 1: "72-143", 4: ""}, local_cpus="0-71", numa_node=4)
    assert skv.host_node_for_pci("0000:01:00.0", root) == 0


def test_without_local_cpus_the_device_node_if_it_has_cpus(skv, tmp_path):
    root = make_tree(tmp_path, {0: "0-3", 1: "4-7"}, numa_node=1)
    assert skv.host_node_for_pci("0000:01:00.0", root) == 1
    root2 = make_tree(tmp_path / "b", {0: "0-3", 2: ""}, numa_node=2)  # the device node has no CPUs
    assert skv.host_node_for_pci("0000:01:00.0", root2) == -1


def test_unknown_topology_gives_no_preference(skv, tmp_path):
    root = make_tree(tmp_path, {0: "0-15"}, numa_node=-1)
    assert skv.host_node_for_pci("0000:01:00.0", root) == -1
    assert skv.host_node_for_pci("0000:09:00.0", root) == -1      # no such device
    assert skv.host_node_for_pci("0000:01:00.0", str(tmp_path / "none")) == -1


def test_bus_id_forms_and_cpulist_syntax(skv, tmp_path):
    """CUDA may print an 8-digit domain and upper-case hex; cpulists mix ranges and singles."""
    root = make_tree(tmp_path, {0: "0-3,8-11", 1: "4-7,12,13-15"}, dev="0008:0a:00.0", local_cpus="12,14-15")
    assert skv.host_node_for_pci("00000008:0A:00.0", root) == 1
    assert skv.host_node_for_pci("0008:0A:00.0", root) == 1


def test_overlap_ties_go_to_the_lowest_node(skv, tmp_path):
    root = make_tree(tmp_path, {2: "0-3", 1: "4-7"}, local_cpus="2-5")
    assert skv.host_node_for_pci("0000:01:00.0", root) == 1


def test_null_arguments_are_rejected(skv):
    import ctypes
    n = ctypes.c_int32()
    assert skv.skv_host_node_for_pci(None, None, ctypes.byref(n)) == skv.SKV_ERR_INVALID_ARG
    assert skv.skv_host_node_for_pci(None, b"0000:01:00.0", None) == skv.SKV_ERR_INVALID_ARG
    assert skv.skv_pool_placement(None, None, None, None) == skv.SKV_ERR_INVALID_ARG
