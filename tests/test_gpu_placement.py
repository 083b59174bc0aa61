"""The host pool's NUMA placement on the GPU machine: skv_create asks for the host
node nearest the GPU, read from the real sysfs, and the kernel's report of a
sample of pool pages agrees; SKV_POOL_NODE=-1 asks for nothing.  (GPU)"""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _bus_id(dev=0):
    p = torch.cuda.get_device_properties(dev)
    if all(hasattr(p, a) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
        return f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    import subprocess
    out = subprocess.run(["nvidia-smi", "-i", str(dev), "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                         capture_output=True, text=True, check=True).stdout.strip()
    return out


def test_pool_is_asked_for_and_lands_on_the_nearest_node(monkeypatch):
    from sparse_attention_kv_skv_gb300 import Config, Context, skv
    monkeypatch.delenv("SKV_POOL_NODE", raising=False)
    want = skv.host_node_for_pci(_bus_id())
    with Context(Config(max_requests=4, num_layers=2, max_context=65536, topk=64, hot_slots=128,
                        max_batch=4)) as ctx:
        wanted, seen, frac = ctx.pool_placement()
        print(f"pool placement: nearest node {want}, asked {wanted}, seen {seen} ({frac:.2f} of the sample)")
        assert wanted == want
        if wanted >= 0 and seen >= 0:
            assert seen == wanted and frac >= 0.9


def test_no_preference_when_told(monkeypatch):
    from sparse_attention_kv_skv_gb300 import Config, Context
    monkeypatch.setenv("SKV_POOL_NODE", "-1")
    with Context(Config(max_requests=1, num_layers=1, max_context=1024, topk=16, hot_slots=32,
                        max_batch=1)) as ctx:
        assert ctx.pool_placement()[0] == -1
