"""Host NUMA placement on a real GPU: a cache's pinned pages are requested on
the node sysfs gives for the GPU's PCI device and land there; DKV_NUMA=0
turns the placement off."""
import os

import pytest

import zero_copy_offloaded_gb300 as dkv

pytestmark = pytest.mark.gpu


def _bus_id():
    import torch
    p = torch.cuda.get_device_properties(0)
    return f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"


def test_cache_pages_on_the_gpus_node():
    want = dkv.dkv_pci_numa_node(_bus_id())
    c = dkv.KVCache(2, 8, 128, 4096, "bf16")
    try:
        info = dkv.dkv_cache_info(c.h)
        assert info["numa_node_wanted"] == want
        if want >= 0:
            assert info["numa_node"] == want
        print(f"GPU {_bus_id()}: host node wanted {want}, first page on {info['numa_node']}")
    finally:
        c.free()


def test_placement_off(monkeypatch):
    monkeypatch.setenv("DKV_NUMA", "0")
    c = dkv.KVCache(1, 2, 64, 64, "bf16")
    try:
        assert dkv.dkv_cache_info(c.h)["numa_node_wanted"] == -1
    finally:
        c.free()
