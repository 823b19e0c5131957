"""Host NUMA placement of the pinned caches, without a GPU: the node of a
GPU's host link is read from a fake sysfs tree (bus ids as CUDA prints them),
and a page allocated under the library's placement scope lands on the node
asked for and leaves the thread's policy as it found it.  Two gloo ranks each
resolve their own fake GPU to its own node, as replicas do on an 8-GPU host."""
import os

import pytest

import zero_copy_offloaded_gb300 as dkv


def _fake_sysfs(root, nodes):
    for bus_id, value in nodes.items():
        d = os.path.join(root, "bus", "pci", "devices", bus_id)
        os.makedirs(d, exist_ok=True)
        with open(os.path.join(d, "numa_node"), "w") as f:
            f.write(value)
    return str(root)


def test_pci_numa_node_from_sysfs(tmp_path):
    root = _fake_sysfs(tmp_path, {"0000:1b:00.0": "1\n", "0009:01:00.0": "3\n",
                                  "0000:2a:00.0": "-1\n", "0000:3c:00.0": "x\n",
                                  "0000:4d:00.0": ""})
    # CUDA prints hex digits upper-case; sysfs names them lower-case
    assert dkv.dkv_pci_numa_node("0000:1B:00.0", root) == 1
    assert dkv.dkv_pci_numa_node("00000009:01:00.0", root) == 3   # 8-digit domain
    assert dkv.dkv_pci_numa_node("0000:2A:00.0", root) == -1      # no node
    assert dkv.dkv_pci_numa_node("0000:3C:00.0", root) == -1      # malformed
    assert dkv.dkv_pci_numa_node("0000:4D:00.0", root) == -1      # empty
    assert dkv.dkv_pci_numa_node("0000:5e:00.0", root) == -1      # absent
    assert dkv.dkv_pci_numa_node("not a bus id", root) == -1


def _online_nodes():
    try:
        with open("/sys/devices/system/node/has_memory") as f:
            spec = f.read().strip()
    except OSError:
        return []
    nodes = []
    for part in spec.split(","):
        if "-" in part:
            a, b = part.split("-")
            nodes += list(range(int(a), int(b) + 1))
        elif part:
            nodes.append(int(part))
    return nodes


def test_placement_scope_puts_pages_on_the_node_and_restores_the_policy():
    nodes = _online_nodes()
    if not nodes:
        pytest.skip("no NUMA information on this machine")
    for n in nodes:
        assert dkv.dkv_numa_probe(n) == n
    # no preference (negative node): the page lands wherever the default policy puts it
    assert dkv.dkv_numa_probe(-1) in nodes
    # an impossible node changes nothing (the scope is not taken)
    assert dkv.dkv_numa_probe(1000) in nodes


def _rank_main(rank, world, root, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import torch
    bus = ["0000:1B:00.0", "0000:9C:00.0"][rank]    # this rank's (fake) GPU
    node = torch.tensor([dkv.dkv_pci_numa_node(bus, root)])
    got = [torch.zeros(1, dtype=node.dtype) for _ in range(world)]
    dist.all_gather(got, node)
    if rank == 0:
        out.put([int(t.item()) for t in got])
    dist.destroy_process_group()


def test_two_ranks_resolve_their_own_nodes(tmp_path):
    import multiprocessing as mp
    import socket
    root = _fake_sysfs(tmp_path, {"0000:1b:00.0": "0\n", "0000:9c:00.0": "1\n"})
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=_rank_main, args=(r, 2, root, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
    assert all(p.exitcode == 0 for p in ps)
    assert q.get(timeout=10) == [0, 1]
