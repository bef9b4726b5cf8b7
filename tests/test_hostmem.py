"""hostmem on the host: the available-memory estimate and the refusal of a
page-locked buffer the host cannot hold, before any CUDA call."""
import pytest
import torch

from zero_sharded_mixed_04_gb300 import hostmem


def test_available_host_bytes_is_positive():
    avail = hostmem.available_host_bytes()
    assert avail is None or avail > 0


def test_oversized_buffer_is_refused_before_touching_memory():
    avail = hostmem.available_host_bytes()
    if avail is None:
        pytest.skip("no memory information on this host")
    with pytest.raises(RuntimeError, match="page-locked host memory requested"):
        hostmem.HostBuffer(avail // 2 + 1, torch.bfloat16)   # 1.0x of what is available
    # the same buffer shared among four ranks is refused at a quarter of the size
    with pytest.raises(RuntimeError):
        hostmem.HostBuffer(int(0.3 * avail) // 4, torch.float32, share=4)


def test_parse_cpulist():
    assert hostmem.parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert hostmem.parse_cpulist("") == set()


def _fake_sysfs(tmp_path, nodes, bus_id, numa_node, local_cpus):
    for n, cpus in nodes.items():
        d = tmp_path / "devices" / "system" / "node" / f"node{n}"
        d.mkdir(parents=True)
        (d / "cpulist").write_text(cpus + "\n")
    dev = tmp_path / "bus" / "pci" / "devices" / bus_id
    dev.mkdir(parents=True)
    (dev / "numa_node").write_text(f"{numa_node}\n")
    (dev / "local_cpulist").write_text(local_cpus + "\n")
    return str(tmp_path)


def test_gpu_numa_node_from_the_pci_function(tmp_path):
    root = _fake_sysfs(tmp_path, {0: "0-71", 1: "72-143", 2: ""}, "0009:01:00.0", 1, "72-143")
    assert hostmem.gpu_numa_node(bus_id="0009:01:00.0", sysfs=root) == 1


def test_gpu_numa_node_from_local_cpus_when_the_function_does_not_say(tmp_path):
    # numa_node -1 (unknown) or a node without CPUs (the GPU's own memory)
    root = _fake_sysfs(tmp_path, {0: "0-71", 1: "72-143", 4: ""}, "0019:01:00.0", 4, "72-100")
    assert hostmem.gpu_numa_node(bus_id="0019:01:00.0", sysfs=root) == 1
    root2 = _fake_sysfs(tmp_path / "b", {0: "0-15"}, "0000:05:00.0", -1, "0-15")
    assert hostmem.gpu_numa_node(bus_id="0000:05:00.0", sysfs=root2) == 0


def test_gpu_numa_node_unknown(tmp_path):
    assert hostmem.gpu_numa_node(bus_id="0000:00:00.0", sysfs=str(tmp_path)) is None


def test_preferred_node_on_this_host():
    """mbind and move_pages on a small mapping of this host: either they work
    and the sampled pages sit on the preferred node, or they are unavailable
    (no such call on this machine, or a sandbox refuses it)."""
    import mmap
    import numpy as np
    nodes = hostmem.cpu_nodes()
    if not nodes:
        pytest.skip("no NUMA information")
    node = min(nodes)
    n = 64 * 4096
    m = mmap.mmap(-1, n, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
    raw = np.frombuffer(m, dtype=np.uint8)
    ok = hostmem.mbind_preferred(raw.ctypes.data, n, node)
    raw[::4096] = 1
    frac = hostmem.pages_on_node(raw.ctypes.data, n, node)
    if ok and frac is not None:
        assert frac == 1.0
    del raw
    m.close()
