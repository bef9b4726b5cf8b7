"""Page-locked host buffers backed by huge pages.

A buffer is an anonymous mapping advised for transparent huge pages, faulted
in, and registered with the CUDA driver (cudaHostRegister), so the GPU's copy
engines and kernels reach it like any pinned memory.  On a GB300 host whose
memory had been through heavy use (the GPU test suite just before), steps that
streamed 16 GB of gradients per step from a buffer of torch's pinned allocator
stalled intermittently, 77 to 290 ms for a 77 ms step, while the copies alone
ran at the full 211 GB/s.  From a huge-page buffer the same steps took 77 ms,
with an occasional 105 ms one.  If the mapping or the registration fails, the
buffer comes from torch's pinned allocator instead; ``kind`` says which.

Pages of the mapping are faulted in before registration, so a request larger
than the host can hold would meet the kernel's out-of-memory killer rather
than an error.  A buffer is therefore refused (RuntimeError) unless it fits in
80 % of the memory available to this process, shared by ``share`` such
buffers allocated at once (one per rank on the node, say).

NUMA placement.  A host with several memory nodes serves a GPU fastest from
the node next to it.  Given ``numa_node``, the mapping is given that node as
its preferred node (``mbind`` with MPOL_PREFERRED) before its pages are
faulted in, whichever CPU the process runs on; the kernel falls back to other
nodes only when that one is full.  ``gpu_numa_node`` finds the node: the GPU's
PCI function's ``numa_node``, else the node of the CPUs listed as local to it.
Nodes without CPUs (a GPU's own memory exposed as a node, say) are never
chosen.  Afterwards ``pages_on_node`` samples where the pages actually are.
"""
from __future__ import annotations

import ctypes
import mmap
import os
import platform
import subprocess

import numpy as np
import torch

_PAGE = 4096
_MPOL_PREFERRED = 1
# system call numbers of mbind and move_pages (Linux, per architecture)
_SYSCALLS = {"aarch64": {"mbind": 235, "move_pages": 239},
             "x86_64": {"mbind": 237, "move_pages": 279}}
SYSFS = "/sys"


def parse_cpulist(text: str) -> set[int]:
    """CPUs of a sysfs cpulist such as "0-3,8,10-11"."""
    cpus: set[int] = set()
    for part in text.strip().split(","):
        if not part:
            continue
        if "-" in part:
            lo, hi = part.split("-")
            cpus.update(range(int(lo), int(hi) + 1))
        else:
            cpus.add(int(part))
    return cpus


def cpu_nodes(sysfs: str = SYSFS) -> dict[int, set[int]]:
    """NUMA nodes that have CPUs, with their CPUs."""
    out: dict[int, set[int]] = {}
    base = os.path.join(sysfs, "devices", "system", "node")
    try:
        names = os.listdir(base)
    except OSError:
        return out
    for name in names:
        if not (name.startswith("node") and name[4:].isdigit()):
            continue
        try:
            with open(os.path.join(base, name, "cpulist")) as f:
                cpus = parse_cpulist(f.read())
        except OSError:
            continue
        if cpus:
            out[int(name[4:])] = cpus
    return out


def gpu_pci_bus_id(device) -> str | None:
    """The PCI address (domain:bus:device.function) of a CUDA device."""
    try:
        p = torch.cuda.get_device_properties(device)
        return "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except (AttributeError, RuntimeError, AssertionError):
        pass
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        out = subprocess.run(["nvidia-smi", "--query-gpu=uuid,pci.bus_id",
                              "--format=csv,noheader"], capture_output=True, text=True,
                             timeout=30).stdout
        for line in out.splitlines():
            u, bus = [x.strip() for x in line.split(",")]
            if u.endswith(uuid) or uuid.endswith(u.replace("GPU-", "")):
                dom, rest = bus.split(":", 1)
                return f"{int(dom, 16) & 0xffff:04x}:{rest}".lower()
    except (OSError, ValueError, subprocess.SubprocessError):
        pass
    return None


def gpu_numa_node(device=None, bus_id: str | None = None, sysfs: str = SYSFS) -> int | None:
    """The host memory node nearest a GPU, or None if the host does not say."""
    nodes = cpu_nodes(sysfs)
    if len(nodes) == 0:
        return None
    bus_id = bus_id or (gpu_pci_bus_id(device) if device is not None else None)
    if bus_id is None:
        return None
    dev_dir = os.path.join(sysfs, "bus", "pci", "devices", bus_id)
    try:
        with open(os.path.join(dev_dir, "numa_node")) as f:
            n = int(f.read().strip())
        if n in nodes:
            return n
    except (OSError, ValueError):
        pass
    try:
        with open(os.path.join(dev_dir, "local_cpulist")) as f:
            local = parse_cpulist(f.read())
    except (OSError, ValueError):
        return None
    best = max(nodes, key=lambda k: len(nodes[k] & local))
    return best if nodes[best] & local else None


def _syscall(name: str):
    nr = _SYSCALLS.get(platform.machine(), {}).get(name)
    if nr is None:
        return None, None
    libc = ctypes.CDLL(None, use_errno=True)
    return libc.syscall, nr


def mbind_preferred(addr: int, nbytes: int, node: int) -> bool:
    """Give [addr, addr + nbytes) the preferred node ``node`` (MPOL_PREFERRED)."""
    call, nr = _syscall("mbind")
    if call is None or not 0 <= node < 64:
        return False
    mask = ctypes.c_ulong(1 << node)
    rc = call(ctypes.c_long(nr), ctypes.c_void_p(addr), ctypes.c_ulong(nbytes),
              ctypes.c_int(_MPOL_PREFERRED), ctypes.byref(mask), ctypes.c_ulong(65),
              ctypes.c_uint(0))
    return rc == 0


def pages_on_node(addr: int, nbytes: int, node: int, samples: int = 512) -> float | None:
    """Fraction of a sample of the range's (faulted-in) pages that sit on
    ``node``, by move_pages with no target nodes; None if it cannot be read."""
    call, nr = _syscall("move_pages")
    if call is None or nbytes <= 0:
        return None
    n_pages = (nbytes + _PAGE - 1) // _PAGE
    k = max(1, min(samples, n_pages))
    idx = np.unique(np.linspace(0, n_pages - 1, k).astype(np.int64))
    pages = (ctypes.c_void_p * idx.size)(*[addr + int(i) * _PAGE for i in idx])
    status = (ctypes.c_int * idx.size)()
    rc = call(ctypes.c_long(nr), ctypes.c_int(0), ctypes.c_ulong(idx.size), pages, None, status,
              ctypes.c_int(0))
    if rc != 0:
        return None
    st = np.array(status[:], dtype=np.int64)
    return float((st == node).sum()) / st.size


def available_host_bytes() -> int | None:
    """Memory this process may still fault in: MemAvailable, capped by the
    cgroup's limit less its usage where one is set.  None if unknown."""
    avail = None
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    avail = int(line.split()[1]) * 1024
    except OSError:
        pass
    try:
        with open("/sys/fs/cgroup/memory.max") as f:
            limit = f.read().strip()
        with open("/sys/fs/cgroup/memory.current") as f:
            used = int(f.read().strip())
        if limit != "max":
            room = int(limit) - used
            avail = room if avail is None else min(avail, room)
    except (OSError, ValueError):
        pass
    return avail


class HostBuffer:
    """``numel`` elements of ``dtype`` in page-locked host memory, as the torch
    tensor ``tensor``.  Call ``close()`` once no tensor view of it is in use;
    it unregisters the memory."""

    def __init__(self, numel: int, dtype: torch.dtype, share: int = 1,
                 numa_node: int | None = None):
        nbytes = numel * torch.empty((), dtype=dtype).element_size()
        avail = available_host_bytes()
        if avail is not None and nbytes > 0.8 * avail / max(1, share):
            raise RuntimeError(f"{nbytes} B of page-locked host memory requested, "
                               f"{avail} B available for {max(1, share)} such buffer(s)")
        self._map = None
        self._raw = None
        self.kind = "torch pinned allocator"
        self.numa_node = None        # the preferred node the mapping was given
        self.numa_placed = None      # sampled fraction of its pages on that node
        try:
            if nbytes == 0:
                raise ValueError("empty buffer")
            m = mmap.mmap(-1, nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
            if hasattr(mmap, "MADV_HUGEPAGE"):
                m.madvise(mmap.MADV_HUGEPAGE)
            raw = np.frombuffer(m, dtype=np.uint8)
            if numa_node is not None and mbind_preferred(raw.ctypes.data, nbytes, numa_node):
                self.numa_node = numa_node
            raw[::_PAGE] = 0  # fault every page in, huge pages where the kernel has them
            if self.numa_node is not None:
                self.numa_placed = pages_on_node(raw.ctypes.data, nbytes, self.numa_node)
            err = torch.cuda.cudart().cudaHostRegister(raw.ctypes.data, nbytes, 0)
            if int(err) != 0:
                raise RuntimeError(f"cudaHostRegister returned {int(err)}")
            self._map, self._raw = m, raw
            self.tensor = torch.from_numpy(raw).view(dtype)
            self.kind = "huge-page mapping, cudaHostRegister"
        except (OSError, RuntimeError, ValueError, AttributeError):
            self.tensor = torch.empty(numel, dtype=dtype, pin_memory=True)

    def close(self) -> None:
        if self._raw is not None:
            self.tensor = None
            torch.cuda.cudart().cudaHostUnregister(self._raw.ctypes.data)
            self._raw = None
            self._map = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # the CUDA runtime may already be gone at exit
            pass
