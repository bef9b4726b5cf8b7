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
"""
from __future__ import annotations

import mmap
import os

import numpy as np
import torch

_PAGE = 4096


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

    def __init__(self, numel: int, dtype: torch.dtype, share: int = 1):
        nbytes = numel * torch.empty((), dtype=dtype).element_size()
        avail = available_host_bytes()
        if avail is not None and nbytes > 0.8 * avail / max(1, share):
            raise RuntimeError(f"{nbytes} B of page-locked host memory requested, "
                               f"{avail} B available for {max(1, share)} such buffer(s)")
        self._map = None
        self._raw = None
        self.kind = "torch pinned allocator"
        try:
            if nbytes == 0:
                raise ValueError("empty buffer")
            m = mmap.mmap(-1, nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
            if hasattr(mmap, "MADV_HUGEPAGE"):
                m.madvise(mmap.MADV_HUGEPAGE)
            raw = np.frombuffer(m, dtype=np.uint8)
            raw[::_PAGE] = 0  # fault every page in, huge pages where the kernel has them
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
