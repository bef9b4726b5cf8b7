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
