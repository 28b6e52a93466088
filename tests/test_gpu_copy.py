"""sd_copy: kernel copies between device memory and pinned host memory (reached by
the device at the same address), bit for bit, at sizes from one 16-byte word to
several megabytes, inside and outside a CUDA graph."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_sparse_decode_gb300 import build as b
    b.build()
    import top_sparse_decode_gb300 as m
    m.lib()
    return m


@pytest.mark.parametrize("nbytes", [16, 8192, 16512, 3 * (1 << 20) + 48])
def test_copy_host_device_round_trip(sd, nbytes):
    rng = np.random.default_rng(nbytes)
    src = torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8)).pin_memory()
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dev2 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    sd.sd_copy(dev, src)    # pinned host -> device
    sd.sd_copy(dev2, dev)   # device -> device
    sd.sd_copy(back, dev2)  # device -> pinned host
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), src)
    assert torch.equal(back, src)


def test_copy_in_a_graph(sd):
    n = 16512
    src = torch.arange(n // 4, dtype=torch.int32).pin_memory()
    dev = torch.empty(n // 4, dtype=torch.int32, device="cuda")
    back = torch.zeros(n // 4, dtype=torch.int32).pin_memory()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            sd.sd_copy(dev, src)
            sd.sd_copy(back, dev)
    torch.cuda.current_stream().wait_stream(s)
    for k in range(3):
        src.copy_(torch.arange(n // 4, dtype=torch.int32) * (k + 2))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(back, src)
