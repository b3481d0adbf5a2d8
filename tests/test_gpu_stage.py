"""Host staging (mla_stage_copy): bit-exact round trips between pinned host
memory and device memory at the decode step's sizes and at ragged ones,
and the host-side rejection of memory the SMs cannot reach."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import mla_latent_kv_uk_gb300 as mod
    return mod


# 16 B, one CTA's round and a ragged tail, the decode step's packed input
# and output (B = 32, H = 128), and several full grids
SIZES = [16, 256 * 4 * 16 + 48, 1581312, 1064960, (64 << 20) + 16 * 7]


@pytest.mark.parametrize("nbytes", SIZES)
def test_round_trip_bit_exact(m, nbytes):
    g = torch.Generator().manual_seed(nbytes % 1000003)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).pin_memory()
    dev = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    m.mla_stage_copy(dev, src)
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    m.mla_stage_copy(back, dev)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), src)
    assert torch.equal(back, src)
    assert m.mla_get_device_error() == 0


def test_typed_views_and_neighbours_untouched(m):
    # a bf16 tensor staged into the middle of a larger device buffer: the
    # bytes around it keep their values
    x = torch.randn(32, 128, 192, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    host = x.pin_memory()
    buf = torch.full((host.numel() + 64,), -3.0, dtype=torch.bfloat16, device="cuda")
    view = buf[32:32 + host.numel()].view(32, 128, 192)
    m.mla_stage_copy(view, host)
    torch.cuda.synchronize()
    assert torch.equal(view.cpu(), x)
    assert torch.all(buf[:32].cpu() == -3.0) and torch.all(buf[-32:].cpu() == -3.0)


def test_inside_a_cuda_graph(m):
    n = 1 << 20
    src = torch.randint(0, 256, (n,), dtype=torch.uint8).pin_memory()
    dev = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out = torch.zeros(n, dtype=torch.uint8).pin_memory()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        m.mla_stage_copy(dev, src)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        m.mla_stage_copy(dev, src)
        dev.add_(1)
        m.mla_stage_copy(out, dev)
    for _ in range(3):
        src.random_(0, 200)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, src + 1)


def test_rejects_memory_the_sms_cannot_reach(m):
    n = 4096
    dev = torch.zeros(n, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(n, dtype=torch.uint8)
    pinned = torch.zeros(n, dtype=torch.uint8).pin_memory()
    L, s = m.lib, m._stream()
    import ctypes
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    # pageable host memory, device to device, host to host: refused on the
    # host, nothing launched
    assert L.mla_stage_copy(P(dev), P(pageable), n, s) == 1
    assert L.mla_stage_copy(P(pageable), P(dev), n, s) == 1
    dev2 = torch.zeros(n, dtype=torch.uint8, device="cuda")
    assert L.mla_stage_copy(P(dev2), P(dev), n, s) == 1
    pinned2 = torch.zeros(n, dtype=torch.uint8).pin_memory()
    assert L.mla_stage_copy(P(pinned2), P(pinned), n, s) == 1
    with pytest.raises(ValueError):
        m.mla_stage_copy(dev, pageable)
    torch.cuda.synchronize()
    assert m.mla_get_device_error() == 0
