"""Page-locked host buffers used by the streamed validator and the end-to-end
bench leg: registered with the driver (so copies from them are asynchronous
DMA), the right size and type, and a round trip through the device returns
the same bytes."""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("numel", [1, 4097, 3 << 20])
def test_pinned_buffer_round_trip(numel):
    from decode_gemv_sign_gb300.hostmem import PinnedBuffer

    b = PinnedBuffer(torch, numel, torch.int16)
    h = b.tensor
    assert h.dtype == torch.int16 and h.numel() == numel and h.is_pinned()
    g = torch.Generator().manual_seed(numel)
    h.copy_(torch.randint(-32768, 32767, (numel,), dtype=torch.int16, generator=g))
    want = h.clone()
    d = torch.empty(numel, dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d.copy_(h, non_blocking=True)
    s.synchronize()
    h2 = PinnedBuffer(torch, numel, torch.int16)
    with torch.cuda.stream(s):
        h2.tensor.copy_(d, non_blocking=True)
    s.synchronize()
    assert torch.equal(h2.tensor, want)
    b.release()
    h2.release()
    b.release()  # releasing twice is harmless
