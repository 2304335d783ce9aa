"""dec_read_stream, the read-only HBM stream the bench reports as context for the weight
streams: it reads dec_read_stream_bytes(n) bytes (whole 256 KB chunks), writes nothing
(the buffer is unchanged), leaves the device status clean and can be called again at once
(its chunk counter is zeroed before every launch); below one chunk it launches nothing."""
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import split_switched_decode_gb300 as ssd
    ssd.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    return torch, ssd, dev


@pytest.mark.parametrize("nbytes", [64 << 20, (64 << 20) + 12345 * 16, (256 << 10) + 16, 4096])
def test_read_stream_reads_and_writes_nothing(env, nbytes):
    torch, ssd, dev = env
    g = torch.Generator(device=dev).manual_seed(5)
    buf = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=dev, generator=g)
    ref = buf.clone()
    for _ in range(3):
        n = ssd.dec_read_stream(buf)
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    assert torch.equal(buf, ref)
    assert n == (nbytes // (256 << 10)) * (256 << 10)
    assert n <= nbytes
