"""dec_read_stream, the read-only HBM stream the bench reports as context for the weight
streams: it reads exactly dec_read_stream_bytes(n) bytes, writes nothing (the buffer is
unchanged) and leaves the device status clean; below 16 KB per SM it launches nothing."""
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


@pytest.mark.parametrize("nbytes", [64 << 20, (64 << 20) + 12345 * 16, 4096])
def test_read_stream_reads_and_writes_nothing(env, nbytes):
    torch, ssd, dev = env
    g = torch.Generator(device=dev).manual_seed(5)
    buf = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=dev, generator=g)
    ref = buf.clone()
    n = ssd.dec_read_stream(buf)
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    assert torch.equal(buf, ref)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    assert n == (nbytes // sms // 16384) * 16384 * sms
    assert n <= nbytes
