"""The read-only bandwidth probe consumes every byte it is timed on.

The probe's checksum is the XOR, over every 256-byte-aligned offset, of the
four 32-bit words at that offset: each lane of the probe consumes the first
16 bytes of each 256-byte piece its bulk copy brought in.  A probe that
skipped copies, or read the wrong bytes, gives another checksum.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def expected(buf):
    if buf.size == 0:
        return 0
    w = np.ascontiguousarray(buf.reshape(-1, 256)[:, :16]).view("<u4")
    return int(np.bitwise_xor.reduce(w.reshape(-1)))


@pytest.mark.parametrize("nbytes", [0, 256, 4096, 256 * 1000 + 256 * 7, 256 * 152 * 32 * 3 + 256 * 5,
                                    64 << 20])
def test_read_probe_checksum(nbytes):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import weight_quantized_decode_gb300 as q
    rng = np.random.Generator(np.random.PCG64(nbytes + 11))
    host = rng.integers(0, 256, size=nbytes, dtype=np.uint8)
    buf = torch.from_numpy(host).cuda()
    out = q.qmv_read_probe(buf)
    torch.cuda.synchronize()
    assert int(out.cpu().numpy().view(np.uint32)[0]) == expected(host)
    assert q.qmv_device_status() == 0


def test_read_probe_rejects_bad_sizes():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import weight_quantized_decode_gb300 as q
    buf = torch.zeros(300, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmvError):
        q.qmv_read_probe(buf)
