"""w4_stream_read (the read-ceiling diagnostic the benchmark uses): it reads
every byte it is given.  The bulk-copy ring folds word 64*l of every 8 KB
record (l = 0..31) into one xor, which the host recomputes; the 128-bit-load
mode must be deterministic and report no wait that gave up."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def w4():
    from int4_weight_only_w4_gb300 import w4 as mod
    return mod


@pytest.mark.parametrize("records", [1, 7, 304, 1000])
def test_ring_reads_every_record(w4, records):
    rng = np.random.default_rng(records)
    host = rng.integers(0, 2 ** 32, size=records * 2048, dtype=np.uint64).astype(np.uint32)
    buf = torch.from_numpy(host.view(np.int32)).cuda()
    out = torch.zeros(2, dtype=torch.int32, device="cuda")
    w4.stream_read(buf, w4.STREAM_READ_RING, out)
    got = out.cpu().numpy().view(np.uint32)
    want = np.bitwise_xor.reduce(host.reshape(records, 2048)[:, ::64].ravel())
    assert got[1] == 0
    assert got[0] == want


def test_ld128_deterministic(w4):
    buf = torch.randint(-2 ** 31, 2 ** 31 - 1, (3 << 20,), dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(2):
        out = torch.zeros(2, dtype=torch.int32, device="cuda")
        w4.stream_read(buf, w4.STREAM_READ_LD128, out)
        outs.append(out.cpu().numpy())
    assert np.array_equal(outs[0], outs[1]) and outs[0][1] == 0


def test_stream_read_argument_errors(w4):
    buf = torch.zeros(8192 + 16, dtype=torch.uint8, device="cuda")
    out = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(w4.W4Error):
        w4.stream_read(buf, w4.STREAM_READ_RING, out)     # not a multiple of 8 KB
    with pytest.raises(w4.W4Error):
        w4.stream_read(buf, 7, out)                        # unknown mode
