"""Streaming-read probe (the memory-roofline measurement helper), GPU.

The probe XORs every 32-bit word of a buffer into a device word; the value is
checked against numpy's XOR of the same bytes for empty, tiny, ragged (not a
multiple of the probe's grid-stride step) and large buffers, and the argument
checks refuse ragged sizes and misaligned pointers.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
q = pytest.importorskip("bit_quantized_weight_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    yield


@pytest.mark.parametrize("nbytes", [0, 16, 4096 + 48, 3 * 2 ** 20 + 16, 64 * 2 ** 20 + 4096 + 32])
def test_read_probe_xor(nbytes):
    rng = np.random.default_rng(nbytes + 7)
    host = rng.integers(0, 2 ** 32, size=nbytes // 4, dtype=np.uint32)
    buf = torch.from_numpy(host.view(np.int32)).cuda()
    seed = 0x5A5A1234
    sink = torch.tensor([seed], dtype=torch.int32, device="cuda")
    q.read_probe(buf, sink)
    torch.cuda.synchronize()
    want = np.bitwise_xor.reduce(host, initial=np.uint32(seed)) if nbytes else np.uint32(seed)
    assert int(sink.cpu().numpy().view(np.uint32)[0]) == int(want)


def test_read_probe_rejects_ragged_and_misaligned():
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = q.lib()
    stream = torch.cuda.current_stream().cuda_stream
    assert L.qg_read_probe(buf.data_ptr(), 20, sink.data_ptr(), stream) == q.QG_ERR_INVALID_ARG
    assert L.qg_read_probe(buf.data_ptr() + 4, 32, sink.data_ptr(), stream) == q.QG_ERR_MISALIGNED
    assert L.qg_read_probe(None, 32, sink.data_ptr(), stream) == q.QG_ERR_INVALID_ARG
    torch.cuda.synchronize()
