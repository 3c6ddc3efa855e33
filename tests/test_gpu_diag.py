"""The diagnostic read stream reads every word of its buffer exactly once: the xor of
all CTAs' folds equals the xor of every 32-bit word of the buffer."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mem():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_decode_quantize_gb300 as m
    from block_quantized_decode_quantize_gb300 import build
    build.build()
    m.lib()
    return m


@pytest.mark.parametrize("nbytes,ctas", [(16, 1), (4096 * 16 + 48, 2), ((1 << 26) + 16 * 7, 4)])
def test_read_stream_reads_every_word_once(mem, nbytes, ctas):
    raw = np.random.default_rng(nbytes).integers(0, 1 << 32, size=nbytes // 4, dtype=np.uint32)
    buf = torch.from_numpy(raw.view(np.int32)).cuda()
    sink = mem.memra_read_stream(buf, ctas_per_sm=ctas)
    torch.cuda.synchronize()
    folded = np.bitwise_xor.reduce(sink.cpu().numpy().view(np.uint32))
    assert folded == np.bitwise_xor.reduce(raw)


def test_read_stream_rejects_bad_sizes(mem):
    buf = torch.zeros((8,), dtype=torch.int32, device="cuda")
    lib = mem.lib()
    sink = torch.zeros((1024,), dtype=torch.int32, device="cuda")
    assert lib.memra_read_stream(buf.data_ptr(), 24, sink.data_ptr(), 2, None) == 1  # not /16
    assert lib.memra_read_stream(buf.data_ptr(), 32, sink.data_ptr(), 5, None) == 1  # ctas
    assert lib.memra_read_stream(buf.data_ptr() + 4, 16, sink.data_ptr(), 1, None) == 2
