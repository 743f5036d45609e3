"""The bench's same-size bandwidth yardsticks move the bytes they claim to.

They are plain kernels with no computation of the page: qsa_testing_stream_yardstick has
the K1 kernels' byte patterns, and qsa_testing_gather_yardstick the paged decode scoring's
(one 256-byte V-tail a block at the pool's block pitch in, 4 bytes a block out).  Their
outputs are XORs of what they read, checked here against numpy on a random byte buffer,
with unit counts that leave ragged groups and CTAs.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _qsa():
    import sparse_attention_indexer_qsa_gb300 as qsa
    return qsa


@pytest.mark.parametrize("units,pitch,offset,nbytes", [(1001, 6144, 512, 256), (37, 48, 16, 16),
                                                       (130, 1024, 0, 512), (1, 6144, 512, 256)])
def test_gather_yardstick_xors_each_units_words(units, pitch, offset, nbytes):
    qsa = _qsa()
    rng = np.random.default_rng(units + nbytes)
    size = (units - 1) * pitch + offset + nbytes
    host = rng.integers(0, 256, size=size + 64, dtype=np.uint8)
    src = torch.from_numpy(host).cuda()
    dst = torch.full((units + 1,), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    qsa.qsa_testing_gather_yardstick(dst, src, units, pitch, offset, nbytes)
    torch.cuda.synchronize()
    got = dst.cpu().numpy().view(np.uint32)
    idx = np.arange(units)[:, None] * pitch + offset + np.arange(nbytes)[None, :]
    words = host[idx].reshape(units, nbytes // 4, 4).copy().view("<u4").reshape(units, nbytes // 4)
    want = np.bitwise_xor.reduce(words, axis=1)
    assert np.array_equal(got[:units], want)
    assert got[units] == 0x5A5A5A5A  # nothing written past the last unit


def test_stream_yardstick_xors_each_units_rows():
    qsa = _qsa()
    units, rows, rp, up, off, nb = 333, 4, 1280, 5120, 1024, 256
    rng = np.random.default_rng(3)
    size = (units - 1) * up + (rows - 1) * rp + off + nb
    host = rng.integers(0, 256, size=size, dtype=np.uint8)
    src = torch.from_numpy(host).cuda()
    dst = torch.zeros(units * nb + 16, dtype=torch.uint8, device="cuda")
    qsa.qsa_testing_stream_yardstick(dst, src, units, rows, rp, up, off, nb)
    torch.cuda.synchronize()
    got = dst.cpu().numpy()
    base = np.arange(units)[:, None] * up + off + np.arange(nb)[None, :]
    want = host[base]
    for r in range(1, rows):
        want = want ^ host[base + r * rp]
    assert np.array_equal(got[:units * nb].reshape(units, nb), want)
    assert not got[units * nb:].any()
