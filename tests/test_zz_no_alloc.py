"""qsa_index_scores_no_alloc: the scoring entry point for callers that cannot
allocate device memory (an engine whose memory manager owns every allocation,
code recording into a captured stream, latency-critical paths that cannot take
cudaMalloc's implicit synchronisation).  Its scratch is one static device array
shared by all calls.

Checked through the C ABI (ctypes on the shared library, no torch allocation
inside the call) against qsa_index_scores on the same inputs, on two calls in a
row, so that the second call starts from the array contents the first one left.
This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _lib():
    import sparse_attention_indexer_qsa_gb300 as qsa
    return qsa, qsa.load()


@pytest.mark.parametrize("B,S,NB,ctx", [(2, 1000, 250, [1000, 377]), (8, 4096, 1024, None)])
def test_no_alloc_matches_scores_on_consecutive_calls(B, S, NB, ctx):
    qsa, L = _lib()
    g = torch.Generator(device="cuda").manual_seed(B * S)
    q = torch.randn((B, S, 4, 128), device="cuda", generator=g).to(torch.bfloat16)
    kb = torch.randn((B, NB, 128), device="cuda", generator=g).to(torch.bfloat16)
    if ctx is None:
        c = torch.full((B,), S, dtype=torch.int32, device="cuda")
    else:
        c = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    rows = B * S
    ref = torch.empty((rows, NB), dtype=torch.float32, device="cuda")
    out = torch.full((rows, NB), 7.0, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = lambda o, r0, n: (0, o.data_ptr() + 4 * 0, q.data_ptr(), kb.data_ptr(), c.data_ptr(),
                             B, S, NB, r0, n, stream)
    assert L.qsa_index_scores(*args(ref, 0, rows)) == 0, qsa.qsa_last_error()
    for call in range(2):
        out.fill_(float(call + 3))
        assert L.qsa_index_scores_no_alloc(*args(out, 0, rows)) == 0, qsa.qsa_last_error()
        torch.cuda.synchronize()
        # same kernel and numerics: identical bits (within every tolerance the tests use)
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32)), f"call {call}"
    # a row chunk through the same shared scratch
    half = rows // 2
    part = torch.empty((rows - half, NB), dtype=torch.float32, device="cuda")
    assert L.qsa_index_scores_no_alloc(0, part.data_ptr(), q.data_ptr(), kb.data_ptr(), c.data_ptr(),
                                       B, S, NB, half, rows - half, stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(part.view(torch.int32), ref[half:].view(torch.int32))
    assert qsa.qsa_device_fault_flags() == 0


def test_no_alloc_rejects_bad_arguments_without_launching():
    qsa, L = _lib()
    P = 0x1000
    assert L.qsa_index_scores_no_alloc(0, P, P, None, P, 1, 8, 2, 0, 8, None) == -1
    assert L.qsa_index_scores_no_alloc(0, P, P, P, P, 2, 8, 2, 10, 7, None) == -3
    # work units beyond the static counter's range: 2^31-1 rows of one token each is
    # impossible here, but huge numBlocks with many rows exceeds the limit
    assert L.qsa_index_scores_no_alloc(0, P, P, P, P, 1, 2**30, 2**28, 0, 2**30, None) == -2
    assert "static scratch" in qsa.qsa_last_error()
