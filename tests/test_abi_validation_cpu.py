"""Host-side validation of the fused-K1, selection, paged-pool and decode entry points,
without a GPU.

Every check in the C ABI runs before the library touches CUDA, so each bad argument
must come back as its status code and a message here. A call whose arguments pass
must reach the device query and, on a host with no GPU, fail loudly with
QSA_E_CUDA: there is no host fallback that could return QSA_OK.
"""
import ctypes

import pytest
import torch

# Some calls below pass validation on purpose, with fake device addresses.  Where a GPU is
# visible they would launch kernels on those addresses, so the whole file runs only on hosts
# without one (the GPU tests check the same validation with real buffers).
pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="fake device addresses: host without a GPU only")

E_NULL, E_SHAPE, E_RANGE, E_DTYPE, E_ALIGN, E_CUDA, E_DEVICE = -1, -2, -3, -4, -5, -6, -7
P = 0x1000  # a 16-byte aligned fake device address: never dereferenced on these paths


@pytest.fixture(scope="module")
def qsa():
    from sparse_attention_indexer_qsa_gb300 import build as b
    b.build()
    import sparse_attention_indexer_qsa_gb300 as q
    return q


def pool(qsa, **kw):
    f = dict(poolPtr=P, pageTable=P, maxPagesPerSeq=4, numPages=8, numKVHeads=2, poolHeadDim=384, headSize=256)
    f.update(kw)
    st = qsa.PoolState(f["poolPtr"], f["pageTable"], f["maxPagesPerSeq"], f["numPages"], f["numKVHeads"],
                       f["poolHeadDim"], f["headSize"])
    return ctypes.byref(st), st


def test_fused_qk_prep(qsa):
    L = qsa.load()
    ok = lambda **o: [o.get(k, v) for k, v in dict(dt=0, qn=P, kb=P, iq=P, cs=P, ctx=P, wq=P, wk=P, eps=1e-6,
                                                    B=2, S=9, NB=3, st=None).items()]
    assert L.qsa_index_qk_prep(*ok(dt=3)) == E_DTYPE
    assert L.qsa_index_qk_prep(*ok(kb=None)) == E_NULL
    assert L.qsa_index_qk_prep(*ok(wk=None)) == E_NULL
    assert L.qsa_index_qk_prep(*ok(B=0)) == E_SHAPE
    assert L.qsa_index_qk_prep(*ok(NB=2)) == E_SHAPE          # numBlocks < ceilDiv(9, 4)
    assert L.qsa_index_qk_prep(*ok(B=65536, S=65536, NB=16384)) == E_SHAPE
    assert L.qsa_index_qk_prep(*ok(kb=P + 8)) == E_ALIGN
    assert L.qsa_index_qk_prep(*ok(ctx=P + 2)) == E_ALIGN
    assert "qsa_index_qk_prep" in qsa.qsa_last_error()


def test_selection_entries(qsa):
    L = qsa.load()
    assert L.qsa_index_ids_fill(None, 4, 8, None) == E_NULL
    assert L.qsa_index_ids_fill(P, -1, 8, None) == E_SHAPE
    assert L.qsa_index_ids_fill(P, 4, 0, None) == E_SHAPE
    assert L.qsa_index_ids_fill(P + 2, 4, 8, None) == E_ALIGN
    assert L.qsa_index_ids_fill(P, 0, 8, None) == 0           # empty: no device needed
    for fn in (L.qsa_index_expand, L.qsa_index_topk_expand):
        ok = lambda **o: [o.get(k, v) for k, v in dict(out=P, inp=P, ctx=P, B=2, S=16, NB=4, r0=0, n=32,
                                                        st=None).items()]
        assert fn(*ok(out=None)) == E_NULL
        assert fn(*ok(inp=None)) == E_NULL
        assert fn(*ok(S=0)) == E_SHAPE
        assert fn(*ok(NB=3)) == E_SHAPE                     # < ceilDiv(16, 4)
        assert fn(*ok(r0=1)) == E_RANGE                     # rows [1, 33) outside [0, 32)
        assert fn(*ok(r0=-1, n=1)) == E_RANGE
        assert fn(*ok(n=-1)) == E_RANGE
        assert fn(*ok(ctx=P + 1)) == E_ALIGN
        assert fn(*ok(n=0)) == 0
    # the fused top-k keeps a row's keys on chip: rows of at most 65536 blocks
    assert L.qsa_index_topk_expand(P, P, P, 1, 8, 65537, 0, 8, None) == E_SHAPE
    assert "65536" in qsa.qsa_last_error()


def test_fused_scores_topk_expand(qsa):
    L = qsa.load()
    ok = lambda **o: [o.get(k, v) for k, v in dict(dt=0, out=P, q=P, kb=P, ctx=P, B=2, S=16, NB=4, r0=0, n=32,
                                                    st=None).items()]
    f = L.qsa_index_scores_topk_expand
    assert f(*ok(dt=2)) == E_DTYPE
    for arg in ("out", "q", "kb", "ctx"):
        assert f(*ok(**{arg: None})) == E_NULL
    assert f(*ok(S=0)) == E_SHAPE
    assert f(*ok(NB=3)) == E_SHAPE                        # < ceilDiv(16, 4)
    assert f(*ok(r0=1)) == E_RANGE
    assert f(*ok(n=-1)) == E_RANGE
    assert f(*ok(q=P + 8)) == E_ALIGN
    assert f(*ok(kb=P + 8)) == E_ALIGN
    assert f(*ok(out=P + 2)) == E_ALIGN
    assert f(*ok(n=0)) == 0
    # a row's selection state lives in shared memory: rows of at most 4096 blocks
    assert f(*ok(NB=4097)) == E_SHAPE
    assert "4096" in qsa.qsa_last_error()


def test_stream_yardstick(qsa):
    L = qsa.load()
    ok = lambda **o: [o.get(k, v) for k, v in dict(dst=P, src=P, units=8, rows=4, rp=1280, up=5120, off=1024,
                                                    nb=256, st=None).items()]
    f = L.qsa_testing_stream_yardstick
    assert f(*ok(dst=None)) == E_NULL
    assert f(*ok(rows=0)) == E_SHAPE
    assert f(*ok(rows=9)) == E_SHAPE
    assert f(*ok(nb=24)) == E_SHAPE
    assert f(*ok(nb=2048)) == E_SHAPE
    assert f(*ok(units=-1)) == E_SHAPE
    assert f(*ok(off=8)) == E_ALIGN
    assert f(*ok(src=P + 8)) == E_ALIGN
    assert f(*ok(units=0)) == 0
    assert f(*ok()) == E_CUDA


def test_gather_yardstick(qsa):
    L = qsa.load()
    ok = lambda **o: [o.get(k, v) for k, v in dict(dst=P, src=P, units=8, up=6144, off=512, nb=256,
                                                    st=None).items()]
    f = L.qsa_testing_gather_yardstick
    assert f(*ok(dst=None)) == E_NULL
    assert f(*ok(nb=8)) == E_SHAPE
    assert f(*ok(nb=768)) == E_SHAPE  # a multiple of 16 but not a power of two
    assert f(*ok(nb=1024)) == E_SHAPE
    assert f(*ok(units=-1)) == E_SHAPE
    assert f(*ok(off=8)) == E_ALIGN
    assert f(*ok(up=6152)) == E_ALIGN
    assert f(*ok(src=P + 8)) == E_ALIGN
    assert f(*ok(dst=P + 2)) == E_ALIGN
    assert f(*ok(units=0)) == 0
    assert f(*ok()) == E_CUDA


def test_pool_state_is_checked_by_every_paged_entry(qsa):
    L = qsa.load()
    calls = {
        "k_compress_paged": lambda ps: L.qsa_index_k_compress_paged(0, P, P, P, P, P, 1e-6, ps, 2, 8, 2, 0, 2, 0,
                                                                      None),
        "raw_k_tail_write_prefill": lambda ps: L.qsa_raw_k_tail_write_prefill(0, P, P, ps, 2, 8, None),
        "pre_decode": lambda ps: L.qsa_indexer_pre_decode(0, P, P, P, P, P, P, 1e-6, ps, 2, None),
        "scores_decode": lambda ps: L.qsa_index_scores_decode(0, P, P, P, ps, 2, 64, None),
        "decode_step": lambda ps: L.qsa_indexer_decode_step(0, P, P, P, P, P, P, P, P, 1e-6, ps, None, 0, 2, 64,
                                                             None),
    }
    for name, call in calls.items():
        assert call(None) == E_NULL, name
        assert call(pool(qsa, poolPtr=0)[0]) == E_NULL, name
        assert call(pool(qsa, pageTable=0)[0]) == E_NULL, name
        assert call(pool(qsa, maxPagesPerSeq=0)[0]) == E_SHAPE, name
        assert call(pool(qsa, numPages=0)[0]) == E_SHAPE, name
        assert call(pool(qsa, numKVHeads=0)[0]) == E_SHAPE, name
        assert call(pool(qsa, headSize=-8)[0]) == E_SHAPE, name
        assert call(pool(qsa, headSize=300)[0]) == E_SHAPE, name       # headSize + 128 > poolHeadDim
        assert call(pool(qsa, headSize=252, poolHeadDim=384)[0]) == E_ALIGN, name
        assert call(pool(qsa, poolHeadDim=388, headSize=256)[0]) == E_ALIGN, name
        assert call(pool(qsa, poolPtr=P + 8)[0]) == E_ALIGN, name
        assert call(pool(qsa, pageTable=P + 2)[0]) == E_ALIGN, name
        assert "pool" in qsa.qsa_last_error(), name


def test_paged_and_decode_shapes_ranges_and_alignment(qsa):
    L = qsa.load()
    ps, _keep = pool(qsa)
    # paged K1b: the sub-range contract of K1b
    kcp = lambda **o: L.qsa_index_k_compress_paged(*[o.get(k, v) for k, v in dict(
        dt=0, kb=P, iq=P, cs=P, ctx=P, wk=P, eps=1e-6, ps=ps, B=2, S=8, NB=2, b0=0, b1=2, past=0,
        st=None).items()])
    assert kcp(dt=2) == E_DTYPE
    assert kcp(NB=0, b1=0) == E_SHAPE
    assert kcp(b0=1, b1=0) == E_RANGE
    assert kcp(b1=3) == E_RANGE
    assert kcp(past=-4) == E_RANGE
    assert kcp(iq=P + 4) == E_ALIGN
    assert kcp(b0=1, b1=1) == 0                                     # empty range
    # raw K-tails, pre-decode, decode scores
    assert L.qsa_raw_k_tail_write_prefill(0, P, P, ps, 0, 8, None) == E_SHAPE
    assert L.qsa_raw_k_tail_write_prefill(0, P + 2, P, ps, 1, 8, None) == E_ALIGN
    assert L.qsa_indexer_pre_decode(0, P, P, P, P, P, P, 1e-6, ps, 0, None) == E_SHAPE
    assert L.qsa_indexer_pre_decode(0, P, P, P, P, None, P, 1e-6, ps, 2, None) == E_NULL
    assert L.qsa_indexer_pre_decode(0, P, P, P + 4, P, P, P, 1e-6, ps, 2, None) == E_ALIGN
    assert L.qsa_index_scores_decode(0, P, P, P, ps, 2, 0, None) == E_SHAPE
    assert L.qsa_index_scores_decode(0, P, P, P, ps, 2, 65535 * 256 + 1, None) == E_SHAPE
    assert L.qsa_index_scores_decode(0, P, P + 2, P, ps, 2, 64, None) == E_ALIGN
    # decode top-k: split counters optional; rows of at most 65536 blocks
    assert L.qsa_topk_expand_decode(P, None, P, None, 0, 2, 64, None) == E_NULL
    assert L.qsa_topk_expand_decode(P, P, P, P, -1, 2, 64, None) == E_SHAPE
    assert L.qsa_topk_expand_decode(P, P, P, None, 0, 2, 65537, None) == E_SHAPE
    assert L.qsa_topk_expand_decode(P, P, P, P + 2, 2, 2, 64, None) == E_ALIGN
    # the one-launch decode step: batch limit 4096, maxBlocks limit 65536
    step = lambda **o: L.qsa_indexer_decode_step(*[o.get(k, v) for k, v in dict(
        dt=0, out=P, lg=P, qn=P, iq=P, cs=P, ctx=P, wq=P, wk=P, eps=1e-6, ps=ps, split=None, nkv=0, B=2,
        maxb=64, st=None).items()])
    assert step(out=None) == E_NULL
    assert step(B=0) == E_SHAPE
    assert step(B=4097) == E_SHAPE
    assert step(maxb=0) == E_SHAPE
    assert step(maxb=65537) == E_SHAPE
    assert step(split=P, nkv=-1) == E_SHAPE
    assert step(wq=P + 2) == E_ALIGN
    assert step(split=P + 1, nkv=2) == E_ALIGN


def test_no_gpu_means_a_loud_cuda_error(qsa):
    """Arguments that pass every check reach the device query, which fails on this host."""
    L = qsa.load()
    ps, _keep = pool(qsa)
    assert L.qsa_index_qk_prep(0, P, P, P, P, P, P, P, 1e-6, 2, 9, 3, None) == E_CUDA
    assert L.qsa_index_ids_fill(P, 4, 8, None) == E_CUDA
    assert L.qsa_index_expand(P, P, P, 2, 16, 4, 0, 32, None) == E_CUDA
    assert L.qsa_index_topk_expand(P, P, P, 2, 16, 4, 0, 32, None) == E_CUDA
    assert L.qsa_index_k_compress_paged(0, P, P, P, P, P, 1e-6, ps, 2, 8, 2, 0, 2, 0, None) == E_CUDA
    assert L.qsa_raw_k_tail_write_prefill(0, P, P, ps, 2, 8, None) == E_CUDA
    assert L.qsa_indexer_pre_decode(0, P, P, P, P, P, P, 1e-6, ps, 2, None) == E_CUDA
    assert L.qsa_index_scores_decode(0, P, P, P, ps, 2, 64, None) == E_CUDA
    assert L.qsa_topk_expand_decode(P, P, P, None, -1, 2, 64, None) == E_CUDA   # no counters: heads unused
    assert L.qsa_indexer_decode_step(0, P, P, P, P, P, P, P, P, 1e-6, ps, P, 4, 4096, 65536, None) == E_CUDA
    assert L.qsa_index_q_prep(0, P, P, P, P, P, 1e-6, 1, 8, None) == E_CUDA
    assert L.qsa_index_scores(0, P, P, P, P, 1, 8, 2, 0, 8, None) == E_CUDA
    assert L.qsa_index_scores_no_alloc(0, P, P, P, P, 1, 8, 2, 0, 8, None) == E_CUDA
    assert L.qsa_index_scores_topk_expand(0, P, P, P, P, 2, 16, 4, 0, 32, None) == E_CUDA
    assert "cudaGetDevice" in qsa.qsa_last_error()
    flags = ctypes.c_uint32(0)
    assert L.qsa_device_fault_flags(ctypes.byref(flags), 1, None) == E_CUDA
    assert L.qsa_device_fault_flags(None, 1, None) == E_NULL
