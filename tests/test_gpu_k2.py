"""GPU parity of K2 (tcgen05 block scoring) against the CPU oracle.

Masks (-FLT_MAX cells, padded rows) must match bit for bit; visible logits within
the tolerance of tolerance.py ("Qsa Indexer Kernels", launchQsaIndexScores).
Every shape, the B=8, S=16384 scoring workload included, is compared with the
oracle element by element on every row; the oracle runs on all host cores for
the large workload.  The CUDA-core cross-check kernel is held to the same bar.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import workloads
from tolerance import check_logits, check_logits_torch, check_t, logits_floor

pytestmark = pytest.mark.gpu
NEG_MAX = np.float32(-np.finfo(np.float32).max)


def _gpu():
    import gpu_util
    return gpu_util


def _rand_inputs(dtype, B, S, NB, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    q = workloads.round_to_t(rng.standard_normal((B, S, 4, 128)) * scale, dtype)
    kb = workloads.round_to_t(rng.standard_normal((B, NB, 128)) * scale, dtype)
    return q, kb


def _compare(dtype, got, q, kb, ctx, row_start, num_rows):
    B, S = q.shape[:2]
    ref = oracle.scores(dtype, q, kb, ctx, row_start, num_rows)
    rows = np.arange(row_start, row_start + num_rows)
    b = rows // S
    fl = logits_floor(q.reshape(B * S, 4, 128)[rows], kb[b], dtype)
    ok, st = check_logits(got, ref, dtype, fl)
    print(f"K2 {dtype} B={B} S={S} NB={kb.shape[1]} rows=[{row_start},+{num_rows}): {st}")
    assert ok, st


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("B,S,NB,ctx", [
    (1, 64, 16, [50]),            # tiny
    (2, 1000, 250, [1000, 377]),  # ragged: S % 64 != 0, NB % 128 != 0
    (1, 777, 300, [700]),         # NB > ceilDiv(S, 4): extra masked columns
    (3, 130, 33, [130, 0, 1]),    # empty and one-token sequences
    (1, 4, 1, [4]),
    (2, 2048, 512, [2048, 1500]), # several g-tiles and token tiles
])
@pytest.mark.parametrize("impl", ["tcgen05", "cuda_core"])
def test_scores_match_oracle(impl, dtype, B, S, NB, ctx):
    """The tensor-core K2 and the CUDA-core cross-check kernel, each against the oracle."""
    g_ = _gpu()
    q, kb = _rand_inputs(dtype, B, S, NB, seed=S + NB)
    ctx = np.asarray(ctx, np.int32)
    qd, kd, cd = g_.dev(q), g_.dev(kb), g_.dev(ctx)
    got = g_.scores(dtype, qd, kd, cd, B, S, NB, 0, B * S, cuda_core=impl == "cuda_core")
    _compare(dtype, got, q, kb, ctx, 0, B * S)
    g_.assert_no_device_faults()


def test_chunks_equal_one_shot_bitwise():
    g_ = _gpu()
    dtype = "bf16"
    B, S, NB = 3, 700, 175
    q, kb = _rand_inputs(dtype, B, S, NB, seed=5)
    ctx = np.array([700, 333, 699], np.int32)
    qd, kd, cd = g_.dev(q), g_.dev(kb), g_.dev(ctx)
    full = g_.scores(dtype, qd, kd, cd, B, S, NB, 0, B * S)
    _compare(dtype, full, q, kb, ctx, 0, B * S)
    for start, n in ((0, 1), (1, 63), (37, 700), (699, 2), (700, 700), (1337, 763), (2099, 1)):
        part = g_.scores(dtype, qd, kd, cd, B, S, NB, start, n)
        assert np.array_equal(part.view(np.uint32), full[start:start + n].view(np.uint32)), (start, n)
    again = g_.scores(dtype, qd, kd, cd, B, S, NB, 0, B * S)
    assert np.array_equal(again.view(np.uint32), full.view(np.uint32)), "not deterministic"
    g_.assert_no_device_faults()


def test_nan_in_unread_rows_is_harmless():
    g_ = _gpu()
    dtype = "bf16"
    B, S, NB = 2, 300, 80
    q, kb = _rand_inputs(dtype, B, S, NB, seed=9)
    ctx = np.array([250, 0], np.int32)
    clean = g_.scores(dtype, g_.dev(q), g_.dev(kb), g_.dev(ctx), B, S, NB, 0, B * S)
    qn, kn = q.copy(), kb.copy()
    qn[0, 250:] = workloads.NAN_BITS[dtype]
    qn[1] = workloads.NAN_BITS[dtype]
    kn[0, 250 // 4:] = workloads.NAN_BITS[dtype]
    kn[1] = workloads.NAN_BITS[dtype]
    dirty = g_.scores(dtype, g_.dev(qn), g_.dev(kn), g_.dev(ctx), B, S, NB, 0, B * S)
    assert np.array_equal(dirty.view(np.uint32), clean.view(np.uint32))


@pytest.fixture(scope="module")
def scoring_pipeline():
    """B=8, S=16384: indexQk ~ N(0,1) -> GPU K1a/K1b -> qNormed, kbar (as the
    scoring workload specifies), for ctx = S and for ctx ~ U{1..S}."""
    import sparse_attention_indexer_qsa_gb300 as qsa
    g_ = _gpu()
    out = {}
    for full in (True, False):
        wl = workloads.scoring("bf16", full_context=full)
        d = g_.DevWorkload(wl)
        B, S, NB = wl.B, wl.S, wl.num_blocks
        qn = torch.empty((B, S, 4, 128), dtype=torch.bfloat16, device="cuda")
        kb = torch.empty((B, NB, 128), dtype=torch.bfloat16, device="cuda")
        qsa.qsa_index_q_prep(qn, d.index_qk, d.cos_sin, d.ctx, d.w_q, wl.eps, B, S)
        qsa.qsa_index_k_compress(kb, d.index_qk, d.cos_sin, d.ctx, d.w_k, wl.eps, B, S, NB, 0, NB, 0)
        out[full] = (wl, d, qn, kb)
    return out


def _host_threads():
    return max(1, len(os.sched_getaffinity(0)))


def _oracle_scores_threaded(pool, q_host, kb_host, ctx, row_lo, n_rows, piece=256):
    """oracle.scores over global rows [row_lo, row_lo + n_rows), in pieces spread over
    host threads (each C call releases the GIL; the pieces write disjoint rows)."""
    out = np.empty((n_rows, kb_host.shape[1]), np.float32)

    def work(a):
        n = min(piece, n_rows - a)
        out[a:a + n] = oracle.scores("bf16", q_host, kb_host, ctx, row_lo + a, n)

    list(pool.map(work, range(0, n_rows, piece)))
    return out


@pytest.mark.parametrize("full", [True, False])
def test_scoring_workload_every_row_against_oracle(scoring_pipeline, full):
    """B=8, S=16384: all 131072 x 4096 logits against the oracle, element by element
    (masks bit-exact, values within the logits tolerance), one sequence at a time."""
    import sparse_attention_indexer_qsa_gb300 as qsa
    wl, d, qn, kb = scoring_pipeline[full]
    B, S, NB = wl.B, wl.S, wl.num_blocks
    rows = B * S
    logits = torch.empty((rows, NB), dtype=torch.float32, device="cuda")
    qsa.qsa_index_scores(logits, qn, kb, d.ctx, B, S, NB, 0, rows)
    torch.cuda.synchronize()
    assert qsa.qsa_device_fault_flags() == 0
    q_host = qn.view(torch.int16).cpu().numpy().view(np.uint16)
    kb_host = kb.view(torch.int16).cpu().numpy().view(np.uint16)
    ctx = wl.context_lengths
    worst, n_vis = 0.0, 0
    with ThreadPoolExecutor(_host_threads()) as pool:
        for b in range(B):
            ref = torch.from_numpy(_oracle_scores_threaded(pool, q_host, kb_host, ctx, b * S, S)).cuda()
            qa = qn[b].double().abs().sum(1)                         # [S, 128]
            fl = (qa @ kb[b].double().abs().T) * (2.0 ** -16) / np.sqrt(128.0)
            ok, st = check_logits_torch(logits[b * S:(b + 1) * S], ref, "bf16", fl)
            assert ok, (b, st)
            worst = max(worst, st["max_err_over_tol"])
            n_vis += st["visible"]
            del ref, fl
    # the visible-count structure in closed form: row t shows min(NB, (t+1)//4) blocks iff t < ctx_b
    t = torch.arange(S, device="cuda")
    masked = logits.view(B, S, NB) == float(NEG_MAX)
    nvis = torch.where(t[None, :] < d.ctx[:, None].long(), torch.clamp((t + 1) // 4, max=NB)[None, :],
                       torch.zeros_like(t)[None, :])
    assert torch.equal((~masked).sum(-1), nvis), "visible-count structure differs"
    print(f"K2 scoring full={full}: {rows} rows, {n_vis} visible logits, "
          f"max |gpu - oracle| / tolerance = {worst:.3e}")
    del logits, masked
    torch.cuda.empty_cache()


def test_scoring_workload_k1_against_oracle(scoring_pipeline):
    """The qNormed and kbar the scoring workload is built from (GPU K1a / K1b of the
    padded variant) against the oracle's K1a / K1b, one sequence a thread."""
    wl, d, qn, kb = scoring_pipeline[False]
    B, S, NB = wl.B, wl.S, wl.num_blocks
    q_host = qn.view(torch.int16).cpu().numpy().view(np.uint16)
    kb_host = kb.view(torch.int16).cpu().numpy().view(np.uint16)

    def one(b):
        iq = np.ascontiguousarray(wl.index_qk[b:b + 1])
        c = wl.context_lengths[b:b + 1]
        rq = oracle.q_prep("bf16", iq, wl.cos_sin, c, wl.w_q, wl.eps)[0]
        rk = oracle.k_compress("bf16", iq, wl.cos_sin, c, wl.w_k, wl.eps, NB, 0, NB, 0)[0]
        vis_t = np.arange(S) < int(c[0])
        vis_g = np.array([oracle.block_valid(g, int(c[0]), S, 0) for g in range(NB)])
        assert not q_host[b][~vis_t].any() and not kb_host[b][~vis_g].any(), b
        ok_q, st_q = check_t(q_host[b][vis_t], rq[vis_t], "bf16")
        ok_k, st_k = check_t(kb_host[b][vis_g], rk[vis_g], "bf16")
        return b, ok_q and ok_k, st_q, st_k

    with ThreadPoolExecutor(min(B, _host_threads())) as pool:
        for b, ok, st_q, st_k in pool.map(one, range(B)):
            assert ok, (b, st_q, st_k)


def test_scoring_workload_chunked_equals_one_shot(scoring_pipeline):
    import sparse_attention_indexer_qsa_gb300 as qsa
    wl, d, qn, kb = scoring_pipeline[False]
    B, S, NB = wl.B, wl.S, wl.num_blocks
    rows = B * S
    one = torch.empty((rows, NB), dtype=torch.float32, device="cuda")
    qsa.qsa_index_scores(one, qn, kb, d.ctx, B, S, NB, 0, rows)
    chunk = 8192
    part = torch.empty((chunk, NB), dtype=torch.float32, device="cuda")
    for start in range(0, rows, chunk * 5):       # every fifth 8192-row chunk
        qsa.qsa_index_scores(part, qn, kb, d.ctx, B, S, NB, start, chunk)
        torch.cuda.synchronize()
        assert torch.equal(part.view(torch.int32), one[start:start + chunk].view(torch.int32)), start
    assert qsa.qsa_device_fault_flags() == 0
