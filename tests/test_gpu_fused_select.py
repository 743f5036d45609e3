"""GPU parity of qsa_index_scores_topk_expand: prefill scoring fused with the top-512
selection + expand ("Qsa Indexer Kernels": launchQsaIndexScores, then the selection
between launchQsaIndexIdsFill and launchQsaIndexExpand), which never writes the logits.

Index work, so the bar is bit-exact: for the same arguments the fused entry point
must write exactly the outIdx of qsa_index_scores into a logits buffer followed by
qsa_index_topk_expand on it (itself held to the oracle in test_gpu_select.py), and
exactly the oracle's selection on those logits.  Covered: the B=8, S=16384 scoring
workload in both context settings, row chunks, ragged and padded shapes, extra
masked columns, both dtypes, and inputs built to defeat the first-pass bins: every
logit +0 (one tie class), a few distinct kbar rows repeated (wide tie classes that
need the refinement passes), and q scaled far above and below the bins' range.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
W = oracle.INDEX_WIDTH
SENT = -7


def _qsa():
    import sparse_attention_indexer_qsa_gb300 as qsa
    return qsa


def _gu():
    import gpu_util
    return gpu_util


def _two_calls(dtype, qd, kd, cd, B, S, NB, row_start, n):
    """qsa_index_scores into a logits buffer, then qsa_index_topk_expand on it."""
    qsa = _qsa()
    logits = torch.empty((max(n, 1), NB), dtype=torch.float32, device="cuda")
    out = torch.full((B * S, W), SENT, dtype=torch.int32, device="cuda")
    qsa.qsa_index_scores(logits, qd, kd, cd, B, S, NB, row_start, n, dtype=dtype)
    qsa.qsa_index_topk_expand(out, logits, cd, B, S, NB, row_start, n)
    return out, logits


def _fused(dtype, qd, kd, cd, B, S, NB, row_start, n):
    qsa, g_ = _qsa(), _gu()
    out = g_.Guarded(B * S * W * 4, init=np.full((B * S, W), SENT, np.int32))
    qsa.qsa_index_scores_topk_expand(out.ptr, qd, kd, cd, B, S, NB, row_start, n, dtype=dtype)
    res = out.numpy(np.int32, (B * S, W))          # also checks the red zones
    assert qsa.qsa_device_fault_flags(clear=True) == 0
    return res


def _check_equal(dtype, q, kb, ctx, row_start=0, n=None, q_dev=None, kb_dev=None):
    g_ = _gu()
    B, S = q.shape[:2]
    NB = kb.shape[1]
    n = B * S - row_start if n is None else n
    qd = g_.dev(q, g_.t_dtype(dtype)) if q_dev is None else q_dev
    kd = g_.dev(kb, g_.t_dtype(dtype)) if kb_dev is None else kb_dev
    cd = g_.dev(np.asarray(ctx, np.int32))
    ref, _ = _two_calls(dtype, qd, kd, cd, B, S, NB, row_start, n)
    got = _fused(dtype, qd, kd, cd, B, S, NB, row_start, n)
    ref = ref.cpu().numpy()
    bad = np.nonzero((got != ref).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first {bad[:8].tolist()}"
    outside = np.ones(B * S, bool)
    outside[row_start:row_start + n] = False
    assert np.all(got[outside] == SENT), "rows outside the chunk were written"
    return got


def _rand(dtype, B, S, NB, seed, q_scale=1.0):
    rng = np.random.default_rng(seed)
    q = workloads.round_to_t(rng.standard_normal((B, S, 4, 128)) * q_scale, dtype)
    kb = workloads.round_to_t(rng.standard_normal((B, NB, 128)), dtype)
    return q, kb


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("B,S,NB,ctx", [
    (1, 64, 16, [50]),                 # no row has more than 512 visible blocks
    (2, 3000, 750, [3000, 2101]),      # selection rows, ragged tile at the end
    (1, 2600, 700, [2600]),            # numBlocks > ceilDiv(seqLen, 4): masked columns
    (3, 2200, 550, [2200, 0, 2053]),   # an empty sequence, rows just past 512 blocks
    (1, 16384, 4096, [16384]),         # the longest rows the fused kernel takes
])
def test_fused_equals_two_calls(dtype, B, S, NB, ctx):
    q, kb = _rand(dtype, B, S, NB, seed=S + NB)
    _check_equal(dtype, q, kb, ctx)


def test_fused_chunks():
    dtype = "bf16"
    B, S, NB = 2, 4100, 1025
    q, kb = _rand(dtype, B, S, NB, seed=3)
    ctx = np.array([4100, 3001], np.int32)
    g_ = _gu()
    qd, kd = g_.dev(q, torch.bfloat16), g_.dev(kb, torch.bfloat16)
    for start, n in ((0, 1), (2047, 3), (2100, 700), (4099, 2), (4100, 4100), (5000, 3200), (8199, 1)):
        _check_equal(dtype, q, kb, ctx, start, n, q_dev=qd, kb_dev=kd)


@pytest.mark.parametrize("case", ["all_zero_kbar", "repeated_kbar", "q_large", "q_tiny", "negative_q"])
def test_fused_ties_and_refinement(case):
    """Inputs whose keys crowd one first-pass bin: exact ties (every logit +0, or a few
    repeated kbar rows) and values far outside the bins' range (clamped end bins)."""
    dtype = "bf16"
    B, S, NB = 1, 6000, 1500
    q, kb = _rand(dtype, B, S, NB, seed=11)
    ctx = [6000]
    if case == "all_zero_kbar":
        kb[:] = 0
    elif case == "repeated_kbar":
        kb[0] = kb[0, np.arange(NB) % 7]
    elif case == "q_large":
        q, _ = _rand(dtype, B, S, NB, seed=11, q_scale=2.0 ** 12)
    elif case == "q_tiny":
        q, _ = _rand(dtype, B, S, NB, seed=11, q_scale=2.0 ** -12)
    elif case == "negative_q":
        # every dot of heads 1-3 negative against a positive kbar: many exact +0 logits
        kb = workloads.round_to_t(np.abs(np.random.default_rng(5).standard_normal((B, NB, 128))), dtype)
        qf = np.random.default_rng(6).standard_normal((B, S, 4, 128))
        qf[:, :, 1:] = -np.abs(qf[:, :, 1:])
        q = workloads.round_to_t(qf, dtype)
    _check_equal(dtype, q, kb, ctx)


def test_fused_never_reads_padded_rows_and_is_deterministic():
    dtype = "bf16"
    B, S, NB = 2, 2600, 650
    q, kb = _rand(dtype, B, S, NB, seed=21)
    ctx = np.array([2300, 2600], np.int32)
    g_ = _gu()
    qd, kd, cd = g_.dev(q, torch.bfloat16), g_.dev(kb, torch.bfloat16), g_.dev(ctx)
    clean = _fused(dtype, qd, kd, cd, B, S, NB, 0, B * S)
    qn, kn = q.copy(), kb.copy()
    qn[0, 2300:] = workloads.NAN_BITS[dtype]
    kn[0, 2300 // 4:] = workloads.NAN_BITS[dtype]
    dirty = _fused(dtype, g_.dev(qn, torch.bfloat16), g_.dev(kn, torch.bfloat16), cd, B, S, NB, 0, B * S)
    assert np.array_equal(dirty, clean)
    again = _fused(dtype, qd, kd, cd, B, S, NB, 0, B * S)
    assert np.array_equal(again, clean)


@pytest.fixture(scope="module")
def scoring_inputs():
    """B=8, S=16384: qNormed and kbar from the GPU K1a/K1b of the scoring workload."""
    qsa, g_ = _qsa(), _gu()
    out = {}
    for full in (True, False):
        wl = workloads.scoring("bf16", full_context=full)
        d = g_.DevWorkload(wl)
        B, S, NB = wl.B, wl.S, wl.num_blocks
        qn = torch.empty((B, S, 4, 128), dtype=torch.bfloat16, device="cuda")
        kb = torch.empty((B, NB, 128), dtype=torch.bfloat16, device="cuda")
        qsa.qsa_index_qk_prep(qn, kb, d.index_qk, d.cos_sin, d.ctx, d.w_q, d.w_k, wl.eps, B, S, NB)
        out[full] = (wl, d, qn, kb)
    return out


@pytest.mark.parametrize("full", [True, False])
def test_scoring_workload_fused_equals_two_calls_and_oracle(scoring_inputs, full):
    """Every row of the B=8, S=16384 workload: the fused outIdx equals the two calls' and
    the oracle's selection (stable descending sort + expand, as a block set) on the
    same logits."""
    qsa = _qsa()
    wl, d, qn, kb = scoring_inputs[full]
    B, S, NB = wl.B, wl.S, wl.num_blocks
    rows = B * S
    ref, logits = _two_calls("bf16", qn, kb, d.ctx, B, S, NB, 0, rows)
    got = torch.full((rows, W), SENT, dtype=torch.int32, device="cuda")
    qsa.qsa_index_scores_topk_expand(got, qn, kb, d.ctx, B, S, NB, 0, rows)
    torch.cuda.synchronize()
    assert qsa.qsa_device_fault_flags(clear=True) == 0
    diff = (got != ref).any(dim=1)
    assert not bool(diff.any()), f"{int(diff.sum())} rows differ from the two calls"
    # the oracle's selection on the same logits (a stable descending sort of each row,
    # then expand), compared as block sets: the kernels emit them in ascending order
    got_h = got.cpu().numpy()
    lg = logits.cpu().numpy()
    ctx = wl.context_lengths
    t_all = np.tile(np.arange(S), B)
    b_all = np.repeat(np.arange(B), S)
    unpadded = t_all < ctx[b_all]
    n_vis = np.where(unpadded, np.minimum((t_all + 1) // 4, NB), 0)
    n_all = np.where(unpadded, 4 * n_vis + (t_all + 1) % 4, 0)
    # rows with at most 512 visible blocks: every block, then the tail, then -1
    short = np.nonzero(n_vis <= 512)[0]
    k = np.arange(W)[None, :]
    want = np.where(k < n_all[short][:, None], k, -1)
    assert np.array_equal(got_h[short], want), "a row without selection differs"
    sel_rows = np.nonzero(n_vis > 512)[0]

    def piece(lo):
        rs = sel_rows[lo:lo + 1024]
        ora = np.stack([oracle.select_expand_row(lg[r], int(t_all[r]), int(ctx[b_all[r]])) for r in rs])
        g = got_h[rs]
        ob = np.sort(ora[:, :2048:4] // 4, axis=1)
        gb = g[:, :2048:4] // 4
        assert np.array_equal(gb, ob), "selected block sets differ from the oracle's"
        assert np.all(np.diff(gb, axis=1) > 0)
        assert np.array_equal(g[:, :2048].reshape(-1, 512, 4), gb[:, :, None] * 4 + np.arange(4))
        assert np.array_equal(g[:, 2048:], ora[:, 2048:]), "causal tail differs"
        return len(rs)

    with ThreadPoolExecutor(max(1, len(os.sched_getaffinity(0)))) as pool:
        assert sum(pool.map(piece, range(0, len(sel_rows), 1024))) == len(sel_rows)
    del logits, ref, got
    torch.cuda.empty_cache()
