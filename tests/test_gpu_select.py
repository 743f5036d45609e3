"""GPU parity of the prefill selection ("Qsa Indexer Kernels": launchQsaIndexIdsFill,
launchQsaIndexExpand, and the stable descending segmented sort between them).

Index work, so everything is exact: qsa_index_ids_fill and qsa_index_expand are
bit-identical to the oracle.  qsa_index_topk_expand selects exactly the blocks the
page's three-step pipeline puts first (the oracle's sort-based selection on the
same logits, and the pipeline run on the GPU: ids fill, a stable descending sort,
expand); the page calls the emitted token ids "unsorted", and the kernel emits
the selected blocks in ascending order as the page's decode top-k does, so the
comparison is: same block set, ascending order, identical tail and -1 padding.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
W = oracle.INDEX_WIDTH
NEG_MAX = float(-np.finfo(np.float32).max)
SENT = -7


def _qsa():
    import sparse_attention_indexer_qsa_gb300 as qsa
    return qsa


def _gu():
    import gpu_util
    return gpu_util


def test_ids_fill_matches_oracle():
    qsa, g_ = _qsa(), _gu()
    for rows, nb in ((1, 1), (3, 7), (1000, 250), (5, 4096)):
        out = g_.Guarded(rows * nb * 4, fill=0xEE)
        qsa.qsa_index_ids_fill(out.ptr, rows, nb)
        assert np.array_equal(out.numpy(np.int32, (rows, nb)), oracle.ids_fill(rows, nb))


def _logits_like_k2(B, S, NB, ctx, seed, levels=None):
    """Synthetic chunk logits with the K2 mask structure; `levels` draws values from
    a small set (heavy ties), else continuous values."""
    rng = np.random.default_rng(seed)
    if levels is None:
        v = rng.gamma(2.0, 1.0, (B * S, NB)).astype(np.float32)
    else:
        v = rng.choice(np.asarray(levels, np.float32), (B * S, NB))
    t = np.tile(np.arange(S), B)
    b = np.repeat(np.arange(B), S)
    vis = (np.arange(NB)[None, :] < ((t + 1) // 4)[:, None]) & (t < np.asarray(ctx)[b])[:, None]
    return np.where(vis, v, np.float32(NEG_MAX)).astype(np.float32)


def assert_same_selection(got, ref, rows=None):
    """got: topk_expand rows (ascending blocks); ref: sorted-pipeline rows (oracle or GPU)."""
    got = np.asarray(got)
    ref = np.asarray(ref)
    for r in (range(got.shape[0]) if rows is None else rows):
        g, f = got[r], ref[r]
        n = int((f >= 0).sum())
        assert int((g >= 0).sum()) == n, r
        assert np.all(g[n:] == -1) and np.all(f[n:] == -1), r
        tail = n % 4 if n < 2048 else n - 2048
        k = n - tail
        assert np.array_equal(g[k:n], f[k:n]), r                       # causal tail
        gb, fb = g[:k:4] // 4, f[:k:4] // 4
        assert np.array_equal(g[:k].reshape(-1, 4), gb[:, None] * 4 + np.arange(4)), r
        assert np.all(np.diff(gb) > 0), r                                # ascending blocks
        assert np.array_equal(gb, np.sort(fb)), r                        # the same block set


def _run_topk(logits_rows, ctx, B, S, NB, row_start):
    qsa, g_ = _qsa(), _gu()
    n = logits_rows.shape[0]
    out = g_.Guarded(B * S * W * 4, init=np.full((B * S, W), SENT, np.int32))
    qsa.qsa_index_topk_expand(out.ptr, g_.dev(logits_rows), g_.dev(np.asarray(ctx, np.int32)), B, S, NB,
                              row_start, n)
    return out.numpy(np.int32, (B * S, W))


@pytest.mark.parametrize("case", ["continuous", "ties", "zeros"])
def test_topk_expand_matches_oracle(case):
    B, S, NB = 2, 2900, 760            # nVis up to 725: both sides of 512, ragged sizes
    ctx = [2900, 1777]
    levels = {"continuous": None, "ties": [0.0, 0.5, 1.0, 2.0], "zeros": [0.0, -0.0, 1.0]}[case]
    lg = _logits_like_k2(B, S, NB, ctx, seed=len(case), levels=levels)
    got = _run_topk(lg, ctx, B, S, NB, 0)
    ref = oracle.select_expand(lg, ctx, B, S, 0)
    assert_same_selection(got, ref)


def test_topk_expand_chunks_and_untouched_rows():
    B, S, NB = 3, 700, 175
    ctx = [700, 0, 333]
    lg = _logits_like_k2(B, S, NB, ctx, seed=3)
    for start, n in ((0, 1), (37, 700), (699, 2), (1399, 701)):
        got = _run_topk(lg[start:start + n], ctx, B, S, NB, start)
        ref = oracle.select_expand(lg[start:start + n], ctx, B, S, start,
                                   out_idx=np.full((B * S, W), SENT, np.int32))
        outside = np.ones(B * S, bool)
        outside[start:start + n] = False
        assert np.all(got[outside] == SENT), (start, n)                  # untouched rows
        assert_same_selection(got, ref, rows=range(start, start + n))


def test_expand_matches_oracle_and_page_pipeline_matches_topk():
    """ids fill -> stable descending sort (torch) -> qsa_index_expand selects the same
    blocks as the fused qsa_index_topk_expand, and expand equals the oracle's expand."""
    qsa, g_ = _qsa(), _gu()
    B, S, NB = 2, 2400, 600
    ctx = [2400, 1999]
    lg = _logits_like_k2(B, S, NB, ctx, seed=11, levels=[0.0, 0.25, 0.5, 3.0])
    rows = B * S
    d_lg = g_.dev(lg)
    d_ctx = g_.dev(np.asarray(ctx, np.int32))
    ids = torch.empty((rows, NB), dtype=torch.int32, device="cuda")
    qsa.qsa_index_ids_fill(ids, rows, NB)
    bits = d_lg.view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    u = torch.where(bits >= 2**31, (~bits) & 0xFFFFFFFF, bits | 2**31)   # order-preserving map
    order = torch.sort(u, dim=1, descending=True, stable=True).indices
    sorted_ids = torch.gather(ids, 1, order.to(torch.int64)).to(torch.int32).contiguous()
    out_pipe = torch.full((rows, W), SENT, dtype=torch.int32, device="cuda")
    qsa.qsa_index_expand(out_pipe, sorted_ids, d_ctx, B, S, NB, 0, rows)
    out_fused = torch.full((rows, W), SENT, dtype=torch.int32, device="cuda")
    qsa.qsa_index_topk_expand(out_fused, d_lg, d_ctx, B, S, NB, 0, rows)
    torch.cuda.synchronize()
    assert_same_selection(out_fused.cpu().numpy(), out_pipe.cpu().numpy())
    si = sorted_ids.cpu().numpy()
    pipe = out_pipe.cpu().numpy()
    rng = np.random.default_rng(5)
    for r in rng.integers(0, rows, 200).tolist() + [0, 1, 2, 3, rows - 1]:
        b, t = divmod(r, S)
        assert np.array_equal(pipe[r], oracle.expand_row(si[r], t, ctx[b])), r


def test_topk_expand_on_scoring_workload():
    """B=8, S=16384: GPU K1 -> K2 logits -> selection; sampled rows bit-exact against
    the oracle on the same logits, structure checked on every row."""
    qsa, g_ = _qsa(), _gu()
    wl = workloads.scoring("bf16", full_context=False)
    d = g_.DevWorkload(wl)
    B, S, NB = wl.B, wl.S, wl.num_blocks
    rows = B * S
    qn = torch.empty((B, S, 4, 128), dtype=torch.bfloat16, device="cuda")
    kb = torch.empty((B, NB, 128), dtype=torch.bfloat16, device="cuda")
    qsa.qsa_index_qk_prep(qn, kb, d.index_qk, d.cos_sin, d.ctx, d.w_q, d.w_k, wl.eps, B, S, NB)
    logits = torch.empty((rows, NB), dtype=torch.float32, device="cuda")
    qsa.qsa_index_scores(logits, qn, kb, d.ctx, B, S, NB, 0, rows)
    out = torch.empty((rows, W), dtype=torch.int32, device="cuda")
    qsa.qsa_index_topk_expand(out, logits, d.ctx, B, S, NB, 0, rows)
    torch.cuda.synchronize()
    ctx = wl.context_lengths
    rng = np.random.default_rng(7)
    picks = set(rng.integers(0, rows, 64).tolist())
    for b in (0, B - 1):
        for t in (0, 1, 3, 4, 2047, 2048, 2051, 4095, S - 1, int(ctx[b]) - 1, int(ctx[b])):
            if 0 <= t < S:
                picks.add(b * S + t)
    picks = sorted(picks)
    got = out[picks].cpu().numpy()
    lg = logits[picks].cpu().numpy()
    ref = np.stack([oracle.select_expand_row(lg[i], r % S, int(ctx[r // S])) for i, r in enumerate(picks)])
    assert_same_selection(got, ref)
    # structure on every row: 4*kSel + tail entries, then -1; entries within [0, t]
    t = torch.arange(S, device="cuda").repeat(B)
    bb = torch.arange(B, device="cuda").repeat_interleave(S)
    valid = t < d.ctx.long()[bb]
    nvis = (t + 1) // 4
    want = torch.where(valid, 4 * torch.clamp(nvis, max=512) + (t + 1) % 4, torch.zeros_like(t))
    used = (out >= 0).sum(1)
    assert torch.equal(used, want)
    pos = torch.arange(W, device="cuda")[None, :]
    assert torch.equal(out >= 0, pos < want[:, None])
    assert bool((out.max(1).values <= t).all())
    assert qsa.qsa_device_fault_flags() == 0


def _rows_of(kind, n, NB, seed):
    rng = np.random.default_rng(seed)
    if kind == "normal":                       # both signs: no common leading key bits
        v = rng.standard_normal((n, NB)).astype(np.float32)
        v[:, ::97] = -0.0
        v[:, 1::89] = 0.0
    elif kind == "equal":                      # every key identical
        v = np.full((n, NB), 1.5, np.float32)
    elif kind == "narrow":                     # keys sharing most leading bits
        v = (1.0 + rng.integers(0, 64, (n, NB)) * np.float32(2.0 ** -20)).astype(np.float32)
    else:
        v = rng.gamma(2.0, 1.0, (n, NB)).astype(np.float32)
    return v


@pytest.mark.parametrize("NB", [3001, 4096, 6000, 8192, 12007, 16384, 20000, 65536])
@pytest.mark.parametrize("kind", ["gamma", "normal", "equal", "narrow"])
def test_topk_expand_long_rows(NB, kind):
    """Rows up to the 65536-block limit: every mask width (4096 blocks per 32-bit word a
    thread), rows not 16-byte aligned, ragged nVis, keys of both signs, all-equal and
    narrow ranges (the threshold bin holding more candidates than its list)."""
    qsa, g_ = _qsa(), _gu()
    S = 4 * NB
    out = torch.full((S, W), SENT, dtype=torch.int32, device="cuda")
    d_ctx = g_.dev(np.array([S], np.int32))
    ts = sorted({min(x, S - 3) for x in (4 * 513 - 1, 4 * 4096 - 2, 4 * min(NB, 8192) + 1, 4 * NB - 1, S - 3,
                                         4 * (NB // 3) + 2)})
    for j, start in enumerate(ts):
        n = 3
        lg = _rows_of(kind, n, NB, seed=NB + j)
        for i in range(n):                                         # the K2 mask beyond nVis
            lg[i, min(NB, (start + i + 1) // 4):] = NEG_MAX
        qsa.qsa_index_topk_expand(out, g_.dev(lg), d_ctx, 1, S, NB, start, n)
        got = out[start:start + n].cpu().numpy()
        ref = np.stack([oracle.select_expand_row(lg[i], start + i, S) for i in range(n)])
        assert_same_selection(got, ref)
    assert qsa.qsa_device_fault_flags() == 0


@pytest.mark.parametrize("maxb", [700, 4100, 9000, 17000])
def test_topk_expand_decode_long_rows(maxb):
    """Decode top-k over long rows is bit-exact against the oracle (ascending emission)."""
    qsa, g_ = _qsa(), _gu()
    B = 5
    ctx = np.array([4 * maxb, 4 * maxb - 1, 2051, 0, 4 * (maxb // 2) + 3], np.int32)
    lg = _rows_of("normal", B, maxb, seed=maxb)
    lg[1, ::3] = lg[1, 5]                                           # heavy ties in one row
    out = g_.Guarded(B * W * 4, init=np.full((B, W), SENT, np.int32))
    split = torch.full((B, 3), 9, dtype=torch.int32, device="cuda")
    qsa.qsa_topk_expand_decode(out.ptr, g_.dev(lg), g_.dev(ctx), split, 3, B, maxb)
    assert np.array_equal(out.numpy(np.int32, (B, W)), oracle.topk_expand_decode(lg, ctx))
    assert not split.any()


def test_topk_expand_never_reads_masked_cells():
    """Logits at g >= nVis (K2's -FLT_MAX cells) replaced by NaN: the same output."""
    B, S, NB = 2, 3000, 750
    ctx = [3000, 2222]
    lg = _logits_like_k2(B, S, NB, ctx, seed=21)
    ref = _run_topk(lg, ctx, B, S, NB, 0)
    poisoned = lg.copy()
    poisoned[poisoned == np.float32(NEG_MAX)] = np.nan
    assert np.isnan(poisoned).any()
    assert np.array_equal(_run_topk(poisoned, ctx, B, S, NB, 0), ref)


def test_two_identical_runs_give_identical_out_idx():
    """Two identical runs of the prefill and decode selections give bitwise-identical
    outIdx ("Qsa Indexer Kernels", launchQsaTopKExpandDecode: determinism), with heavy
    ties, so that tie order is part of the check."""
    qsa, g_ = _qsa(), _gu()
    B, S, NB = 2, 3000, 760
    ctx = [3000, 2222]
    lg = _logits_like_k2(B, S, NB, ctx, seed=71, levels=[0.0, 0.25, 1.0, 3.0])
    a = _run_topk(lg, ctx, B, S, NB, 0)
    b = _run_topk(lg, ctx, B, S, NB, 0)
    assert np.array_equal(a, b)
    dl = torch.from_numpy(lg[S - 8:S + 8].copy()).cuda()           # 16 rows as a decode batch
    dctx = torch.full((16,), 4 * NB - 1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(2):
        o = torch.empty((16, W), dtype=torch.int32, device="cuda")
        qsa.qsa_topk_expand_decode(o, dl, dctx, None, 2, 16, NB)
        outs.append(o.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
