"""GPU parity of the paged persistence and decode path ("Qsa Indexer Kernels":
QsaIndexerPoolState, launchQsaIndexKCompressPaged, launchQsaRawKTailWritePrefill,
launchQsaIndexerPreDecode, launchQsaIndexScoresDecode, launchQsaTopKExpandDecode).

Bit-exact where the page demands it: the paged K1b's dense output equals the plain
K1b, pool writes land exactly where the addressing contract puts them, raw K tails
are bit copies, the decode block compression equals prefill K1b, decode q equals
prefill q at the same position, decode scores equal prefill K2's row of the same
token (both on the tensor cores, the same MMA along K), and the decode top-k equals
the oracle on the same logits.  Decode scores are also compared with the oracle
within the logits tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import pool_util
import workloads
from tolerance import check_logits, logits_floor

pytestmark = pytest.mark.gpu
NEG_MAX = np.float32(-np.finfo(np.float32).max)


def _qsa():
    import sparse_attention_indexer_qsa_gb300 as qsa
    return qsa


def _gu():
    import gpu_util
    return gpu_util


class DevPool:
    def __init__(self, host_pool):
        g_ = _gu()
        self.host = host_pool
        self.pool = g_.dev(host_pool.pool)
        self.table = g_.dev(host_pool.page_table)
        self.state = _qsa().pool_state(self.pool, self.table, host_pool.num_pages, host_pool.num_kv_heads,
                                       host_pool.pool_head_dim, host_pool.head_size)

    def numpy(self):
        torch.cuda.synchronize()
        return self.pool.cpu().numpy().view(np.uint16)


def _expected_v_tails(pool0, kbar, ctx, past_len, S, blocks):
    """Pool after a paged K1b: V-tails of valid blocks with usable slots hold kbar rows."""
    exp = oracle.Pool(pool0.pool.copy(), pool0.page_table, pool0.num_pages, pool0.num_kv_heads,
                      pool0.pool_head_dim, pool0.head_size)
    for b in range(kbar.shape[0]):
        for g in blocks:
            if oracle.block_valid(g, int(ctx[b]), S, past_len):
                tail = pool_util.v_tail(exp, b, g)
                if tail is not None:
                    tail[:] = kbar[b, g]
    return exp.pool


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_paged_compress_and_raw_tails(dtype):
    qsa, g_ = _qsa(), _gu()
    B, S = 3, 700
    wl = workloads.custom(B, S, [700, 513, 3], dtype=dtype, seed=21, nan_padding=True)
    d = g_.DevWorkload(wl)
    NB = wl.num_blocks
    host_pool = pool_util.make_pool(B, S, seed=5, unused_slots=((0, 1, 2), (1, 0, 1), (1, 1, 3)))
    dp = DevPool(host_pool)
    plain = g_.k_compress(d, NB, 0, NB, 0)
    kb = g_.Guarded(B * NB * 128 * 2, init=np.full((B, NB, 128), 0x1234, np.uint16))
    qsa.qsa_index_k_compress_paged(kb.ptr, d.index_qk, d.cos_sin, d.ctx, d.w_k, wl.eps, dp.state, B, S, NB, 0, NB,
                                   0, dtype=dtype)
    dense = kb.numpy(np.uint16, (B, NB, 128))
    assert np.array_equal(dense, plain), "paged dense output differs from K1b"
    assert np.array_equal(dp.numpy(), _expected_v_tails(host_pool, plain, wl.context_lengths, 0, S, range(NB)))
    # raw K tails of the trailing incomplete blocks: a bit copy, nowhere else
    before = dp.numpy().copy()
    qsa.qsa_raw_k_tail_write_prefill(d.index_qk, d.ctx, dp.state, B, S, dtype=dtype)
    ref = oracle.Pool(before.copy(), host_pool.page_table, host_pool.num_pages)
    oracle.raw_k_tail_write_prefill(wl.index_qk, wl.context_lengths, ref)
    assert np.array_equal(dp.numpy(), ref.pool)
    assert not np.array_equal(ref.pool, before)                        # something was written
    # a sub-range recompress with pastLen writes the same V-tails
    dp2 = DevPool(pool_util.make_pool(B, S, seed=5, unused_slots=((0, 1, 2), (1, 0, 1), (1, 1, 3))))
    P = 128
    sub = d.index_qk[:, P:].contiguous()
    kb2 = torch.zeros((B, NB, 128), dtype=torch.int16, device="cuda")
    for bB, bE in workloads.subrange_tiles(9, P, NB):
        qsa.qsa_index_k_compress_paged(kb2, sub, d.cos_sin, d.ctx, d.w_k, wl.eps, dp2.state, B, S - P, NB, bB, bE,
                                       P, dtype=dtype)
    blocks = [g for g in range(NB) if 4 * g >= P]
    exp = _expected_v_tails(dp2.host, plain, wl.context_lengths, P, S - P, blocks)
    assert np.array_equal(dp2.numpy(), exp)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_decode_loop_matches_oracle_and_prefill(dtype):
    """Prefill, then one token per step across nVis = 512 and a 128-token page edge."""
    qsa, g_ = _qsa(), _gu()
    B = 3
    total = [2100, 2060, 300]
    prefill = [2040, 2046, 250]
    S = max(total)
    wl = workloads.custom(B, S, total, dtype=dtype, seed=31, nan_padding=True, max_positions=S)
    d = g_.DevWorkload(wl)
    NB = (S + 3) // 4
    maxb = NB + 3
    host_pool = pool_util.make_pool(B, S, seed=8)
    dp = DevPool(host_pool)
    # prefill: paged K1b + raw tails of each sequence's first `prefill` tokens
    pctx = g_.dev(np.array(prefill, np.int32))
    kb = torch.empty((B, NB, 128), dtype=torch.int16, device="cuda")
    qsa.qsa_index_k_compress_paged(kb, d.index_qk, d.cos_sin, pctx, d.w_k, wl.eps, dp.state, B, S, NB, 0, NB, 0,
                                   dtype=dtype)
    qsa.qsa_raw_k_tail_write_prefill(d.index_qk, pctx, dp.state, B, S, dtype=dtype)
    # reference: the whole sequences through prefill K1a / K1b on the GPU
    full_q = g_.q_prep(d)
    full_k = g_.k_compress(d, NB, 0, NB, 0)
    # prefill K2 over the whole sequences: the decode scores of token t are its row t
    k2 = g_.scores(dtype, g_.dev(full_q), g_.dev(full_k), g_.dev(np.array(total, np.int32)), B, S, NB, 0, B * S)
    q = torch.empty((B, 1, 4, 128), dtype=torch.int16, device="cuda")
    logits = torch.full((B, maxb), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.empty((B, 2051), dtype=torch.int32, device="cuda")
    split = torch.full((B, 2), 7, dtype=torch.int32, device="cuda")
    for step in range(max(t - p for t, p in zip(total, prefill))):
        pos = [p + step for p in prefill]
        ctx = np.array([ps + 1 if ps < t else 0 for ps, t in zip(pos, total)], np.int32)
        rows = np.stack([wl.index_qk[b, min(pos[b], S - 1)] for b in range(B)])
        d_rows, d_ctx = g_.dev(rows), g_.dev(ctx)
        qsa.qsa_indexer_pre_decode(q, d_rows, d.cos_sin, d_ctx, d.w_q, d.w_k, wl.eps, dp.state, B, dtype=dtype)
        logits.fill_(float("nan"))
        qsa.qsa_index_scores_decode(logits, q, d_ctx, dp.state, B, maxb, dtype=dtype)
        qsa.qsa_topk_expand_decode(out, logits, d_ctx, split, 2, B, maxb)
        torch.cuda.synchronize()
        qh = q.cpu().numpy().view(np.uint16)
        lg = logits.cpu().numpy()
        oh = out.cpu().numpy()
        assert not split.any()
        split.fill_(7)
        pool_now = dp.numpy()
        ref_pool = oracle.Pool(pool_now, host_pool.page_table, host_pool.num_pages)
        for b in range(B):
            if ctx[b] <= 0:
                assert not qh[b].any() and np.all(oh[b] == -1)
                continue
            assert np.array_equal(qh[b, 0], full_q[b, pos[b]]), (step, b)   # decode q == prefill q
        # scores against the oracle on the GPU's q and pool
        ref = oracle.scores_decode(dtype, qh, ctx, ref_pool, maxb)
        for b in range(B):
            nv = int(ctx[b]) // 4
            assert np.all(np.isnan(lg[b, nv:])), (step, b)                 # only the valid prefix
            if nv:
                kb_b = np.stack([pool_util.v_tail(ref_pool, b, g) for g in range(nv)])
                fl = logits_floor(qh[b, 0][None], kb_b, dtype)
                ok, st = check_logits(lg[b, :nv][None], ref[b, :nv][None], dtype, fl)
                assert ok, (step, b, st)
                # the same MMA shape along K and the same K order as prefill K2: the same bits
                assert np.array_equal(lg[b, :nv].view(np.uint32), k2[b * S + pos[b], :nv].view(np.uint32)), (step, b)
        # top-k: bit-exact against the oracle on the same logits
        assert np.array_equal(oh, oracle.topk_expand_decode(lg, ctx)), step
        # and the prefill selection kernel picks the same blocks for the same logits
        for b in range(B):
            if ctx[b] <= 0:
                continue
            t = int(ctx[b]) - 1
            one = torch.full((S * 1, 2051), -5, dtype=torch.int32, device="cuda")
            row = torch.from_numpy(lg[b:b + 1, :NB].copy()).cuda()
            row[:, int(ctx[b]) // 4:] = float(NEG_MAX)
            qsa.qsa_index_topk_expand(one, row, g_.dev(np.array([S], np.int32)), 1, S, NB, t, 1)
            assert np.array_equal(one[t].cpu().numpy(), oh[b]), (step, b)
    # every block completed by prefill or decode holds the prefill K1b bits
    pool_end = oracle.Pool(dp.numpy(), host_pool.page_table, host_pool.num_pages)
    for b in range(B):
        for g in range(total[b] // 4):
            assert np.array_equal(pool_util.v_tail(pool_end, b, g), full_k[b, g]), (b, g)
        for t in range(total[b] - total[b] % 4, total[b]):
            assert np.array_equal(pool_util.k_tail(pool_end, b, t), wl.index_qk[b, t, 512:])
    assert qsa.qsa_device_fault_flags() == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("nkv,phd,hs,B,max_tokens", [(1, 128, 0, 40, 4100), (2, 384, 256, 6, 4100),
                                                     (4, 200, 72, 3, 2000)])
def test_paged_scores_layouts_and_unusable_slots(dtype, nkv, phd, hs, B, max_tokens):
    """qsa_index_scores_decode against the oracle on pools of several head layouts, with
    V page slots that are -1, point outside the pool or lie past maxPagesPerSeq (those
    blocks score -FLT_MAX), nVis from 0 to past the table, runs of several 128-block
    tiles (B=40) and partial tiles and pages."""
    qsa, g_ = _qsa(), _gu()
    rng = np.random.default_rng(90 + nkv)
    hp = pool_util.make_pool(B, max_tokens, seed=41 + nkv, num_kv_heads=nkv, pool_head_dim=phd, head_size=hs)
    hp.pool[...] = workloads.round_to_t(rng.standard_normal(hp.pool.shape), dtype).reshape(hp.pool.shape)
    max_pages = hp.page_table.shape[2]
    hp.page_table[0, 1, 3] = -1                               # a hole in sequence 0
    hp.page_table[1 % B, 1, 5] = 2 * hp.num_pages + 7         # outside the pool
    hp.page_table[2 % B, 1, 0] = -1                           # the first page
    maxb = max_pages * 32 + 40                                # the last 40 blocks lie past the table
    fixed = [4 * maxb, 0, 1, 3, 4, 5, 2047, 2048, 4 * 32 * max_pages + 3, 4 * 129 + 2]
    ctx = np.array([fixed[b] if b < len(fixed) else int(rng.integers(0, 4 * maxb + 1)) for b in range(B)], np.int32)
    q = workloads.round_to_t(rng.standard_normal((B, 1, 4, 128)), dtype).reshape(B, 1, 4, 128)
    dp = DevPool(hp)
    logits = torch.full((B, maxb), float("nan"), dtype=torch.float32, device="cuda")
    qsa.qsa_index_scores_decode(logits, g_.dev(q), g_.dev(ctx), dp.state, B, maxb, dtype=dtype)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    ref = oracle.scores_decode(dtype, q, ctx, hp, maxb)
    n_unusable = 0
    for b in range(B):
        nv = min(int(ctx[b]) // 4, maxb)
        assert np.all(np.isnan(lg[b, nv:])), b                       # only the valid prefix
        if nv == 0:
            continue
        tails = [pool_util.v_tail(hp, b, g) if (4 * g) // 128 < max_pages else None for g in range(nv)]
        unusable = np.array([t is None or not (0 <= hp.page_table[b, 1, (4 * g) // 128] < 2 * hp.num_pages)
                             for g, t in enumerate(tails)])
        n_unusable += int(unusable.sum())
        assert np.array_equal(ref[b, :nv] == NEG_MAX, unusable), b
        kb_b = np.stack([t if (t is not None and not u) else np.zeros(128, np.uint16)
                         for t, u in zip(tails, unusable)])
        fl = logits_floor(q[b, 0][None], kb_b, dtype)
        ok, st = check_logits(lg[b, :nv][None], ref[b, :nv][None], dtype, fl)
        assert ok, (b, st)
    assert n_unusable > 40
    assert qsa.qsa_device_fault_flags() == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_paged_scores_ignore_tails_past_nvis(dtype):
    """The paged scores copy a visible block's whole page: V-tails of blocks past nVis on
    that page (and every page after it) set to NaN change no visible score's bits."""
    qsa, g_ = _qsa(), _gu()
    B = 4
    ctx = np.array([1000, 517, 4 * 96 + 3, 130], np.int32)    # nVis 250, 129, 96, 32
    maxb = 260
    rng = np.random.default_rng(33)
    hp = pool_util.make_pool(B, 1100, seed=34)
    hp.pool[...] = workloads.round_to_t(rng.standard_normal(hp.pool.shape, dtype=np.float32),
                                        dtype).reshape(hp.pool.shape)
    q = workloads.round_to_t(rng.standard_normal((B, 1, 4, 128)), dtype).reshape(B, 1, 4, 128)

    def run(pool_h):
        logits = torch.full((B, maxb), float("nan"), dtype=torch.float32, device="cuda")
        qsa.qsa_index_scores_decode(logits, g_.dev(q), g_.dev(ctx), DevPool(pool_h).state, B, maxb, dtype=dtype)
        torch.cuda.synchronize()
        return logits.cpu().numpy()
    clean = run(hp)
    poisoned = oracle.Pool(hp.pool.copy(), hp.page_table, hp.num_pages)
    nan_bits = workloads.NAN_BITS[dtype]
    for b in range(B):
        for g in range(int(ctx[b]) // 4, (1100 + 3) // 4):
            tail = pool_util.v_tail(poisoned, b, g)
            if tail is not None:
                tail[:] = nan_bits
    dirty = run(poisoned)
    for b in range(B):
        nv = int(ctx[b]) // 4
        assert np.array_equal(clean[b, :nv].view(np.uint32), dirty[b, :nv].view(np.uint32)), b
        assert not np.isnan(dirty[b, :nv]).any(), b
        assert np.all(np.isnan(dirty[b, nv:])), b
    assert qsa.qsa_device_fault_flags() == 0


def test_bounded_wait_runs_out_reports_and_leaves_the_context_usable():
    """The decode engine's bounded wait, on an mbarrier nothing arrives on, gives up after
    its limit, sets its fault bit (read on the host, then cleared), and the next launches
    on the same context compute correct scores."""
    import time
    qsa, g_ = _qsa(), _gu()
    assert qsa.qsa_device_fault_flags(clear=True) == 0
    t0 = time.perf_counter()
    qsa.qsa_testing_bounded_wait_probe(200)
    flags = qsa.qsa_device_fault_flags(clear=True)
    assert time.perf_counter() - t0 >= 0.2
    assert flags == 4 << 16
    assert qsa.qsa_device_fault_flags() == 0
    # the context still works
    B, dtype = 2, "bf16"
    rng = np.random.default_rng(5)
    hp = pool_util.make_pool(B, 600, seed=6)
    hp.pool[...] = workloads.round_to_t(rng.standard_normal(hp.pool.shape, dtype=np.float32),
                                        dtype).reshape(hp.pool.shape)
    ctx = np.array([600, 517], np.int32)
    maxb = 152
    q = workloads.round_to_t(rng.standard_normal((B, 1, 4, 128)), dtype).reshape(B, 1, 4, 128)
    logits = torch.full((B, maxb), float("nan"), dtype=torch.float32, device="cuda")
    qsa.qsa_index_scores_decode(logits, g_.dev(q), g_.dev(ctx), DevPool(hp).state, B, maxb, dtype=dtype)
    lg = logits.cpu().numpy()
    ref = oracle.scores_decode(dtype, q, ctx, hp, maxb)
    for b in range(B):
        nv = int(ctx[b]) // 4
        kb_b = np.stack([pool_util.v_tail(hp, b, g) for g in range(nv)])
        ok, st = check_logits(lg[b, :nv][None], ref[b, :nv][None], dtype, logits_floor(q[b, 0][None], kb_b, dtype))
        assert ok, (b, st)
    assert qsa.qsa_device_fault_flags() == 0


def test_decode_validation_rejects_bad_pools():
    qsa = _qsa()
    P = 0x1000
    bad = qsa.PoolState(P, P, 4, 8, 2, 384, 300)           # headSize + 128 > poolHeadDim
    with pytest.raises(qsa.QsaError) as e:
        qsa.qsa_index_scores_decode(P, P, P, bad, 2, 16, stream=0, dtype="bf16")
    assert e.value.status == -2
    odd = qsa.PoolState(P, P, 4, 8, 2, 384, 250)            # tails not 16-byte aligned
    with pytest.raises(qsa.QsaError) as e:
        qsa.qsa_indexer_pre_decode(P, P, P, P, P, P, 1e-6, odd, 2, stream=0, dtype="bf16")
    assert e.value.status == -5
    null = qsa.PoolState(0, P, 4, 8, 2, 384, 256)
    with pytest.raises(qsa.QsaError) as e:
        qsa.qsa_raw_k_tail_write_prefill(P, P, null, 2, 8, stream=0, dtype="bf16")
    assert e.value.status == -1


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fused_decode_step_bit_identical_to_three_calls(dtype):
    """qsa_indexer_decode_step against qsa_indexer_pre_decode + qsa_index_scores_decode +
    qsa_topk_expand_decode on two copies of one prefilled pool, token by token: q, the
    logits prefix, outIdx, the split counters and both pools stay bit-identical.  One
    sequence has an unusable K page (its block compress is skipped), one runs past its
    length (ctx 0), and nVis crosses 512 and a 128-block CTA edge."""
    qsa, g_ = _qsa(), _gu()
    B = 4
    total = [2150, 2060, 700, 520]
    prefill = [2040, 2046, 640, 300]
    S = max(total)
    wl = workloads.custom(B, S, total, dtype=dtype, seed=71, nan_padding=True, max_positions=S)
    d = g_.DevWorkload(wl)
    NB = (S + 3) // 4
    maxb = NB + 7
    unused = ((2, 0, 5),)                           # sequence 2: K page of tokens 640..767 unusable
    pools = [DevPool(pool_util.make_pool(B, S, seed=12, unused_slots=unused)) for _ in range(2)]
    pctx = g_.dev(np.array(prefill, np.int32))
    kb = torch.empty((B, NB, 128), dtype=torch.int16, device="cuda")
    for dp in pools:
        qsa.qsa_index_k_compress_paged(kb, d.index_qk, d.cos_sin, pctx, d.w_k, wl.eps, dp.state, B, S, NB, 0, NB,
                                       0, dtype=dtype)
        qsa.qsa_raw_k_tail_write_prefill(d.index_qk, pctx, dp.state, B, S, dtype=dtype)

    def bufs():
        return dict(q=torch.empty((B, 1, 4, 128), dtype=torch.int16, device="cuda"),
                    logits=torch.full((B, maxb), float("nan"), device="cuda"),
                    out=torch.empty((B, 2051), dtype=torch.int32, device="cuda"),
                    split=torch.full((B, 3), 9, dtype=torch.int32, device="cuda"))
    three, fused = bufs(), bufs()
    for step in range(max(t - p for t, p in zip(total, prefill))):
        pos = [p + step for p in prefill]
        ctx = np.array([ps + 1 if ps < t else 0 for ps, t in zip(pos, total)], np.int32)
        rows = np.stack([wl.index_qk[b, min(pos[b], S - 1)] for b in range(B)])
        d_rows, d_ctx = g_.dev(rows), g_.dev(ctx)
        st0, st1 = pools[0].state, pools[1].state
        three["logits"].fill_(float("nan"))
        fused["logits"].fill_(float("nan"))
        qsa.qsa_indexer_pre_decode(three["q"], d_rows, d.cos_sin, d_ctx, d.w_q, d.w_k, wl.eps, st0, B, dtype=dtype)
        qsa.qsa_index_scores_decode(three["logits"], three["q"], d_ctx, st0, B, maxb, dtype=dtype)
        qsa.qsa_topk_expand_decode(three["out"], three["logits"], d_ctx, three["split"], 3, B, maxb)
        qsa.qsa_indexer_decode_step(fused["out"], fused["logits"], fused["q"], d_rows, d.cos_sin, d_ctx, d.w_q,
                                    d.w_k, wl.eps, st1, fused["split"], 3, B, maxb, dtype=dtype)
        torch.cuda.synchronize()
        for name in ("q", "out", "split"):
            assert torch.equal(three[name], fused[name]), (step, name)
        for b in range(B):
            nv = int(ctx[b]) // 4
            assert torch.equal(three["logits"][b, :nv].view(torch.int32), fused["logits"][b, :nv].view(torch.int32))
            assert torch.isnan(fused["logits"][b, nv:]).all(), (step, b)    # only the valid prefix
        assert not fused["split"].any()
        three["split"].fill_(9)
        fused["split"].fill_(9)
        if step % 16 == 0 or step in (53, 60, 61):
            assert np.array_equal(pools[0].numpy(), pools[1].numpy()), step
    assert np.array_equal(pools[0].numpy(), pools[1].numpy())
    assert qsa.qsa_device_fault_flags() == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fused_decode_step_long_rows(dtype):
    """The one-launch step against the three calls on rows of ~40000 visible blocks: the
    selection's widest mask path (8 words a thread at 256 threads; 16 at the separate
    top-k's 128), runs of many 128-block tiles and a block compress at a page edge.  The
    pool (one KV head, 128-dim rows, the V-tail the whole row) is filled with random T
    values directly."""
    qsa, g_ = _qsa(), _gu()
    B = 2
    ctx = np.array([4 * 40000, 4 * 39000 + 2], np.int32)   # a block completes / a K-tail is written
    maxb = 40005
    rng = np.random.default_rng(77)
    hp = pool_util.make_pool(B, int(ctx.max()) + 8, seed=13, num_kv_heads=1, pool_head_dim=128, head_size=0)
    hp.pool[...] = workloads.round_to_t(rng.standard_normal(hp.pool.shape, dtype=np.float32),
                                        dtype).reshape(hp.pool.shape)
    rows = workloads.round_to_t(rng.standard_normal((B, 640)), dtype).reshape(B, 640)
    cos_sin = g_.dev(workloads.cos_sin_table(int(ctx.max()) + 8))
    w_q = g_.dev(workloads.gamma(rng, dtype))
    w_k = g_.dev(workloads.gamma(rng, dtype))
    pools = [DevPool(hp) for _ in range(2)]
    d_rows, d_ctx = g_.dev(rows), g_.dev(ctx)

    def bufs():
        return dict(q=torch.empty((B, 1, 4, 128), dtype=torch.int16, device="cuda"),
                    logits=torch.full((B, maxb), float("nan"), device="cuda"),
                    out=torch.empty((B, 2051), dtype=torch.int32, device="cuda"),
                    split=torch.full((B, 3), 9, dtype=torch.int32, device="cuda"))
    three, fused = bufs(), bufs()
    st0, st1 = pools[0].state, pools[1].state
    qsa.qsa_indexer_pre_decode(three["q"], d_rows, cos_sin, d_ctx, w_q, w_k, 1e-6, st0, B, dtype=dtype)
    qsa.qsa_index_scores_decode(three["logits"], three["q"], d_ctx, st0, B, maxb, dtype=dtype)
    qsa.qsa_topk_expand_decode(three["out"], three["logits"], d_ctx, three["split"], 3, B, maxb)
    qsa.qsa_indexer_decode_step(fused["out"], fused["logits"], fused["q"], d_rows, cos_sin, d_ctx, w_q, w_k, 1e-6,
                                st1, fused["split"], 3, B, maxb, dtype=dtype)
    torch.cuda.synchronize()
    for name in ("q", "out", "split"):
        assert torch.equal(three[name], fused[name]), name
    for b in range(B):
        nv = int(ctx[b]) // 4
        assert torch.equal(three["logits"][b, :nv].view(torch.int32), fused["logits"][b, :nv].view(torch.int32)), b
        assert torch.isnan(fused["logits"][b, nv:]).all(), b
        assert not torch.isnan(fused["logits"][b, :nv]).any(), b
    assert not fused["split"].any()
    assert np.array_equal(pools[0].numpy(), pools[1].numpy())
    # the selection itself, against the oracle on the same logits
    assert np.array_equal(fused["out"].cpu().numpy(),
                          oracle.topk_expand_decode(fused["logits"].cpu().numpy(), ctx))
    assert qsa.qsa_device_fault_flags() == 0


def test_fused_decode_step_at_the_batch_limit():
    """4096 sequences (the largest batch of the one-launch step: its arrival-counter set)
    with contexts from 1 to 2400 tokens, every input drawn on the device: the one launch
    and the three separate calls give the same bits on every output and in the pool."""
    qsa = _qsa()
    B, max_ctx = 4096, 2400
    pages = (max_ctx + 127) // 128
    num_pages = B * pages
    gen = torch.Generator(device="cuda").manual_seed(17)
    pool0 = torch.randn((2 * num_pages, 128, 1, 128), device="cuda", generator=gen).to(torch.bfloat16)
    perm = torch.randperm(num_pages, device="cuda", generator=gen).to(torch.int32).view(B, pages)
    table = torch.stack([perm, torch.roll(perm, 1, 0) + num_pages], dim=1).contiguous()   # [B, 2, pages]
    ctx = torch.randint(1, max_ctx + 1, (B,), device="cuda", generator=gen, dtype=torch.int32)
    rows = torch.randn((B, 640), device="cuda", generator=gen).to(torch.bfloat16)
    cs = torch.randn((max_ctx, 64), device="cuda", generator=gen)
    wq = (torch.randn(128, device="cuda", generator=gen) * 0.1).to(torch.bfloat16)
    wk = (torch.randn(128, device="cuda", generator=gen) * 0.1).to(torch.bfloat16)
    maxb = (max_ctx + 3) // 4
    pools = [pool0.clone(), pool0.clone()]
    states = [qsa.pool_state(p_, table, num_pages, numKVHeads=1, poolHeadDim=128, headSize=0) for p_ in pools]

    def bufs():
        return dict(q=torch.empty((B, 1, 4, 128), dtype=torch.bfloat16, device="cuda"),
                    logits=torch.full((B, maxb), float("nan"), device="cuda"),
                    out=torch.empty((B, 2051), dtype=torch.int32, device="cuda"),
                    split=torch.full((B, 4), 3, dtype=torch.int32, device="cuda"))
    three, fused = bufs(), bufs()
    qsa.qsa_indexer_pre_decode(three["q"], rows, cs, ctx, wq, wk, 1e-6, states[0], B)
    qsa.qsa_index_scores_decode(three["logits"], three["q"], ctx, states[0], B, maxb)
    qsa.qsa_topk_expand_decode(three["out"], three["logits"], ctx, three["split"], 4, B, maxb)
    for _ in range(2):   # twice: the counters must be back at zero after the first launch
        fused["logits"].fill_(float("nan"))
        qsa.qsa_indexer_decode_step(fused["out"], fused["logits"], fused["q"], rows, cs, ctx, wq, wk, 1e-6,
                                    states[1], fused["split"], 4, B, maxb)
        torch.cuda.synchronize()
        for name in ("q", "out", "split"):
            assert torch.equal(three[name], fused[name]), name
        nv = (ctx // 4).cpu().numpy()
        lt, lf = three["logits"].cpu().numpy(), fused["logits"].cpu().numpy()
        for b in range(B):
            assert np.array_equal(lt[b, :nv[b]].view(np.uint32), lf[b, :nv[b]].view(np.uint32)), b
            assert np.all(np.isnan(lf[b, nv[b]:])), b
        assert torch.equal(pools[0], pools[1])
    assert qsa.qsa_device_fault_flags() == 0


@pytest.mark.parametrize("B", [1, 64, 65])
def test_fused_decode_step_histogram_batch_edge(B):
    """Batches up to 64 sequences count each row's first-digit histogram while scoring
    (the last CTA copies and zeroes it); larger ones count it in the selection.  On both
    sides of that edge, with rows of 500 to 4096 visible blocks, two launches in a row
    equal the three separate calls bit for bit, and the selection equals the oracle's
    on the same logits."""
    qsa = _qsa()
    max_ctx = 16384
    pages = (max_ctx + 127) // 128
    num_pages = B * pages
    gen = torch.Generator(device="cuda").manual_seed(29 + B)
    pool0 = torch.randn((2 * num_pages, 128, 1, 128), device="cuda", generator=gen).to(torch.bfloat16)
    perm = torch.randperm(num_pages, device="cuda", generator=gen).to(torch.int32).view(B, pages)
    table = torch.stack([perm, perm + num_pages], dim=1).contiguous()
    ctx = torch.randint(2000, max_ctx + 1, (B,), device="cuda", generator=gen, dtype=torch.int32)
    ctx[0] = max_ctx
    rows = torch.randn((B, 640), device="cuda", generator=gen).to(torch.bfloat16)
    cs = torch.randn((max_ctx, 64), device="cuda", generator=gen)
    wq = (torch.randn(128, device="cuda", generator=gen) * 0.1).to(torch.bfloat16)
    wk = (torch.randn(128, device="cuda", generator=gen) * 0.1).to(torch.bfloat16)
    maxb = max_ctx // 4
    pools = [pool0.clone(), pool0.clone()]
    states = [qsa.pool_state(p_, table, num_pages, numKVHeads=1, poolHeadDim=128, headSize=0) for p_ in pools]

    def bufs():
        return dict(q=torch.empty((B, 1, 4, 128), dtype=torch.bfloat16, device="cuda"),
                    logits=torch.full((B, maxb), float("nan"), device="cuda"),
                    out=torch.empty((B, 2051), dtype=torch.int32, device="cuda"),
                    split=torch.full((B, 2), 3, dtype=torch.int32, device="cuda"))
    three, fused = bufs(), bufs()
    qsa.qsa_indexer_pre_decode(three["q"], rows, cs, ctx, wq, wk, 1e-6, states[0], B)
    qsa.qsa_index_scores_decode(three["logits"], three["q"], ctx, states[0], B, maxb)
    qsa.qsa_topk_expand_decode(three["out"], three["logits"], ctx, three["split"], 2, B, maxb)
    for _ in range(2):   # twice: the histograms and counters must be back at zero after the first
        fused["logits"].fill_(float("nan"))
        qsa.qsa_indexer_decode_step(fused["out"], fused["logits"], fused["q"], rows, cs, ctx, wq, wk, 1e-6,
                                    states[1], fused["split"], 2, B, maxb)
        torch.cuda.synchronize()
        for name in ("q", "out", "split"):
            assert torch.equal(three[name], fused[name]), name
        assert torch.equal(pools[0], pools[1])
    nv = (ctx // 4).cpu().numpy()
    lf = fused["logits"].cpu().numpy()
    for b in range(B):
        assert np.array_equal(three["logits"][b, :nv[b]].cpu().numpy().view(np.uint32), lf[b, :nv[b]].view(np.uint32)), b
    want = oracle.topk_expand_decode(np.where(np.isnan(lf), np.float32(-np.finfo(np.float32).max), lf), ctx.cpu().numpy())
    assert np.array_equal(fused["out"].cpu().numpy(), want)
    assert qsa.qsa_device_fault_flags() == 0


def test_fused_decode_step_recounts_histograms_that_do_not_total_the_row():
    """The one-launch step's selection checks that the first-digit counts it copies total
    the row's visible blocks, and counts the row itself when they do not (as after a launch
    whose waits ran out).  Every histogram offset by 7 in bin 0: two launches in a row still
    equal the three separate calls bit for bit, and so does one after the reset."""
    qsa = _qsa()
    B, max_ctx = 8, 12000
    pages = (max_ctx + 127) // 128
    num_pages = B * pages
    gen = torch.Generator(device="cuda").manual_seed(41)
    pool0 = torch.randn((2 * num_pages, 128, 1, 128), device="cuda", generator=gen).to(torch.bfloat16)
    perm = torch.randperm(num_pages, device="cuda", generator=gen).to(torch.int32).view(B, pages)
    table = torch.stack([perm, perm + num_pages], dim=1).contiguous()
    ctx = torch.randint(2100, max_ctx + 1, (B,), device="cuda", generator=gen, dtype=torch.int32)
    rows = torch.randn((B, 640), device="cuda", generator=gen).to(torch.bfloat16)
    cs = torch.randn((max_ctx, 64), device="cuda", generator=gen)
    wq = (torch.randn(128, device="cuda", generator=gen) * 0.1).to(torch.bfloat16)
    wk = (torch.randn(128, device="cuda", generator=gen) * 0.1).to(torch.bfloat16)
    maxb = max_ctx // 4
    pools = [pool0.clone(), pool0.clone()]
    states = [qsa.pool_state(p_, table, num_pages, numKVHeads=1, poolHeadDim=128, headSize=0) for p_ in pools]

    def bufs():
        return dict(q=torch.empty((B, 1, 4, 128), dtype=torch.bfloat16, device="cuda"),
                    logits=torch.full((B, maxb), float("nan"), device="cuda"),
                    out=torch.empty((B, 2051), dtype=torch.int32, device="cuda"),
                    split=torch.full((B, 2), 3, dtype=torch.int32, device="cuda"))
    three, fused = bufs(), bufs()
    qsa.qsa_indexer_pre_decode(three["q"], rows, cs, ctx, wq, wk, 1e-6, states[0], B)
    qsa.qsa_index_scores_decode(three["logits"], three["q"], ctx, states[0], B, maxb)
    qsa.qsa_topk_expand_decode(three["out"], three["logits"], ctx, three["split"], 2, B, maxb)
    try:
        qsa.qsa_testing_decode_step_histograms(7)
        for n in range(3):
            if n == 2:
                qsa.qsa_testing_decode_step_histograms(0)
            qsa.qsa_indexer_decode_step(fused["out"], fused["logits"], fused["q"], rows, cs, ctx, wq, wk, 1e-6,
                                        states[1], fused["split"], 2, B, maxb)
            torch.cuda.synchronize()
            for name in ("q", "out", "split"):
                assert torch.equal(three[name], fused[name]), (n, name)
            assert torch.equal(pools[0], pools[1]), n
    finally:
        qsa.qsa_testing_decode_step_histograms(0)
        torch.cuda.synchronize()
    assert qsa.qsa_device_fault_flags() == 0


def test_fused_decode_steps_in_flight_on_two_streams():
    """Launches of the one-launch step overlap on two streams (each launch takes its own
    arrival-counter set): 24 launches, alternating streams, on two independent problems,
    each equal bit for bit to its three-call reference."""
    qsa = _qsa()
    B, max_ctx = 48, 3000
    pages = (max_ctx + 1 + 127) // 128     # contexts up to max_ctx + 1
    num_pages = B * pages
    gen = torch.Generator(device="cuda").manual_seed(23)
    probs = []
    for _ in range(2):
        pool = torch.randn((2 * num_pages, 128, 1, 128), device="cuda", generator=gen).to(torch.bfloat16)
        perm = torch.randperm(num_pages, device="cuda", generator=gen).to(torch.int32).view(B, pages)
        table = torch.stack([perm, perm + num_pages], dim=1).contiguous()
        ctx = torch.randint(1, max_ctx + 1, (B,), device="cuda", generator=gen, dtype=torch.int32)
        ctx[ctx % 4 == 0] += 1            # no block completes: the pool is only read, so launches repeat
        rows = torch.randn((B, 640), device="cuda", generator=gen).to(torch.bfloat16)
        st = qsa.pool_state(pool, table, num_pages, numKVHeads=1, poolHeadDim=128, headSize=0)
        probs.append(dict(pool=pool, table=table, ctx=ctx, rows=rows, st=st))
    cs = torch.randn((max_ctx + 8, 64), device="cuda", generator=gen)   # positions up to max_ctx
    wq = (torch.randn(128, device="cuda", generator=gen) * 0.1).to(torch.bfloat16)
    wk = (torch.randn(128, device="cuda", generator=gen) * 0.1).to(torch.bfloat16)
    maxb = (max_ctx + 4) // 4

    def bufs():
        return dict(q=torch.empty((B, 1, 4, 128), dtype=torch.bfloat16, device="cuda"),
                    logits=torch.full((B, maxb), float("nan"), device="cuda"),
                    out=torch.empty((B, 2051), dtype=torch.int32, device="cuda"),
                    split=torch.full((B, 2), 3, dtype=torch.int32, device="cuda"))
    refs = []
    for p_ in probs:
        r = bufs()
        qsa.qsa_indexer_pre_decode(r["q"], p_["rows"], cs, p_["ctx"], wq, wk, 1e-6, p_["st"], B)
        qsa.qsa_index_scores_decode(r["logits"], r["q"], p_["ctx"], p_["st"], B, maxb)
        qsa.qsa_topk_expand_decode(r["out"], r["logits"], p_["ctx"], r["split"], 2, B, maxb)
        refs.append(r)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[bufs() for _ in range(12)] for _ in range(2)]
    for i in range(12):
        for k in range(2):
            with torch.cuda.stream(streams[k]):
                o, p_ = outs[k][i], probs[k]
                qsa.qsa_indexer_decode_step(o["out"], o["logits"], o["q"], p_["rows"], cs, p_["ctx"], wq, wk, 1e-6,
                                            p_["st"], o["split"], 2, B, maxb)
    torch.cuda.synchronize()
    for k in range(2):
        nv = (probs[k]["ctx"] // 4).cpu().numpy()
        lr = refs[k]["logits"].cpu().numpy()
        for i in range(12):
            o = outs[k][i]
            for name in ("q", "out", "split"):
                assert torch.equal(refs[k][name], o[name]), (k, i, name)
            lo = o["logits"].cpu().numpy()
            for b in range(B):
                assert np.array_equal(lr[b, :nv[b]].view(np.uint32), lo[b, :nv[b]].view(np.uint32)), (k, i, b)
    assert qsa.qsa_device_fault_flags() == 0


def test_fused_decode_step_validation():
    qsa = _qsa()
    P = 0x1000
    ok = qsa.PoolState(P, P, 4, 8, 2, 384, 256)
    with pytest.raises(qsa.QsaError) as e:
        qsa.qsa_indexer_decode_step(P, P, P, P, P, P, P, P, 1e-6, ok, 0, 2, 4097, 16, stream=0, dtype="bf16")
    assert e.value.status == -2                                       # batch above the counter set
    with pytest.raises(qsa.QsaError) as e:
        qsa.qsa_indexer_decode_step(P, P, P, P, P, P, P, P, 1e-6, ok, 0, 2, 4, 65537, stream=0, dtype="bf16")
    assert e.value.status == -2
    with pytest.raises(qsa.QsaError) as e:
        qsa.qsa_indexer_decode_step(P, P, P + 2, P, P, P, P, P, 1e-6, ok, 0, 2, 4, 16, stream=0, dtype="bf16")
    assert e.value.status == -5
