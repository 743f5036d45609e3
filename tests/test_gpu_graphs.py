"""CUDA-graph capture and replay of the prefill and decode steps.

A serving engine records its per-step launches into a graph once and replays it with new
inputs written into the same buffers.  Every kernel on both paths is deterministic, so a
replay must give bit-identical outputs to the same calls made eagerly on the same inputs:
the fused K1 ("Qsa Indexer Kernels": launchQsaIndexerPrefill's q-prep and K-compress), the
scores (launchQsaIndexScores, whose work scheduler resets its own counters at the end of
every launch), the fused top-512 selection, and the decode chain (launchQsaIndexerPreDecode,
launchQsaIndexScoresDecode, launchQsaTopKExpandDecode) over a paged pool.
"""
import numpy as np
import pytest
import torch

import pool_util
import workloads

pytestmark = pytest.mark.gpu
W = 2051


def _qsa():
    import sparse_attention_indexer_qsa_gb300 as qsa
    return qsa


def _gu():
    import gpu_util
    return gpu_util


class Prefill:
    """Static buffers and the prefill step (fused K1, K2 in two row chunks, selection)."""

    def __init__(self, B, S, dtype="bf16"):
        qsa, g_ = _qsa(), _gu()
        self.B, self.S, self.NB = B, S, (S + 3) // 4
        wl = workloads.custom(B, S, [S] * B, dtype=dtype, seed=41)
        self.wl, self.dtype = wl, dtype
        td = g_.t_dtype(dtype)
        self.index_qk = g_.dev(wl.index_qk)
        self.cos_sin, self.w_q, self.w_k = g_.dev(wl.cos_sin), g_.dev(wl.w_q), g_.dev(wl.w_k)
        self.ctx = g_.dev(wl.context_lengths)
        self.qn = torch.empty((B, S, 4, 128), dtype=td, device="cuda")
        self.kb = torch.empty((B, self.NB, 128), dtype=td, device="cuda")
        self.logits = torch.empty((B * S, self.NB), dtype=torch.float32, device="cuda")
        self.out = torch.empty((B * S, W), dtype=torch.int32, device="cuda")
        self.qsa = qsa

    def step(self):
        q, B, S, NB = self.qsa, self.B, self.S, self.NB
        q.qsa_index_qk_prep(self.qn, self.kb, self.index_qk, self.cos_sin, self.ctx, self.w_q, self.w_k,
                            self.wl.eps, B, S, NB, dtype=self.dtype)
        half = (B * S) // 2
        q.qsa_index_scores(self.logits, self.qn, self.kb, self.ctx, B, S, NB, 0, half, dtype=self.dtype)
        q.qsa_index_scores(self.logits[half:], self.qn, self.kb, self.ctx, B, S, NB, half, B * S - half,
                           dtype=self.dtype)
        q.qsa_index_topk_expand(self.out, self.logits, self.ctx, B, S, NB, 0, B * S)

    def load(self, seed, ctx):
        rng = np.random.default_rng(seed)
        x = rng.standard_normal(self.index_qk.shape, dtype=np.float32)
        self.index_qk.copy_(torch.from_numpy(x).to(_gu().t_dtype(self.dtype)).view(torch.int16).cuda())
        self.ctx.copy_(torch.tensor(ctx, dtype=torch.int32))

    def snapshot(self):
        torch.cuda.synchronize()
        return [t.clone() for t in (self.qn, self.kb, self.logits, self.out)]


def _same(a, b):
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.uint8) if x.dtype.is_floating_point else x,
                           y.view(torch.uint8) if y.dtype.is_floating_point else y)


def test_prefill_step_graph_replays_bit_identical():
    p = Prefill(B=2, S=3000)
    inputs = [(7, [3000, 2999]), (8, [2047, 3000]), (9, [1, 1500])]
    eager = []
    for seed, ctx in inputs:                         # eager runs (also the first-call set-up)
        p.load(seed, ctx)
        p.step()
        eager.append(p.snapshot())
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            p.step()
    torch.cuda.current_stream().wait_stream(s)
    for rep in range(2):                             # replay every input twice
        for (seed, ctx), ref in zip(inputs, eager):
            p.load(seed, ctx)
            g.replay()
            _same(p.snapshot(), ref)
    assert _qsa().qsa_device_fault_flags() == 0


@pytest.mark.parametrize("fused", [False, True])
def test_decode_step_graph_replays_match_eager(fused):
    """Two copies of a prefilled pool advance token by token: one by eager calls of the
    three decode launches, one by replays of a graph of the same three launches or of the
    one-launch step (qsa_indexer_decode_step); every output and both pools stay
    bit-identical."""
    qsa, g_ = _qsa(), _gu()
    B, S, prefill = 3, 1100, [1020, 1023, 600]
    wl = workloads.custom(B, S, [S] * B, dtype="bf16", seed=43, max_positions=S)
    d = g_.DevWorkload(wl)
    NB = (S + 3) // 4
    maxb = NB + 5
    host_pool = pool_util.make_pool(B, S, seed=9)
    pools, states = [], []
    for _ in range(2):
        pool = g_.dev(host_pool.pool)
        table = g_.dev(host_pool.page_table)
        pools.append((pool, table))
        states.append(qsa.pool_state(pool, table, host_pool.num_pages))
    pctx = g_.dev(np.array(prefill, np.int32))
    kb = torch.empty((B, NB, 128), dtype=torch.bfloat16, device="cuda")
    for st in states:
        qsa.qsa_index_k_compress_paged(kb, d.index_qk, d.cos_sin, pctx, d.w_k, wl.eps, st, B, S, NB, 0, NB, 0,
                                       dtype="bf16")
        qsa.qsa_raw_k_tail_write_prefill(d.index_qk, pctx, st, B, S, dtype="bf16")

    def buffers():
        return dict(row=torch.empty((B, 640), dtype=torch.int16, device="cuda"),
                    ctx=torch.empty((B,), dtype=torch.int32, device="cuda"),
                    q=torch.empty((B, 1, 4, 128), dtype=torch.bfloat16, device="cuda"),
                    logits=torch.full((B, maxb), float("nan"), device="cuda"),
                    out=torch.empty((B, W), dtype=torch.int32, device="cuda"),
                    split=torch.zeros((B, 2), dtype=torch.int32, device="cuda"))

    def step(bf, st):
        qsa.qsa_indexer_pre_decode(bf["q"], bf["row"], d.cos_sin, bf["ctx"], d.w_q, d.w_k, wl.eps, st, B,
                                   dtype="bf16")
        qsa.qsa_index_scores_decode(bf["logits"], bf["q"], bf["ctx"], st, B, maxb, dtype="bf16")
        qsa.qsa_topk_expand_decode(bf["out"], bf["logits"], bf["ctx"], bf["split"], 2, B, maxb)

    def feed(bf, k):
        pos = [p + k for p in prefill]
        ctx = np.array([ps + 1 for ps in pos], np.int32)
        rows = np.stack([wl.index_qk[b, pos[b]] for b in range(B)])
        bf["row"].copy_(torch.from_numpy(rows.view(np.int16)))
        bf["ctx"].copy_(torch.from_numpy(ctx))
        bf["split"].fill_(5)

    def step_fused(bf, st):
        qsa.qsa_indexer_decode_step(bf["out"], bf["logits"], bf["q"], bf["row"], d.cos_sin, bf["ctx"], d.w_q,
                                    d.w_k, wl.eps, st, bf["split"], 2, B, maxb, dtype="bf16")

    graph_step = step_fused if fused else step
    eager_bf, graph_bf = buffers(), buffers()
    feed(eager_bf, 0)
    step(eager_bf, states[0])                        # first-call set-up outside the capture
    if fused:                                        # (token 0's writes again, so idempotent)
        feed(graph_bf, 0)
        graph_step(graph_bf, states[1])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    feed(graph_bf, 0)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            graph_step(graph_bf, states[1])
    torch.cuda.current_stream().wait_stream(s)
    for k in range(0, 70):                           # crosses a 4-token block edge many times
        if k > 0:
            feed(eager_bf, k)
            step(eager_bf, states[0])
        feed(graph_bf, k)
        g.replay()
        torch.cuda.synchronize()
        for name in ("q", "out", "split"):
            assert torch.equal(eager_bf[name], graph_bf[name]), (k, name)
        nv = [(p + k + 1) // 4 for p in prefill]
        for b in range(B):
            assert torch.equal(eager_bf["logits"][b, :nv[b]].view(torch.int32),
                               graph_bf["logits"][b, :nv[b]].view(torch.int32)), (k, b)
        assert not graph_bf["split"].any()
    assert torch.equal(pools[0][0], pools[1][0])    # the two pools evolved identically
    assert qsa.qsa_device_fault_flags() == 0
