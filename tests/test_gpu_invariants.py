"""Exact invariants of the GPU kernels themselves ("Qsa Indexer Kernels":
launchQsaIndexQPrep, launchQsaIndexKCompress, launchQsaIndexScores,
launchQsaIndexScoresDecode), checked bit for bit without the oracle:

- the partial rope leaves dims 64..127 of every head alone, so one input row gives the
  same bits there at every position (K1a) and every block (K1b);
- K2 with kbar = 0 gives zero in every visible cell;
- K2 is positively homogeneous in q: doubling q (exact in T) doubles every visible
  logit exactly, since the products, the sums, relu and the scale all commute with a
  power-of-two factor away from overflow and underflow;
- visible logits are >= 0 (a sum of relus times a positive scale);
- a one-hot q (one non-zero element a in head h, dim d) gives the closed form
  fp32(relu(a * k_d)) * fp32(1/sqrt(128)) with the other heads' +0 added first.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu
NEG_MAX = np.float32(-np.finfo(np.float32).max)
SCALE = np.float32(1.0) / np.sqrt(np.float32(128.0))


def _g():
    import gpu_util
    return gpu_util


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_pass_through_dims_identical_at_every_position(dtype):
    g_ = _g()
    B, S = 2, 333
    wl = workloads.custom(B, S, [S, 250], dtype=dtype, seed=61, nan_padding=True, max_positions=S)
    same = wl.index_qk[0, 7].copy()                 # one row, repeated everywhere
    wl.index_qk[:, :, :] = same
    d = g_.DevWorkload(wl)
    q = g_.q_prep(d)                                # [B, S, 4, 128]
    NB = (S + 3) // 4
    kb = g_.k_compress(d, NB, 0, NB, 0)             # [B, NB, 128]
    for b, c in enumerate(wl.context_lengths):
        hi = q[b, :c, :, 64:]
        assert np.array_equal(hi, np.broadcast_to(hi[0], hi.shape)), b
        assert not q[b, c:].any()                   # padding rows: exact zeros
        assert np.array_equal(q[b, 0], q[0, 0])     # position 0 is the same in every sequence
        nv = c // 4
        khi = kb[b, :nv, 64:]
        assert np.array_equal(khi, np.broadcast_to(khi[0], khi.shape)), b
        # the rotated dims do change with the position
        assert not np.array_equal(q[b, 1, :, :64], q[b, 100, :, :64])


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_k2_zero_kbar_homogeneity_sign_and_one_hot(dtype):
    g_ = _g()
    B, S, NB = 2, 700, 200
    ctx = np.array([700, 421], np.int32)
    rng = np.random.default_rng(62)
    qf = rng.standard_normal((B, S, 4, 128)).astype(np.float32)
    kf = rng.standard_normal((B, NB, 128)).astype(np.float32)
    q = workloads.round_to_t(qf, dtype)
    kb = workloads.round_to_t(kf, dtype)
    d_ctx = g_.dev(ctx)
    rows = B * S
    t = np.arange(S)
    vis = np.zeros((B, S, NB), bool)
    for b in range(B):
        vis[b] = (t[:, None] < ctx[b]) & (np.arange(NB)[None, :] < ((t + 1) // 4)[:, None])
    vis = vis.reshape(rows, NB)

    base = g_.scores(dtype, g_.dev(q), g_.dev(kb), d_ctx, B, S, NB, 0, rows)
    assert np.all(base[~vis] == NEG_MAX)
    assert np.all(base[vis] >= 0)

    # kbar = 0: every visible cell is zero (the sign of a relu'd zero is not specified)
    zero = g_.scores(dtype, g_.dev(q), g_.dev(np.zeros_like(kb)), d_ctx, B, S, NB, 0, rows)
    assert np.all(zero[vis] == 0)
    assert np.all(zero[~vis] == NEG_MAX)

    # q doubled (exact in T for these magnitudes): every visible logit doubles exactly
    q2 = workloads.round_to_t(2.0 * workloads_to_f32(q, dtype), dtype)
    assert np.array_equal(workloads_to_f32(q2, dtype), 2.0 * workloads_to_f32(q, dtype))
    dbl = g_.scores(dtype, g_.dev(q2), g_.dev(kb), d_ctx, B, S, NB, 0, rows)
    assert np.array_equal(dbl[vis], np.float32(2.0) * base[vis])

    # one-hot q: head h_r, dim d_r of row r holds a_r, everything else +0
    hsel = rng.integers(0, 4, rows)
    dsel = rng.integers(0, 128, rows)
    a = rng.standard_normal(rows).astype(np.float32)
    qo = np.zeros((rows, 4, 128), np.float32)
    qo[np.arange(rows), hsel, dsel] = a
    qo_t = workloads.round_to_t(qo, dtype).reshape(B, S, 4, 128)
    a_t = workloads_to_f32(qo_t, dtype).reshape(rows, 4, 128)[np.arange(rows), hsel, dsel]
    one = g_.scores(dtype, g_.dev(qo_t), g_.dev(kb), d_ctx, B, S, NB, 0, rows)
    kf_t = workloads_to_f32(kb, dtype)                                   # [B, NB, 128]
    b_of = np.arange(rows) // S
    k_sel = kf_t[b_of[:, None], np.arange(NB)[None, :], dsel[:, None]]   # [rows, NB]
    prod = a_t[:, None] * k_sel                                          # exact in fp32
    expect = np.maximum(prod, np.float32(0)).astype(np.float32) * SCALE
    assert np.array_equal(one[vis], expect[vis])


def workloads_to_f32(bits, dtype):
    bits = np.asarray(bits, np.uint16)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    return bits.view(np.float16).astype(np.float32)
