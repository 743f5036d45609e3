"""GPU parity of K1a (q-prep) and K1b (K-compress) against the CPU oracle.

Structure (padding rows, invalid blocks, untouched rows, red zones) must match
bit for bit; values within the tolerance of tolerance.py; sub-range
recompression bit-identical to the full-range run ("Qsa Indexer Kernels",
launchQsaIndexQPrep and launchQsaIndexKCompress).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tolerance import check_t, to_f64

pytestmark = pytest.mark.gpu

SENT = 0x1234


def _gpu():
    import gpu_util
    return gpu_util


CONFIGS = {
    "tiny": lambda: workloads.tiny("bf16"),
    "batched_bf16": lambda: workloads.batched("bf16"),
    "batched_fp16": lambda: workloads.batched("fp16"),
    "long": lambda: workloads.long_prefill("bf16"),
}


def _report(name, st):
    print(f"{name}: n={st['n']} max_ulp={st['max_ulp']:.3f} floor_used={st['floor_used']}")


@pytest.fixture(scope="module", params=list(CONFIGS))
def cfg(request):
    g = _gpu()
    wl = CONFIGS[request.param]()
    return request.param, wl, g.DevWorkload(wl)


def test_q_prep_matches_oracle(cfg):
    name, wl, d = cfg
    got = _gpu().q_prep(d)
    ref = oracle.q_prep(wl.dtype, wl.index_qk, wl.cos_sin, wl.context_lengths, wl.w_q, wl.eps)
    t = np.arange(wl.S)[None, :]
    pad = t >= wl.context_lengths[:, None]
    assert not got[pad].any(), "padding rows must be exact +0.0"
    ok, st = check_t(got[~pad], ref[~pad], wl.dtype)
    _report(f"K1a {name}", st)
    assert ok, st


def test_k_compress_full_matches_oracle(cfg):
    name, wl, d = cfg
    NB = wl.num_blocks
    got = _gpu().k_compress(d, NB, 0, NB, 0)
    ref = oracle.k_compress(wl.dtype, wl.index_qk, wl.cos_sin, wl.context_lengths, wl.w_k, wl.eps,
                            NB, 0, NB, 0)
    g = np.arange(NB)[None, :]
    valid = (4 * g + 3) < wl.context_lengths[:, None]
    assert not got[~valid].any(), "invalid blocks must be exact +0.0"
    ok, st = check_t(got[valid], ref[valid], wl.dtype)
    _report(f"K1b {name}", st)
    assert ok, st


def test_k1b_equals_k1a_on_identical_rows():
    """Four identical K rows x at block g give exactly K1a's output for x at row 4g
    (same norm/rope device function, same wK, position 4g)."""
    g_ = _gpu()
    for dtype in ("bf16", "fp16"):
        wl = workloads.custom(2, 256, [256, 201], dtype=dtype, seed=17, nan_padding=False)
        iq = wl.index_qk.copy()
        for blk in range(64):
            iq[:, 4 * blk + 1:4 * blk + 4, 512:] = iq[:, 4 * blk:4 * blk + 1, 512:]
        iq[:, :, 0:128] = iq[:, :, 512:640]          # head 0 := the raw k row
        wl.index_qk = iq
        wl.w_q = wl.w_k                               # same gamma
        d = g_.DevWorkload(wl)
        q = g_.q_prep(d)
        kb = g_.k_compress(d, 64, 0, 64, 0)
        for b in range(2):
            for blk in range(64):
                if 4 * blk + 3 < wl.context_lengths[b]:
                    assert np.array_equal(kb[b, blk], q[b, 4 * blk, 0]), (dtype, b, blk)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("B,S,ctx", [(1, 1, [1]), (1, 3, [3]), (2, 5, [5, 0]), (1, 127, [126]),
                                     (3, 129, [129, 1, 64]), (2, 64, [0, 0]), (1, 4, [4])])
def test_small_odd_shapes(dtype, B, S, ctx):
    g_ = _gpu()
    wl = workloads.custom(B, S, ctx, dtype=dtype, seed=B * 1000 + S, nan_padding=True)
    d = g_.DevWorkload(wl)
    got = g_.q_prep(d)
    ref = oracle.q_prep(dtype, wl.index_qk, wl.cos_sin, wl.context_lengths, wl.w_q, wl.eps)
    ok, st = check_t(got.reshape(-1, 128), ref.reshape(-1, 128), dtype)
    assert ok, st
    NB = wl.num_blocks
    for bB, bE in ((0, NB), (NB // 2, NB), (0, 0)):
        got = g_.k_compress(d, NB, bB, bE, 0)
        ref = oracle.k_compress(dtype, wl.index_qk, wl.cos_sin, wl.context_lengths, wl.w_k, wl.eps,
                                NB, bB, bE, 0, kbar_init=np.full((B, NB, 128), SENT, np.uint16))
        ok, st = check_t(got.reshape(-1, 128), ref.reshape(-1, 128), dtype)
        assert ok, st
        assert np.array_equal(got == SENT, ref == SENT)


def test_decode_parity_subranges_bit_identical():
    """Config: B=16, S=8192, ctx ~ U{4..8192}.  Full compress once, then recompress
    tiles of 1..64 blocks with pastLen in {0, 4, 128, 4096} from indexQk rows
    [pastLen, S): every block with 4g >= pastLen must be bit-identical to the full
    run, tile blocks below pastLen exact zeros, rows outside the tiles untouched."""
    g_ = _gpu()
    wl = workloads.decode_parity("bf16")
    d = g_.DevWorkload(wl)
    NB = 2048
    full = g_.k_compress(d, NB, 0, NB, 0)
    ref = oracle.k_compress("bf16", wl.index_qk, wl.cos_sin, wl.context_lengths, wl.w_k, wl.eps,
                            NB, 0, NB, 0)
    valid = (4 * np.arange(NB)[None, :] + 3) < wl.context_lengths[:, None]
    assert not full[~valid].any()
    ok, st = check_t(full[valid], ref[valid], "bf16")
    _report("K1b decode-parity full", st)
    assert ok, st
    for P in (0, 4, 128, 4096):
        sub = d.index_qk[:, P:].contiguous()
        S_sub = wl.S - P
        kb = torch.full((wl.B, NB, 128), SENT, dtype=torch.int16, device="cuda")
        tiles = workloads.subrange_tiles(3, P, NB)
        import sparse_attention_indexer_qsa_gb300 as qsa
        for bB, bE in tiles:
            qsa.qsa_index_k_compress(kb, sub, d.cos_sin, d.ctx, d.w_k, wl.eps, wl.B, S_sub, NB,
                                     bB, bE, P, dtype="bf16")
        got = kb.cpu().numpy().view(np.uint16)
        lo = tiles[0][0]
        assert np.all(got[:, :lo] == SENT), "rows before the first tile were written"
        gi = np.arange(NB)
        above = (4 * gi >= P) & (gi >= lo)
        below = (4 * gi < P) & (gi >= lo)
        assert np.array_equal(got[:, above], full[:, above]), f"pastLen={P}: not bit-identical"
        assert not got[:, below].any(), f"pastLen={P}: blocks below pastLen must be zeros"


def test_nan_padding_never_read_and_deterministic():
    g_ = _gpu()
    wl = workloads.batched("bf16")
    d = g_.DevWorkload(wl)
    a = g_.q_prep(d)
    b = g_.q_prep(d)
    assert np.array_equal(a, b)
    NB = wl.num_blocks
    ka = g_.k_compress(d, NB, 0, NB, 0)
    kb = g_.k_compress(d, NB, 0, NB, 0)
    assert np.array_equal(ka, kb)
    assert np.all(np.isfinite(to_f64(a, "bf16"))) and np.all(np.isfinite(to_f64(ka, "bf16")))


def test_host_validation_enqueues_nothing():
    import sparse_attention_indexer_qsa_gb300 as qsa
    g_ = _gpu()
    wl = workloads.tiny("bf16")
    d = g_.DevWorkload(wl)
    out = torch.zeros((1, 64, 4, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qsa.QsaError) as e:
        qsa.qsa_index_q_prep(out.data_ptr() + 2, d.index_qk, d.cos_sin, d.ctx, d.w_q, 1e-6, 1, 64,
                             dtype="bf16")
    assert e.value.status == -5
    with pytest.raises(qsa.QsaError) as e:
        qsa.qsa_index_k_compress(out, d.index_qk, d.cos_sin, d.ctx, d.w_k, 1e-6, 1, 64, 16, 3, 2, 0)
    assert e.value.status == -3
    torch.cuda.synchronize()
    assert not out.view(torch.int16).any()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("B,S,ctx", [(1, 64, [50]), (3, 129, [129, 1, 0]), (2, 1000, [1000, 377]),
                                     (1, 33, [32]), (4, 2048, None), (1, 5, [5])])
def test_fused_qk_prep_bit_identical_to_separate_calls(dtype, B, S, ctx):
    """qsa_index_qk_prep == qsa_index_q_prep + qsa_index_k_compress(0, ceilDiv(S,4), 0)."""
    import sparse_attention_indexer_qsa_gb300 as qsa
    g_ = _gpu()
    if ctx is None:
        wl = workloads.batched(dtype)
    else:
        wl = workloads.custom(B, S, ctx, dtype=dtype, seed=B * 7 + S, nan_padding=True, outlier_frac=0.01)
    d = g_.DevWorkload(wl)
    NB = wl.num_blocks + 3                      # a wider row stride: extra rows untouched
    q_sep = g_.q_prep(d)
    k_sep = g_.k_compress(d, NB, 0, wl.num_blocks, 0)
    qo = g_.Guarded(wl.B * wl.S * 512 * 2)
    ko = g_.Guarded(wl.B * NB * 128 * 2, init=np.full((wl.B, NB, 128), SENT, np.uint16))
    qsa.qsa_index_qk_prep(qo.ptr, ko.ptr, d.index_qk, d.cos_sin, d.ctx, d.w_q, d.w_k, wl.eps, wl.B, wl.S,
                          NB, dtype=dtype)
    q_f = qo.numpy(np.uint16, q_sep.shape)
    k_f = ko.numpy(np.uint16, k_sep.shape)
    assert np.array_equal(q_f, q_sep)
    assert np.array_equal(k_f, k_sep)
    assert np.all(k_f[:, wl.num_blocks:] == SENT)
    g_.assert_no_device_faults()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_cos_sin_rows_past_the_last_needed_position_are_never_read(dtype):
    """cos/sin rows at positions no valid row or block uses (>= max ctx) hold NaN: K1a,
    K1b and the fused pass give the same bits as with a clean table."""
    import sparse_attention_indexer_qsa_gb300 as qsa
    g_ = _gpu()
    wl = workloads.custom(3, 300, [300, 157, 9], dtype=dtype, seed=61, nan_padding=True, max_positions=600)
    d = g_.DevWorkload(wl)
    NB = wl.num_blocks
    clean_q = g_.q_prep(d)
    clean_k = g_.k_compress(d, NB, 0, NB, 0)
    poisoned = wl.cos_sin.copy()
    poisoned[int(wl.context_lengths.max()):] = np.nan
    d.cos_sin = g_.dev(poisoned)
    assert np.array_equal(g_.q_prep(d), clean_q)
    assert np.array_equal(g_.k_compress(d, NB, 0, NB, 0), clean_k)
    td = g_.t_dtype(dtype)
    qn = torch.empty((3, 300, 4, 128), dtype=td, device="cuda")
    kb = torch.empty((3, NB, 128), dtype=td, device="cuda")
    qsa.qsa_index_qk_prep(qn, kb, d.index_qk, d.cos_sin, d.ctx, d.w_q, d.w_k, wl.eps, 3, 300, NB, dtype=dtype)
    torch.cuda.synchronize()
    assert np.array_equal(qn.view(torch.int16).cpu().numpy().view(np.uint16), clean_q)
    assert np.array_equal(kb.view(torch.int16).cpu().numpy().view(np.uint16), clean_k)
