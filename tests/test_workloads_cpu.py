"""The seeded synthetic inputs are what the input recipe says they are.

workloads/ feeds both the CUDA path and the oracle, so a wrong recipe would go unseen by
every parity test.  These checks pin the recipe: shapes, the N(0,1) and N(0, 0.1^2)
draws, the 1 % of rows scaled by 50, NaN in every column of every padding row, the
context-length ranges, the sub-range tiling of the decode-parity configuration, the
cos/sin table's angles, and that a seed fixes every bit.
"""
import math

import numpy as np
import pytest

import workloads

NAN = workloads.NAN_BITS


def _f32(bits, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(workloads.TORCH_DTYPES[dtype])
    return t.float().numpy()


def test_tiny_shapes_distributions_and_determinism():
    wl = workloads.tiny()
    assert (wl.B, wl.S, wl.num_blocks, wl.eps) == (1, 64, 16, 1e-6)
    assert wl.index_qk.shape == (1, 64, 640) and wl.index_qk.dtype == np.uint16
    assert wl.cos_sin.shape == (64, 64) and wl.cos_sin.dtype == np.float32
    assert wl.context_lengths.tolist() == [50] and wl.context_lengths.dtype == np.int32
    x = _f32(wl.index_qk, "bf16")
    assert abs(x.mean()) < 0.03 and abs(x.std() - 1.0) < 0.03
    for w in (wl.w_q, wl.w_k):
        g = _f32(w, "bf16")
        assert g.shape == (128,) and 0.07 < g.std() < 0.13
    again = workloads.tiny()
    assert np.array_equal(again.index_qk, wl.index_qk) and np.array_equal(again.w_k, wl.w_k)
    assert not np.array_equal(workloads.tiny(seed=1).index_qk, wl.index_qk)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_batched_outliers_nan_padding_and_lengths(dtype):
    wl = workloads.batched(dtype)
    assert (wl.B, wl.S, wl.dtype) == (4, 2048, dtype)
    ctx = wl.context_lengths
    assert ctx.min() >= 1 and ctx.max() <= 2048
    t = np.arange(wl.S)[None, :]
    pad = t >= ctx[:, None]
    # every column of every padding row is NaN; no valid row holds a NaN
    assert np.all(wl.index_qk[pad] == NAN[dtype])
    x = _f32(wl.index_qk, dtype)
    assert not np.isnan(x[~pad]).any()
    # outlier rows: all 640 columns scaled by 50, about 1 % of the rows
    rms = np.sqrt((x[~pad].astype(np.float64) ** 2).mean(axis=1))
    out = rms > 10.0
    assert 0.005 < out.mean() < 0.015
    assert np.all((rms[out] > 40.0) & (rms[out] < 60.0))
    assert np.all((rms[~out] > 0.8) & (rms[~out] < 1.2))


def test_long_prefill_has_one_incomplete_last_block():
    wl = workloads.long_prefill()
    assert (wl.B, wl.S, wl.num_blocks) == (1, 32768, 8192)
    c = int(wl.context_lengths[0])
    assert c == 32765
    valid = [g for g in range(wl.num_blocks) if 4 * g + 3 < c]
    assert len(valid) == 8191 and valid[-1] == 8190
    assert wl.cos_sin.shape == (32768, 64)


def test_decode_parity_lengths_and_subrange_tiles():
    wl = workloads.decode_parity()
    assert (wl.B, wl.S, wl.num_blocks) == (16, 8192, 2048)
    ctx = wl.context_lengths
    assert ctx.min() >= 4 and ctx.max() <= 8192
    for past in (0, 4, 128, 4096):
        tiles = workloads.subrange_tiles(3, past, wl.num_blocks)
        assert tiles[0][0] == max(past // 4 - 2, 0) and tiles[-1][1] == wl.num_blocks
        for (a, b), (c, _) in zip(tiles, tiles[1:]):
            assert b == c  # contiguous, in order
        sizes = [b - a for a, b in tiles]
        assert min(sizes) >= 1 and max(sizes) <= 64
        assert tiles == workloads.subrange_tiles(3, past, wl.num_blocks)


def test_scoring_padded_variant_structure():
    wl = workloads.scoring(B=3, S=256, full_context=False)
    assert wl.context_lengths.min() >= 1 and wl.context_lengths.max() <= 256
    pad = np.arange(256)[None, :] >= wl.context_lengths[:, None]
    assert np.all(wl.index_qk[pad] == NAN["bf16"])
    full = workloads.scoring(B=2, S=64, full_context=True)
    assert full.context_lengths.tolist() == [64, 64]
    assert not np.isnan(_f32(full.index_qk, "bf16")).any()


def test_cos_sin_table_angles():
    cs = workloads.cos_sin_table(40000)
    # position 0: cos exactly 1, sin exactly 0 (rope is the identity there)
    assert np.all(cs[0, :32] == 1.0) and np.all(cs[0, 32:] == 0.0)
    for p, i in [(1, 0), (7, 5), (4096, 31), (32767, 17), (39999, 1)]:
        ang = p * 1.0e6 ** (-2.0 * i / 64.0)
        assert cs[p, i] == np.float32(math.cos(ang))
        assert cs[p, 32 + i] == np.float32(math.sin(ang))
