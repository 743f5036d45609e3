"""The algorithmic byte and flop counts behind every roofline fraction bench.py reports.

bench.algorithmic_bytes computes them with vectorised sums.  Here they are pinned to a
plain enumeration of the rows, blocks and cells each kernel touches ("Qsa Indexer
Kernels": launchQsaIndexQPrep reads a valid row's 4 q heads and writes 4 heads, writes
zeros for a padding row; launchQsaIndexKCompress reads the 4 raw K rows of a valid block
and writes one kbar row, writes zeros for an invalid one; launchQsaIndexScores reads q
rows and the visible kbar rows and writes every logit), on ragged shapes, and to the
closed forms of the scoring workload (B=8, S=16384, ctx=S) worked out by hand.
"""
import numpy as np
import pytest

T = 2  # bytes per element


def enumerate_bytes(ctx, B, S, NB):
    k1a = k1b = k2 = select = fused = flops = 0
    positions = set()
    k_positions = set()
    for b in range(B):
        c = max(0, int(ctx[b]))
        for t in range(S):
            if t < c:
                k1a += 4 * 128 * T + 4 * 128 * T  # read q heads, write qNormed
                positions.add(t)
                k2 += 4 * 128 * T  # q row read once
                fused += 4 * 128 * T
                vis = min((t + 1) // 4, NB)
                select += vis * 4
                flops += vis * 4 * 128 * 2
            else:
                k1a += 4 * 128 * T  # zeros written, nothing read
        for g in range(NB):
            if 4 * g + 3 < c:
                k1b += 4 * 128 * T + 128 * T  # four raw K rows read, kbar row written
                k_positions.add(4 * g)
                k2 += 128 * T  # each visible kbar row read once per sequence
                fused += 128 * T
            else:
                k1b += 128 * T
    k1a += len(positions) * 64 * 4  # one FP32 cos/sin row per distinct position
    k1b += len(k_positions) * 64 * 4
    k2 += B * S * NB * 4  # every logit written (masked cells too)
    select += B * S * 2051 * 4  # 2051 token ids per row
    fused += B * S * 2051 * 4  # scoring fused with selection: no logits, the ids written
    return {"k1a": k1a, "k1b": k1b, "k2": k2, "select": select, "fused_select": fused,
            "k2_causal_flops": flops}


@pytest.mark.parametrize("B,S,NB,ctx", [
    (1, 64, 16, [50]),
    (3, 37, 10, [37, 0, 5]),
    (4, 33, 12, [1, 4, 7, 33]),
    (2, 16, 9, [16, 3]),       # NB above ceilDiv(S, 4)
    (2, 12, 3, [-5, 12]),      # a non-positive length is all padding
])
def test_algorithmic_bytes_equal_enumeration(B, S, NB, ctx):
    import bench
    ctx = np.asarray(ctx, np.int32)
    assert bench.algorithmic_bytes(ctx, B, S, NB) == enumerate_bytes(ctx, B, S, NB)


def test_scoring_workload_closed_forms():
    import bench
    B, S, NB = 8, 16384, 4096
    got = bench.algorithmic_bytes(np.full(B, S, np.int32), B, S, NB)
    rows = B * S
    # K2: q rows 131072 x 1 KiB, kbar 8 x 4096 x 256 B, logits 131072 x 4096 x 4 B
    assert got["k2"] == rows * 1024 + B * NB * 256 + rows * NB * 4 == 2_290_089_984
    # sum over t < 16384 of floor((t+1)/4) = 4 * (1 + ... + 4095) + 4096 = 4096 * 8191
    assert got["k2_causal_flops"] == B * 4096 * 8191 * 4 * 128 * 2
    # K1a: every row valid (read 1 KiB, write 1 KiB) plus one cos/sin row per position
    assert got["k1a"] == rows * 2048 + S * 256
    # K1b: every block valid (read 1 KiB, write 256 B) plus one cos/sin row per block index
    assert got["k1b"] == B * NB * 1280 + NB * 256
