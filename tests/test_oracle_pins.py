"""Pins for the CPU oracle against facts that do not come from the oracle itself.

Each test names what fixes the expected value: an IEEE definition checked
against numpy/torch, torch's rms_norm, complex rotation, a closed form, an
invariant, or float64 brute force.  Formulas follow the "Qsa Indexer Kernels"
page (launchQsaIndexQPrep, launchQsaIndexKCompress, launchQsaIndexScores).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from tolerance import check_t, check_logits, logits_floor, to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NEG_MAX = np.float32(-np.finfo(np.float32).max)
DTYPES = ["bf16", "fp16"]


def t_bits(values, dtype):
    return workloads.round_to_t(np.asarray(values, np.float64), dtype)


# ------------------------------------------------------------------ conversions

def test_widening_matches_torch_and_numpy_on_every_pattern():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    bf = oracle.t_to_f32("bf16", allbits)
    ref = torch.from_numpy(allbits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(np.isnan(bf), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(bf[fin].view(np.uint32), ref[fin].view(np.uint32))
    hf = oracle.t_to_f32("fp16", allbits)
    ref16 = allbits.view(np.float16).astype(np.float32)
    assert np.array_equal(np.isnan(hf), np.isnan(ref16))
    fin = ~np.isnan(ref16)
    assert np.array_equal(hf[fin].view(np.uint32), ref16[fin].view(np.uint32))


def _probe_floats(rng):
    # random bit patterns over every exponent, plus every T value and every midpoint
    # between neighbouring T values (the ties), plus signed zeros/inf/extremes
    rnd = rng.integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32).view(np.float32)
    extra = np.array([0.0, -0.0, np.inf, -np.inf, np.finfo(np.float32).max,
                      -np.finfo(np.float32).max, np.finfo(np.float32).tiny, 1e-45, 65504.0,
                      65519.99, 65520.0, 6.1e-5, 5.96e-8, 2.98e-8, 2.99e-8], np.float32)
    return np.concatenate([rnd, extra])


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(11)
    f = _probe_floats(rng)
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = (allb.astype(np.uint32) << 16).view(np.float32)
    mids = ((allb.astype(np.uint32) << 16) | 0x8000).view(np.float32)   # exact ties
    with np.errstate(invalid="ignore"):
        f = np.concatenate([f, vals, mids, np.nextafter(mids, np.float32(np.inf)),
                            np.nextafter(mids, np.float32(-np.inf))])
    got = oracle.f32_to_t("bf16", f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(to_f64(got[nan], "bf16")))


def test_fp16_rounding_matches_numpy():
    rng = np.random.default_rng(12)
    f = _probe_floats(rng)
    allh = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    hv = allh.view(np.float16).astype(np.float64)
    fin = np.isfinite(hv)
    hv = np.unique(hv[fin])
    mids = ((hv[:-1] + hv[1:]) / 2).astype(np.float32)                 # exact in fp32
    f = np.concatenate([f, hv.astype(np.float32), mids, np.nextafter(mids, np.float32(np.inf)),
                        np.nextafter(mids, np.float32(-np.inf))])
    got = oracle.f32_to_t("fp16", f)
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(to_f64(got[nan], "fp16")))


# --------------------------------------------------------------- norm + rope step

def ref_norm_rope64(x, w_bits, eps, cs_row, dtype):
    """float64 reference: torch rms_norm with weight (1 + w), then rotation of the
    complex numbers y_i + i*y_{i+32} by cos + i*sin (i < 32)."""
    w = to_f64(w_bits, dtype)
    xt = torch.from_numpy(np.asarray(x, np.float64))[None, :]
    y = torch.nn.functional.rms_norm(xt, (128,), weight=torch.from_numpy(1.0 + w), eps=eps)
    y = y[0].numpy()
    cs = np.asarray(cs_row, np.float64)
    z = (y[:32] + 1j * y[32:64]) * (cs[:32] + 1j * cs[32:])
    return np.concatenate([z.real, z.imag, y[64:]])


@pytest.mark.parametrize("dtype", DTYPES)
def test_norm_rope_matches_rms_norm_and_complex_rotation(dtype):
    rng = np.random.default_rng(21)
    table = workloads.cos_sin_table(4096)
    floor_used, n = 0, 0
    for trial in range(300):
        scale = [1.0, 50.0, 1e-3][trial % 3]
        x = to_f64(t_bits(rng.standard_normal(128) * scale, dtype), dtype)
        w = t_bits(rng.normal(0, 0.1, 128), dtype)
        pos = int(rng.integers(0, 4096))
        out = oracle.norm_rope(dtype, x, w, 1e-6, table[pos])
        ref = ref_norm_rope64(x, w, 1e-6, table[pos], dtype)
        ok, st = check_t(out, ref, dtype)
        assert ok, (trial, st)
        floor_used += st["floor_used"]
        n += st["n"]
    # every element is within one ulp of T except the rare ones where the rope's
    # subtraction cancels to a tiny value (those pass by the head-relative floor)
    assert floor_used <= n // 1000, (floor_used, n)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("dim", [0, 5, 31, 32, 40, 63, 64, 100, 127])
def test_norm_rope_one_hot_closed_form(dtype, dim):
    # x = v * e_dim, eps = 0: meanSq = v^2/128, y_dim = sign(v) * sqrt(128) * (1 + w_dim);
    # rope moves y_dim to (dim, dim+32) as (y cos, y sin) for dim < 32, to (dim-32, dim)
    # as (-y sin, y cos) for 32 <= dim < 64, and leaves dims >= 64 alone.
    rng = np.random.default_rng(dim)
    table = workloads.cos_sin_table(512)
    for v in (3.0, -0.5):
        w = t_bits(rng.normal(0, 0.1, 128), dtype)
        pos = 257
        x = np.zeros(128)
        x[dim] = v
        out = to_f64(oracle.norm_rope(dtype, x, w, 0.0, table[pos]), dtype)
        y = np.sign(v) * np.sqrt(128.0) * (1.0 + to_f64(w, dtype)[dim])
        exp = np.zeros(128)
        if dim < 32:
            exp[dim] = y * table[pos][dim]
            exp[dim + 32] = y * table[pos][32 + dim]
        elif dim < 64:
            i = dim - 32
            exp[i] = -y * table[pos][32 + i]
            exp[dim] = y * table[pos][i]
        else:
            exp[dim] = y
        ok, st = check_t(t_bits(out, dtype), exp, dtype)
        assert ok, st
        nz = np.flatnonzero(out)
        assert set(nz) <= set(np.flatnonzero(exp)), (nz, np.flatnonzero(exp))


@pytest.mark.parametrize("dtype", DTYPES)
def test_gamma_invariants(dtype):
    rng = np.random.default_rng(31)
    table = workloads.cos_sin_table(1024)
    for _ in range(50):
        x = to_f64(t_bits(rng.standard_normal(128), dtype), dtype)
        pos = int(rng.integers(0, 1024))
        eps = 1e-6
        zero = np.zeros(128, np.uint16)                 # +0.0 in both encodings
        out0 = to_f64(oracle.norm_rope(dtype, x, zero, eps, table[pos]), dtype)
        # zero gamma: unit RMS before rope (times sqrt(meanSq/(meanSq+eps))), rope keeps it
        ms = np.mean(x * x)
        rms = np.sqrt(np.mean(out0 ** 2))
        assert abs(rms - np.sqrt(ms / (ms + eps))) < 2.0 ** -MANT(dtype), rms
        # gamma = -1: (1 + w) = 0 exactly -> all zeros
        minus1 = t_bits(-np.ones(128), dtype)
        assert np.all(to_f64(oracle.norm_rope(dtype, x, minus1, eps, table[pos]), dtype) == 0.0)
        # gamma = +1 doubles every pre-cast value exactly, and the cast commutes with x2
        plus1 = t_bits(np.ones(128), dtype)
        out2 = to_f64(oracle.norm_rope(dtype, x, plus1, eps, table[pos]), dtype)
        assert np.array_equal(out2, 2.0 * out0)


def MANT(dtype):
    return {"bf16": 7, "fp16": 10}[dtype]


@pytest.mark.parametrize("dtype", DTYPES)
def test_gamma_applies_to_its_own_dim(dtype):
    # w = -1 except at one dim: only that dim survives at the identity rope (pos 0)
    table = workloads.cos_sin_table(4)
    rng = np.random.default_rng(41)
    x = to_f64(t_bits(rng.standard_normal(128), dtype), dtype)
    for d0 in (0, 17, 33, 70, 127):
        w = -np.ones(128)
        w[d0] = 0.0
        out = to_f64(oracle.norm_rope(dtype, x, t_bits(w, dtype), 1e-6, table[0]), dtype)
        assert np.flatnonzero(out).tolist() == [d0]


@pytest.mark.parametrize("dtype", DTYPES)
def test_rope_position_zero_is_identity_bitwise(dtype):
    # With integer inputs the sum of squares is exact in any order, so r is unique and
    # swapping the rotated half [0, 64) with the pass-through half [64, 128) must permute
    # the output exactly when the rope is the identity (cos = 1, sin = 0 at position 0).
    table = workloads.cos_sin_table(4)
    assert np.all(table[0, :32] == 1.0) and np.all(table[0, 32:] == 0.0)
    rng = np.random.default_rng(51)
    for _ in range(20):
        x = rng.integers(-8, 9, 128).astype(np.float64)
        x[0] = 5.0
        w = t_bits(rng.normal(0, 0.1, 128), dtype)
        perm = np.concatenate([np.arange(64, 128), np.arange(0, 64)])
        a = oracle.norm_rope(dtype, x, w, 1e-6, table[0])
        b = oracle.norm_rope(dtype, x[perm], w[perm], 1e-6, table[0])
        assert np.array_equal(a[perm], b)


@pytest.mark.parametrize("dtype", DTYPES)
def test_norm_is_scale_invariant_without_eps(dtype):
    rng = np.random.default_rng(61)
    table = workloads.cos_sin_table(64)
    for k in (-3, 1, 4):
        x = to_f64(t_bits(rng.standard_normal(128), dtype), dtype)
        w = t_bits(rng.normal(0, 0.1, 128), dtype)
        a = oracle.norm_rope(dtype, x, w, 0.0, table[9])
        b = oracle.norm_rope(dtype, x * 2.0 ** k, w, 0.0, table[9])
        assert np.array_equal(a, b)


# ------------------------------------------------------------------- block mean

@pytest.mark.parametrize("dtype", DTYPES)
def test_block_mean_special_cases(dtype):
    rng = np.random.default_rng(71)
    for _ in range(20):
        x = t_bits(rng.standard_normal(128) * 30, dtype)
        assert np.array_equal(oracle.block_mean(dtype, x, x, x, x), x)   # (x+x)+x+x exact
        a = t_bits(rng.standard_normal(128), dtype)
        b = t_bits(rng.standard_normal(128), dtype)
        na = a ^ np.uint16(0x8000)
        nb = b ^ np.uint16(0x8000)
        assert np.all(to_f64(oracle.block_mean(dtype, a, na, b, nb), dtype) == 0.0)


@pytest.mark.parametrize("dtype", DTYPES)
def test_block_mean_is_rounded_exact_mean_when_sums_are_exact(dtype):
    # values in [1/8, 8): every partial sum of four is exact in binary32, so the fixed
    # order changes nothing and m must be the correctly rounded exact mean
    rng = np.random.default_rng(81)
    for _ in range(50):
        ks = [t_bits(np.exp2(rng.uniform(-3, 3, 128)) * rng.choice([-1, 1], 128), dtype)
              for _ in range(4)]
        exact = sum(to_f64(k, dtype) for k in ks) / 4.0
        assert np.array_equal(oracle.block_mean(dtype, *ks), t_bits(exact, dtype))


def test_block_mean_fixed_order_golden():
    with open(os.path.join(GOLDEN, "block_mean_order.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        dtype = c["dtype"]
        ks = [t_bits(np.full(128, v), dtype) for v in c["k"]]
        m = to_f64(oracle.block_mean(dtype, *ks), dtype)
        assert np.all(m == c["mean"]), (c, m[:4])


# -------------------------------------------------------------------- K1a whole

@pytest.mark.parametrize("dtype", DTYPES)
def test_q_prep_padding_and_per_head_rows(dtype):
    wl = workloads.custom(2, 40, [37, 0], dtype=dtype, seed=5, nan_padding=True)
    out = oracle.q_prep(dtype, wl.index_qk, wl.cos_sin, wl.context_lengths, wl.w_q, wl.eps)
    for b in range(2):
        for t in range(40):
            if t >= wl.context_lengths[b]:
                assert not out[b, t].any()                     # +0.0 bits everywhere
                continue
            for h in range(4):
                x = to_f64(wl.index_qk[b, t, 128 * h:128 * (h + 1)], dtype)
                ref = ref_norm_rope64(x, wl.w_q, wl.eps, wl.cos_sin[t], dtype)
                ok, st = check_t(out[b, t, h], ref, dtype)
                assert ok, (b, t, h, st)


# -------------------------------------------------------------------- K1b whole

def expected_valid_count(ctx, S, P, bB, bE):
    """Closed form for #{g in [bB, bE): 4g+3 < ctx, 4g >= P, 4g+3-P < S}."""
    lo = max(bB, -(-P // 4))
    hi = min(bE, max(ctx, 0) // 4, (S + P) // 4)
    return max(0, hi - lo)


@pytest.mark.parametrize("dtype", DTYPES)
def test_k_compress_structure_closed_form(dtype):
    rng = np.random.default_rng(91)
    for trial in range(30):
        B = 3
        P = int(rng.choice([0, 1, 3, 4, 7, 12]))
        S = int(rng.integers(1, 60))
        ctx = rng.integers(-2, S + P + 6, size=B).astype(np.int32)
        NB = (S + P + 3) // 4 + int(rng.integers(0, 3))
        bB = int(rng.integers(0, NB + 1))
        bE = int(rng.integers(bB, NB + 1))
        wl = workloads.custom(B, S, np.clip(ctx, 0, None), dtype=dtype, seed=trial, nan_padding=False)
        iq = wl.index_qk.copy()
        # rows past ctx - P are never read: poison them
        for b in range(B):
            iq[b, max(ctx[b] - P, 0):] = workloads.NAN_BITS[dtype]
        sentinel = np.full((B, NB, 128), 0x1234, np.uint16)
        kb = oracle.k_compress(dtype, iq, workloads.cos_sin_table(4 * NB + 4), ctx, wl.w_k,
                               wl.eps, NB, bB, bE, P, kbar_init=sentinel)
        assert np.all(kb[:, :bB] == 0x1234) and np.all(kb[:, bE:] == 0x1234)
        for b in range(B):
            rows = kb[b, bB:bE]
            nonzero = np.any(rows != 0, axis=1)
            assert int(nonzero.sum()) == expected_valid_count(int(ctx[b]), S, P, bB, bE)
            assert np.all(np.isfinite(to_f64(rows, dtype)))


@pytest.mark.parametrize("dtype", DTYPES)
def test_k_compress_identical_rows_equal_normed_row_at_4g(dtype):
    rng = np.random.default_rng(101)
    S = 64
    wl = workloads.custom(1, S, [S], dtype=dtype, seed=3, nan_padding=False)
    iq = wl.index_qk.copy()
    for g in range(S // 4):
        iq[0, 4 * g + 1:4 * g + 4, 512:] = iq[0, 4 * g, 512:]
    kb = oracle.k_compress(dtype, iq, wl.cos_sin, wl.context_lengths, wl.w_k, wl.eps,
                           S // 4, 0, S // 4, 0)
    for g in range(S // 4):
        x = to_f64(iq[0, 4 * g, 512:], dtype)
        assert np.array_equal(kb[0, g], oracle.norm_rope(dtype, x, wl.w_k, wl.eps, wl.cos_sin[4 * g]))
        ok, st = check_t(kb[0, g], ref_norm_rope64(x, wl.w_k, wl.eps, wl.cos_sin[4 * g], dtype), dtype)
        assert ok, st
    del rng


@pytest.mark.parametrize("P", [0, 4, 6, 128])
def test_k_compress_reads_rows_4g_plus_j_minus_pastlen(P):
    # token i's raw k is one-hot at dim 64 + (i mod 64) with value 1; block g's mean is
    # 0.25 at the four dims of tokens 4g..4g+3, so with eps = 0 and w = 0 the output is
    # sqrt(32) exactly there (pass-through half, no rope) and 0 elsewhere.
    dtype = "bf16"
    total = 256
    S = total - P
    iq = np.zeros((1, S, 640), np.uint16)
    one = t_bits([1.0], dtype)[0]
    for i in range(S):
        tok = i + P
        iq[0, i, 512 + 64 + tok % 64] = one
    NB = total // 4
    kb = oracle.k_compress(dtype, iq, workloads.cos_sin_table(total), [total],
                           np.zeros(128, np.uint16), 0.0, NB, 0, NB, P)
    val = t_bits([np.sqrt(32.0)], dtype)[0]
    for g in range(NB):
        if 4 * g < P:
            assert not kb[0, g].any()
            continue
        exp = np.zeros(128, np.uint16)
        for j in range(4):
            exp[64 + (4 * g + j) % 64] = val
        # valid blocks compare by value: 0 * (negative cos) is a legitimate -0.0
        assert np.array_equal(to_f64(kb[0, g], dtype), to_f64(exp, dtype)), g


def test_k_compress_sums_rows_4g_to_4g_plus_3_in_that_order():
    # dim 0 of the block's four rows holds an order-sensitive golden case, every other
    # dim is 1.0 in all rows (mean exactly 1); eps = 0, w = 0, position 0 (rope is the
    # identity there).  The output must equal the norm of [golden mean, 1, 1, ...]: a K
    # compress that read the rows in another order, or summed them in another order,
    # would normalise a different first element.
    with open(os.path.join(GOLDEN, "block_mean_order.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        dtype = c["dtype"]
        iq = np.zeros((1, 4, 640), np.uint16)
        iq[0, :, 512:] = t_bits([1.0], dtype)[0]
        iq[0, :, 512] = t_bits(c["k"], dtype)
        cs = workloads.cos_sin_table(4)
        kb = oracle.k_compress(dtype, iq, cs, [4], np.zeros(128, np.uint16), 0.0, 1, 0, 1, 0)
        x = np.ones(128)
        x[0] = c["mean"]
        assert np.array_equal(kb[0, 0], oracle.norm_rope(dtype, x, np.zeros(128, np.uint16), 0.0, cs[0])), c
        ok, st = check_t(kb[0, 0], ref_norm_rope64(x, np.zeros(128, np.uint16), 0.0, cs[0], dtype), dtype)
        assert ok, (c, st)


@pytest.mark.parametrize("dtype", DTYPES)
def test_k_compress_subrange_equals_full(dtype):
    wl = workloads.custom(3, 96, [96, 50, 7], dtype=dtype, seed=9)
    NB = 24
    full = oracle.k_compress(dtype, wl.index_qk, wl.cos_sin, wl.context_lengths, wl.w_k, wl.eps,
                             NB, 0, NB, 0)
    for P in (0, 4, 5, 20, 64):
        sub = np.ascontiguousarray(wl.index_qk[:, P:])
        for bB, bE in ((0, NB), (max(P // 4 - 2, 0), NB), (P // 4 + 1, min(P // 4 + 3, NB))):
            kb = oracle.k_compress(dtype, sub, wl.cos_sin, wl.context_lengths, wl.w_k, wl.eps,
                                   NB, bB, bE, P)
            for g in range(bB, bE):
                if 4 * g >= P:
                    assert np.array_equal(kb[:, g], full[:, g]), (P, g)
                else:
                    assert not kb[:, g].any()


# ---------------------------------------------------------------------- scores

def brute_scores64(q_bits, kbar_bits, ctx, dtype):
    q = to_f64(q_bits, dtype)          # [B, S, 4, 128]
    k = to_f64(kbar_bits, dtype)       # [B, NB, 128]
    B, S = q.shape[:2]
    NB = k.shape[1]
    dots = np.einsum("bthd,bgd->btgh", q, k)
    val = np.maximum(dots, 0.0).sum(-1) / np.sqrt(128.0)
    t = np.arange(S)[None, :, None]
    g = np.arange(NB)[None, None, :]
    vis = (g < (t + 1) // 4) & (t < np.asarray(ctx)[:, None, None])
    return np.where(vis, val, -np.finfo(np.float32).max).reshape(B * S, NB)


@pytest.mark.parametrize("dtype", DTYPES)
def test_scores_match_float64_brute_force(dtype):
    rng = np.random.default_rng(111)
    B, S, NB = 2, 45, 13
    q = t_bits(rng.standard_normal((B, S, 4, 128)) * 3, dtype)
    kb = t_bits(rng.standard_normal((B, NB, 128)) * 3, dtype)
    ctx = np.array([45, 30], np.int32)
    got = oracle.scores(dtype, q, kb, ctx)
    ref = brute_scores64(q, kb, ctx, dtype).astype(np.float32)
    fl = logits_floor(q.reshape(B * S, 4, 128),
                      np.repeat(kb, S, axis=0).reshape(B * S, NB, 128), dtype)
    ok, st = check_logits(got, ref, dtype, fl)
    assert ok, st
    assert np.all(got[got != NEG_MAX] >= 0.0)


def test_scores_closed_forms():
    dtype = "bf16"
    rng = np.random.default_rng(121)
    B, S, NB = 1, 64, 16
    scale32 = np.float32(1.0) / np.sqrt(np.float32(128.0))
    # one-hot q (head h, dim d, value a) against kbar rows that are one-hot at d
    for h, d in ((0, 3), (2, 127), (3, 64)):
        q = np.zeros((B, S, 4, 128), np.uint16)
        a = 1.5
        q[..., h, d] = t_bits([a], dtype)[0]
        kb = np.zeros((B, NB, 128), np.uint16)
        bvals = t_bits(rng.standard_normal(NB), dtype)
        kb[0, :, d] = bvals
        got = oracle.scores(dtype, q, kb, [S])
        prod = (np.float32(a) * to_f64(bvals, dtype).astype(np.float32))
        exp = (scale32 * np.maximum(prod, np.float32(0))).astype(np.float32)
        for t in range(S):
            nvis = (t + 1) // 4
            assert np.array_equal(got[t, :nvis], exp[:nvis])
            assert np.all(got[t, nvis:] == NEG_MAX)
    # relu per head, not after the head sum: heads v and -v give |v.k| / sqrt(128)
    v = rng.standard_normal(128)
    q = np.zeros((B, S, 4, 128), np.uint16)
    q[..., 0, :] = t_bits(v, dtype)
    q[..., 1, :] = q[..., 0, :] ^ np.uint16(0x8000)
    kb = t_bits(rng.standard_normal((B, NB, 128)), dtype)
    got = oracle.scores(dtype, q, kb, [S])
    exact = np.abs(to_f64(kb[0], dtype) @ to_f64(q[0, 0, 0], dtype)) / np.sqrt(128.0)
    vis = got[S - 1]
    assert np.allclose(vis, exact, rtol=2.0 ** -16, atol=1e-6)
    # zero kbar -> every visible logit is +0
    got0 = oracle.scores(dtype, q, np.zeros_like(kb), [S])
    vis0 = got0[got0 != NEG_MAX]
    assert vis0.size and np.all(vis0.view(np.uint32) == 0)


@pytest.mark.parametrize("dtype", DTYPES)
def test_scores_homogeneous_chunked_and_nan_safe(dtype):
    rng = np.random.default_rng(131)
    B, S, NB = 3, 33, 9
    q = t_bits(rng.standard_normal((B, S, 4, 128)), dtype)
    kb = t_bits(rng.standard_normal((B, NB, 128)), dtype)
    ctx = np.array([33, 10, 0], np.int32)
    full = oracle.scores(dtype, q, kb, ctx)
    # scaling q by 2 scales every visible logit by exactly 2 (relu is positively homogeneous)
    q2 = t_bits(to_f64(q, dtype) * 2.0, dtype)
    full2 = oracle.scores(dtype, q2, kb, ctx)
    vis = full != NEG_MAX
    assert np.array_equal(full2[vis], 2 * full[vis]) and np.array_equal(full2[~vis], full[~vis])
    # chunked rows are the same rows
    for start, n in ((0, 5), (5, 40), (45, 54), (98, 1), (0, 0)):
        part = oracle.scores(dtype, q, kb, ctx, start, n)
        assert np.array_equal(part.view(np.uint32), full[start:start + n].view(np.uint32))
    # padded rows and invisible blocks are never read
    qn = q.copy()
    kbn = kb.copy()
    for b in range(B):
        qn[b, ctx[b]:] = workloads.NAN_BITS[dtype]
        kbn[b, max(0, int(ctx[b]) // 4):] = workloads.NAN_BITS[dtype]
    got = oracle.scores(dtype, qn, kbn, ctx)
    assert np.array_equal(got.view(np.uint32), full.view(np.uint32))
    # mask structure: row t of sequence b shows min(NB, (t+1)//4) blocks iff t < ctx_b
    for r in range(B * S):
        b, t = divmod(r, S)
        nvis = min(NB, (t + 1) // 4) if t < ctx[b] else 0
        assert int(np.sum(full[r] != NEG_MAX)) == nvis
        assert np.all(full[r, nvis:].view(np.uint32) == np.uint32(0xFF7FFFFF))


# ----------------------------------------------------------- prefill selection

def test_orderable_map_is_monotone_and_splits_signed_zero():
    vals = np.array([0.0, -0.0, 1.0, -1.0], np.float32)
    assert oracle.orderable(vals).tolist() == [0x80000000, 0x7FFFFFFF, 0xBF800000, 0x407FFFFF]
    rng = np.random.default_rng(141)
    x = np.sort(np.concatenate([rng.standard_normal(5000).astype(np.float32) * 1e3,
                                np.array([np.finfo(np.float32).max, -np.finfo(np.float32).max,
                                          np.finfo(np.float32).tiny, -np.finfo(np.float32).tiny], np.float32)]))
    u = oracle.orderable(x).astype(np.int64)
    assert np.all(np.diff(u) >= 0)
    assert np.all((np.diff(u) > 0) == (np.diff(x) > 0))


def test_ids_fill_closed_form():
    ids = oracle.ids_fill(3, 7)
    assert np.array_equal(ids, np.tile(np.arange(7, dtype=np.int32), (3, 1)))


def test_expand_row_hand_cases():
    with open(os.path.join(GOLDEN, "expand_rows.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        out = oracle.expand_row(np.array(c["sorted_ids"], np.int32), c["t"], c["ctx"])
        prefix = np.array(c["prefix"], np.int32)
        assert np.array_equal(out[:len(prefix)], prefix), c
        assert np.all(out[len(prefix):] == -1), c


def _check_selection_row(out, logits_row, t, ctx):
    """Properties any correct prefill selection has (independent of how it sorts)."""
    if ctx <= 0 or t >= ctx:
        assert np.all(out == -1)
        return
    nvis = (t + 1) // 4
    ksel = min(512, nvis)
    tail = (t + 1) % 4
    used = out[out >= 0]
    assert used.size == 4 * ksel + tail and np.all(out[used.size:] == -1)
    assert len(set(used.tolist())) == used.size and used.min() >= 0 and used.max() <= t
    blocks = out[:4 * ksel:4] // 4
    assert np.array_equal(out[:4 * ksel].reshape(-1, 4), blocks[:, None] * 4 + np.arange(4))
    assert np.array_equal(out[4 * ksel:4 * ksel + tail], 4 * nvis + np.arange(tail))
    u = oracle.orderable(logits_row[:nvis]).astype(np.int64)
    sel = u[blocks]
    # emitted in descending key order, equal keys by ascending block id
    for a, b, ua, ub in zip(blocks[:-1], blocks[1:], sel[:-1], sel[1:]):
        assert ua > ub or (ua == ub and a < b)
    # every selected key >= every unselected key; at the threshold, the lowest ids win
    rest = np.setdiff1d(np.arange(nvis), blocks)
    if rest.size:
        thr = sel.min()
        assert u[rest].max() <= thr
        tied_rest = rest[u[rest] == thr]
        tied_sel = blocks[sel == thr]
        if tied_rest.size:
            assert tied_sel.max() < tied_rest.min()


def test_select_expand_closed_forms_and_properties():
    NB = 700
    t = 4 * NB - 1                                   # nVis = 700 > 512
    dec = np.linspace(10.0, 1.0, NB, dtype=np.float32)
    out = oracle.select_expand_row(dec, t, t + 1)
    assert np.array_equal(out[:2048:4] // 4, np.arange(512))
    inc = dec[::-1].copy()
    out = oracle.select_expand_row(inc, t, t + 1)
    assert np.array_equal(out[:2048:4] // 4, np.arange(NB - 1, NB - 513, -1))
    flat = np.full(NB, 2.5, np.float32)
    out = oracle.select_expand_row(flat, t, t + 1)
    assert np.array_equal(out[:2048:4] // 4, np.arange(512))   # stable: ascending ids
    rng = np.random.default_rng(151)
    neg = np.float32(-np.finfo(np.float32).max)
    for trial in range(60):
        NB = int(rng.integers(1, 900))
        S = 4 * NB
        t = int(rng.integers(0, S))
        ctx = int(rng.integers(0, S + 1))
        vals = rng.choice([0.0, 0.25, 1.0, 3.0], NB) if trial % 2 else rng.random(NB) * 4
        row = vals.astype(np.float32)
        row[(t + 1) // 4:] = neg
        out = oracle.select_expand_row(row, t, ctx)
        _check_selection_row(out, row, t, ctx)


def test_select_expand_rows_and_golden():
    with open(os.path.join(GOLDEN, "select_rows.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        out = oracle.select_expand_row(np.array(c["logits"], np.float32), c["t"], c["ctx"])
        prefix = np.array(c["prefix"], np.int32)
        assert np.array_equal(out[:len(prefix)], prefix), c
        assert np.all(out[len(prefix):] == -1), c


# ------------------------------------------------------------- decode path

def _decode_sequence(dtype, total, prefill, seed, unused=()):
    """Prefill `prefill` tokens (paged K1b + raw-K tail write), then decode one token at
    a time up to `total`; returns the pool, per-step qNormed and the full workload."""
    import pool_util
    wl = workloads.custom(2, total, [total, total - 3], dtype=dtype, seed=seed, nan_padding=False,
                          max_positions=total)
    pool = pool_util.make_pool(2, total, seed, unused_slots=unused)
    pctx = np.minimum(wl.context_lengths, prefill).astype(np.int32)
    nbp = (prefill + 3) // 4
    iq_pre = np.ascontiguousarray(wl.index_qk[:, :prefill])
    oracle.k_compress_paged(dtype, iq_pre, wl.cos_sin, pctx, wl.w_k, wl.eps, pool, nbp, 0, nbp, 0)
    oracle.raw_k_tail_write_prefill(iq_pre, pctx, pool)
    qs = {}
    for pos in range(prefill, total):
        ctx = np.array([min(pos + 1, c) for c in wl.context_lengths], np.int32)
        active = np.array([pos < c for c in wl.context_lengths])
        ctx = np.where(active, ctx, 0).astype(np.int32)
        rows = np.ascontiguousarray(wl.index_qk[:, pos])
        qs[pos] = (ctx, oracle.pre_decode(dtype, rows, wl.cos_sin, ctx, wl.w_q, wl.w_k, wl.eps, pool))
    return wl, pool, qs


@pytest.mark.parametrize("dtype", DTYPES)
def test_decode_compress_bit_identical_to_prefill_and_addressing(dtype):
    import pool_util
    total, prefill = 300, 133
    wl, pool, qs = _decode_sequence(dtype, total, prefill, seed=7)
    NB = total // 4
    full_k = oracle.k_compress(dtype, wl.index_qk, wl.cos_sin, wl.context_lengths, wl.w_k, wl.eps,
                               (total + 3) // 4, 0, (total + 3) // 4, 0)
    full_q = oracle.q_prep(dtype, wl.index_qk, wl.cos_sin, wl.context_lengths, wl.w_q, wl.eps)
    for b in range(2):
        c = int(wl.context_lengths[b])
        for g in range(c // 4):           # every completed block, prefill or decode made
            assert np.array_equal(pool_util.v_tail(pool, b, g), full_k[b, g]), (b, g)
        for g in range(c // 4, NB):        # never completed: the V-tail row is untouched
            assert np.all(pool_util.v_tail(pool, b, g) == 0x5A5A)
        for t in range(c - c % 4, c):      # raw keys of the open block, bit for bit
            assert np.array_equal(pool_util.k_tail(pool, b, t), wl.index_qk[b, t, 512:])
        for pos in range(prefill, c):
            assert np.array_equal(qs[pos][1][b, 0], full_q[b, pos]), (b, pos)


@pytest.mark.parametrize("dtype", DTYPES)
def test_decode_scores_and_selection_match_prefill(dtype):
    import pool_util
    total, prefill = 2300, 2100
    wl, pool, qs = _decode_sequence(dtype, total, prefill, seed=9)
    full_q = oracle.q_prep(dtype, wl.index_qk, wl.cos_sin, wl.context_lengths, wl.w_q, wl.eps)
    NB = (total + 3) // 4
    full_k = oracle.k_compress(dtype, wl.index_qk, wl.cos_sin, wl.context_lengths, wl.w_k, wl.eps, NB, 0, NB, 0)
    maxb = NB + 5
    for pos in (prefill, prefill + 1, prefill + 3, total - 1):
        ctx, q = qs[pos]
        lg = oracle.scores_decode(dtype, q, ctx, pool, maxb)
        sc = np.full((2, 2), 9, np.int32)
        sel = oracle.topk_expand_decode(lg, ctx, sc)
        assert not sc.any()
        for b in range(2):
            if ctx[b] <= 0:
                assert np.all(sel[b] == -1)
                continue
            t = int(ctx[b]) - 1
            nvis = int(ctx[b]) // 4
            ref = oracle.scores_row(dtype, full_q[b, t], full_k[b], t, int(ctx[b]))
            assert np.array_equal(lg[b, :nvis].view(np.uint32), ref[:nvis].view(np.uint32))
            assert np.all(np.isnan(lg[b, nvis:]))                       # only the prefix written
            pre = oracle.select_expand_row(ref, t, int(ctx[b]))
            n = int((pre >= 0).sum())
            assert int((sel[b] >= 0).sum()) == n and np.all(sel[b][n:] == -1)
            k = 4 * min(512, nvis)
            assert np.array_equal(np.sort(sel[b][:k]), np.sort(pre[:k]))  # identical block sets
            assert np.all(np.diff(sel[b][:k:4]) > 0)                    # ascending block order
            assert np.array_equal(sel[b][k:n], pre[k:n])                # the open block's tokens


def test_unused_page_entries_are_never_dereferenced():
    import pool_util
    dtype = "bf16"
    total, prefill = 520, 300
    # sequence 0: its K page slot 1 and V page slot 2 are unused
    wl, pool, qs = _decode_sequence(dtype, total, prefill, seed=13, unused=((0, 0, 1), (0, 1, 2)))
    table = pool.page_table
    used = set(table[table >= 0].ravel().tolist())
    unused_pages = [p for p in range(2 * pool.num_pages) if p not in used]
    assert np.all(pool.pool[unused_pages] == 0x5A5A)                   # nothing landed elsewhere
    # blocks whose V slot is unused score -FLT_MAX in decode
    ctx, q = qs[total - 1]
    lg = oracle.scores_decode(dtype, q, ctx, pool, total // 4 + 2)
    g_unused = [g for g in range(ctx[0] // 4) if (4 * g) // 128 == 2]
    assert g_unused and np.all(lg[0, g_unused] == NEG_MAX)
