"""CPU oracle for the QSA indexer hot path -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(and its ``--impl reference`` arm) may import this package.  The product path
(``sparse_attention_indexer_qsa_gb300``) never imports it and shares no code
with it.

The arithmetic lives in ``qsa_oracle.c`` (plain C, binary32 per-operation
rounding, ``-ffp-contract=off``), restated from the "Qsa Indexer Kernels" page
(launchQsaIndexQPrep, launchQsaIndexKCompress, launchQsaIndexScores).  This
module only builds that file with gcc and marshals numpy arrays into it.

Arrays of the 2-byte activation type T are passed as ``np.uint16`` bit patterns
(bf16 or fp16, chosen by ``dtype`` = "bf16" | "fp16").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_qsa.so")

# The flags are part of the oracle's definition: IEEE binary32 with one rounding
# per operation (no contraction into FMA, no fast-math reassociation).
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fexcess-precision=standard", "-Wall", "-Wextra"]

DTYPES = {"bf16": 0, "fp16": 1}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``qsa_oracle.c`` into ``_build/liboracle_qsa.so`` (gcc, a second)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # QSA_ORACLE_LIBRARY: a build of a deliberately altered qsa_oracle.c, loaded
        # instead of the real one by tests/test_oracle_mutants.py to show that the pins
        # catch each alteration
        lib = ctypes.CDLL(os.environ.get("QSA_ORACLE_LIBRARY") or build())
        p = ctypes.c_void_p
        i32 = ctypes.c_int32
        f32 = ctypes.c_float
        lib.qsa_oracle_t_to_f32.argtypes = [ctypes.c_int, ctypes.c_uint16]
        lib.qsa_oracle_t_to_f32.restype = f32
        lib.qsa_oracle_f32_to_t.argtypes = [ctypes.c_int, f32]
        lib.qsa_oracle_f32_to_t.restype = ctypes.c_uint16
        lib.qsa_oracle_t_to_f32_array.argtypes = [ctypes.c_int, p, p, ctypes.c_int64]
        lib.qsa_oracle_t_to_f32_array.restype = None
        lib.qsa_oracle_f32_to_t_array.argtypes = [ctypes.c_int, p, p, ctypes.c_int64]
        lib.qsa_oracle_f32_to_t_array.restype = None
        lib.qsa_oracle_norm_rope.argtypes = [ctypes.c_int, p, p, f32, p, p]
        lib.qsa_oracle_norm_rope.restype = None
        lib.qsa_oracle_block_mean.argtypes = [ctypes.c_int, p, p, p, p, p]
        lib.qsa_oracle_block_mean.restype = None
        lib.qsa_oracle_q_prep.argtypes = [ctypes.c_int, p, p, p, p, p, f32, i32, i32]
        lib.qsa_oracle_q_prep.restype = ctypes.c_int
        lib.qsa_oracle_block_valid.argtypes = [i32, i32, i32, i32]
        lib.qsa_oracle_block_valid.restype = ctypes.c_int
        lib.qsa_oracle_k_compress.argtypes = [ctypes.c_int, p, p, p, p, p, f32,
                                              i32, i32, i32, i32, i32, i32]
        lib.qsa_oracle_k_compress.restype = ctypes.c_int
        lib.qsa_oracle_scores_row.argtypes = [ctypes.c_int, p, p, p, i32, i32, i32]
        lib.qsa_oracle_scores_row.restype = None
        lib.qsa_oracle_scores.argtypes = [ctypes.c_int, p, p, p, p, i32, i32, i32, i32, i32]
        lib.qsa_oracle_scores.restype = ctypes.c_int
        lib.qsa_oracle_orderable.argtypes = [f32]
        lib.qsa_oracle_orderable.restype = ctypes.c_uint32
        lib.qsa_oracle_ids_fill.argtypes = [p, i32, i32]
        lib.qsa_oracle_ids_fill.restype = None
        lib.qsa_oracle_expand_row.argtypes = [p, p, i32, i32]
        lib.qsa_oracle_expand_row.restype = None
        lib.qsa_oracle_select_expand_row.argtypes = [p, p, i32, i32, i32, p]
        lib.qsa_oracle_select_expand_row.restype = None
        lib.qsa_oracle_select_expand.argtypes = [p, p, p, i32, i32, i32, i32, i32, p]
        lib.qsa_oracle_select_expand.restype = ctypes.c_int
        pp = ctypes.POINTER(PoolState)
        lib.qsa_oracle_k_compress_paged.argtypes = [ctypes.c_int, p, p, p, p, p, f32, pp,
                                                    i32, i32, i32, i32, i32, i32]
        lib.qsa_oracle_k_compress_paged.restype = ctypes.c_int
        lib.qsa_oracle_raw_k_tail_write_prefill.argtypes = [p, p, pp, i32, i32]
        lib.qsa_oracle_raw_k_tail_write_prefill.restype = ctypes.c_int
        lib.qsa_oracle_pre_decode.argtypes = [ctypes.c_int, p, p, p, p, p, p, f32, pp, i32]
        lib.qsa_oracle_pre_decode.restype = ctypes.c_int
        lib.qsa_oracle_scores_decode.argtypes = [ctypes.c_int, p, p, p, pp, i32, i32]
        lib.qsa_oracle_scores_decode.restype = ctypes.c_int
        lib.qsa_oracle_topk_expand_decode.argtypes = [p, p, p, p, i32, i32, i32, p]
        lib.qsa_oracle_topk_expand_decode.restype = ctypes.c_int
        _lib = lib
        return lib


class PoolState(ctypes.Structure):
    """Mirror of the oracle's pool descriptor (pool, pageTable, sizes)."""
    _fields_ = [("pool", ctypes.c_void_p), ("pageTable", ctypes.c_void_p),
                ("maxPagesPerSeq", ctypes.c_int32), ("numPages", ctypes.c_int32),
                ("numKVHeads", ctypes.c_int32), ("poolHeadDim", ctypes.c_int32),
                ("headSize", ctypes.c_int32)]


class Pool:
    """A host copy of a paged indexer pool: pool [2*numPages, 128, numKVHeads,
    poolHeadDim] uint16 and pageTable [B, 2, maxPagesPerSeq] int32 (V ids already
    offset by +numPages, -1 = unused)."""

    def __init__(self, pool, page_table, num_pages, num_kv_heads=2, pool_head_dim=384, head_size=256):
        self.pool = np.ascontiguousarray(pool, dtype=np.uint16)
        self.page_table = np.ascontiguousarray(page_table, dtype=np.int32)
        self.num_pages = num_pages
        self.num_kv_heads = num_kv_heads
        self.pool_head_dim = pool_head_dim
        self.head_size = head_size

    def state(self):
        return PoolState(self.pool.ctypes.data, self.page_table.ctypes.data, self.page_table.shape[2],
                         self.num_pages, self.num_kv_heads, self.pool_head_dim, self.head_size)


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, f"expected uint16 bit patterns, got {a.dtype}"
    return a


def _f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


# ------------------------------------------------------------------ conversions

def t_to_f32(dtype: str, bits) -> np.ndarray:
    """Widen T bit patterns to binary32 (exact)."""
    lib = _load()
    flat = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16).ravel())
    out = np.empty(flat.shape, np.float32)
    lib.qsa_oracle_t_to_f32_array(DTYPES[dtype], _ptr(flat), _ptr(out), flat.size)
    return out.reshape(np.shape(bits))


def f32_to_t(dtype: str, values) -> np.ndarray:
    """Round binary32 values to T (round to nearest, ties to even)."""
    lib = _load()
    flat = np.ascontiguousarray(np.asarray(values, dtype=np.float32).ravel())
    out = np.empty(flat.shape, np.uint16)
    lib.qsa_oracle_f32_to_t_array(DTYPES[dtype], _ptr(flat), _ptr(out), flat.size)
    return out.reshape(np.shape(values))


# -------------------------------------------------------------- per-vector steps

def norm_rope(dtype: str, x, w, eps: float, cs_row) -> np.ndarray:
    """One 128-vector: RMS norm with (1 + w), partial neox rope with cs_row [64], cast."""
    lib = _load()
    x = _f32(x)
    w = _u16(w)
    cs = _f32(cs_row)
    assert x.shape == (128,) and w.shape == (128,) and cs.shape == (64,)
    out = np.empty(128, np.uint16)
    lib.qsa_oracle_norm_rope(DTYPES[dtype], _ptr(x), _ptr(w), float(eps), _ptr(cs), _ptr(out))
    return out


def block_mean(dtype: str, k0, k1, k2, k3) -> np.ndarray:
    """Fixed-order mean of four K rows, cast to T."""
    lib = _load()
    ks = [_u16(k) for k in (k0, k1, k2, k3)]
    out = np.empty(128, np.uint16)
    lib.qsa_oracle_block_mean(DTYPES[dtype], *(_ptr(k) for k in ks), _ptr(out))
    return out


def block_valid(g: int, ctx: int, seq_len: int, past_len: int) -> bool:
    return bool(_load().qsa_oracle_block_valid(g, ctx, seq_len, past_len))


# ------------------------------------------------------------------ whole steps

def q_prep(dtype: str, index_qk, cos_sin, context_lengths, w_q, eps: float) -> np.ndarray:
    """K1a: indexQk [B, S, 640] -> qNormed [B, S, 4, 128] (T bit patterns)."""
    lib = _load()
    iq = _u16(index_qk)
    B, S, W = iq.shape
    assert W == 640
    cs = _f32(cos_sin)
    ctx = _i32(context_lengths)
    w = _u16(w_q)
    out = np.empty((B, S, 4, 128), np.uint16)
    rc = lib.qsa_oracle_q_prep(DTYPES[dtype], _ptr(out), _ptr(iq), _ptr(cs), _ptr(ctx), _ptr(w),
                               float(eps), B, S)
    assert rc == 0
    return out


def k_compress(dtype: str, index_qk, cos_sin, context_lengths, w_k, eps: float,
               num_blocks: int, block_begin: int, block_end: int, past_len: int,
               kbar_init=None) -> np.ndarray:
    """K1b: writes rows [block_begin, block_end) of kbar [B, num_blocks, 128].

    Rows outside the range keep the contents of ``kbar_init`` (zeros if None).
    """
    lib = _load()
    iq = _u16(index_qk)
    B, S, W = iq.shape
    assert W == 640
    cs = _f32(cos_sin)
    ctx = _i32(context_lengths)
    w = _u16(w_k)
    if kbar_init is None:
        out = np.zeros((B, num_blocks, 128), np.uint16)
    else:
        out = np.array(kbar_init, dtype=np.uint16, copy=True, order="C")
        assert out.shape == (B, num_blocks, 128)
    rc = lib.qsa_oracle_k_compress(DTYPES[dtype], _ptr(out), _ptr(iq), _ptr(cs), _ptr(ctx),
                                   _ptr(w), float(eps), B, S, num_blocks, block_begin,
                                   block_end, past_len)
    assert rc == 0
    return out


def scores(dtype: str, q_normed, kbar, context_lengths, row_start: int = 0,
           num_rows: int | None = None) -> np.ndarray:
    """K2: logits [num_rows, numBlocks] FP32 for global rows [row_start, row_start+num_rows)."""
    lib = _load()
    q = _u16(q_normed)
    kb = _u16(kbar)
    B, S = q.shape[:2]
    assert q.shape[2:] == (4, 128)
    NB = kb.shape[1]
    ctx = _i32(context_lengths)
    if num_rows is None:
        num_rows = B * S - row_start
    out = np.empty((num_rows, NB), np.float32)
    rc = lib.qsa_oracle_scores(DTYPES[dtype], _ptr(out), _ptr(q), _ptr(kb), _ptr(ctx), B, S, NB,
                               row_start, num_rows)
    assert rc == 0
    return out


def scores_row(dtype: str, q_row, kbar_b, t: int, ctx: int) -> np.ndarray:
    """K2 for one query row: q_row [4, 128], kbar_b [numBlocks, 128] -> [numBlocks] FP32."""
    lib = _load()
    q = _u16(q_row)
    kb = _u16(kbar_b)
    assert q.shape == (4, 128)
    NB = kb.shape[0]
    out = np.empty(NB, np.float32)
    lib.qsa_oracle_scores_row(DTYPES[dtype], _ptr(out), _ptr(q), _ptr(kb), int(t), int(ctx), NB)
    return out


# ------------------------------------------------------------ prefill selection

INDEX_WIDTH = 2051   # 512 blocks x 4 tokens + 3 tail tokens
TOPK_BLOCKS = 512


def orderable(values) -> np.ndarray:
    """Order-preserving uint32 map of binary32 values (bits >= 0 ? bits | 2^31 : ~bits)."""
    lib = _load()
    return np.array([lib.qsa_oracle_orderable(float(v)) for v in np.asarray(values, np.float32).ravel()],
                    np.uint32)


def ids_fill(num_rows: int, num_blocks: int) -> np.ndarray:
    lib = _load()
    out = np.empty((num_rows, num_blocks), np.int32)
    lib.qsa_oracle_ids_fill(_ptr(out), num_rows, num_blocks)
    return out


def expand_row(sorted_ids, t: int, ctx: int) -> np.ndarray:
    lib = _load()
    ids = _i32(sorted_ids)
    out = np.empty(INDEX_WIDTH, np.int32)
    lib.qsa_oracle_expand_row(_ptr(out), _ptr(ids), int(t), int(ctx))
    return out


def select_expand_row(logits_row, t: int, ctx: int) -> np.ndarray:
    """Prefill selection of one row: stable descending sort + expand -> [2051] int32."""
    lib = _load()
    row = _f32(logits_row)
    n = row.shape[0]
    scratch = np.empty(4 * max(n, 1), np.uint32)
    out = np.empty(INDEX_WIDTH, np.int32)
    lib.qsa_oracle_select_expand_row(_ptr(out), _ptr(row), n, int(t), int(ctx), _ptr(scratch))
    return out


def select_expand(logits, context_lengths, B: int, S: int, row_start: int = 0,
                  out_idx=None) -> np.ndarray:
    """Rows [row_start, row_start + len(logits)) of outIdx [B*S, 2051]; other rows keep
    out_idx's contents (zeros if None)."""
    lib = _load()
    lg = _f32(logits)
    num_rows, nb = lg.shape
    ctx = _i32(context_lengths)
    out = np.zeros((B * S, INDEX_WIDTH), np.int32) if out_idx is None else np.array(out_idx, np.int32, copy=True)
    scratch = np.empty(4 * max(nb, 1), np.uint32)
    rc = lib.qsa_oracle_select_expand(_ptr(out), _ptr(lg), _ptr(ctx), B, S, nb, row_start, num_rows,
                                      _ptr(scratch))
    assert rc == 0
    return out


# ------------------------------------------------------ paged pool, decode path

def k_compress_paged(dtype, index_qk, cos_sin, context_lengths, w_k, eps, pool: Pool, num_blocks,
                     block_begin, block_end, past_len, kbar_init=None):
    """K1b-paged: returns kbar; pool.pool is updated in place (V-tails of valid blocks)."""
    lib = _load()
    iq = _u16(index_qk)
    B, S, _ = iq.shape
    out = (np.zeros((B, num_blocks, 128), np.uint16) if kbar_init is None
           else np.array(kbar_init, np.uint16, copy=True))
    st = pool.state()
    rc = lib.qsa_oracle_k_compress_paged(DTYPES[dtype], _ptr(out), _ptr(iq), _ptr(_f32(cos_sin)),
                                         _ptr(_i32(context_lengths)), _ptr(_u16(w_k)), float(eps),
                                         ctypes.byref(st), B, S, num_blocks, block_begin, block_end, past_len)
    assert rc == 0
    return out


def raw_k_tail_write_prefill(index_qk, context_lengths, pool: Pool):
    lib = _load()
    iq = _u16(index_qk)
    B, S, _ = iq.shape
    st = pool.state()
    assert lib.qsa_oracle_raw_k_tail_write_prefill(_ptr(iq), _ptr(_i32(context_lengths)), ctypes.byref(st),
                                                   B, S) == 0


def pre_decode(dtype, index_qk_rows, cos_sin, context_lengths, w_q, w_k, eps, pool: Pool):
    """B1: index_qk_rows [B, 640] (one new token each) -> qNormed [B, 1, 4, 128]; pool updated."""
    lib = _load()
    iq = _u16(index_qk_rows).reshape(-1, 640)
    B = iq.shape[0]
    q = np.empty((B, 1, 4, 128), np.uint16)
    st = pool.state()
    assert lib.qsa_oracle_pre_decode(DTYPES[dtype], _ptr(q), _ptr(iq), _ptr(_f32(cos_sin)),
                                     _ptr(_i32(context_lengths)), _ptr(_u16(w_q)), _ptr(_u16(w_k)),
                                     float(eps), ctypes.byref(st), B) == 0
    return q


def scores_decode(dtype, q_normed, context_lengths, pool: Pool, max_blocks, logits_init=None):
    """B2: logits [B, max_blocks]; only [0, ctx/4) of each row is written."""
    lib = _load()
    q = _u16(q_normed).reshape(-1, 4, 128)
    B = q.shape[0]
    out = (np.full((B, max_blocks), np.nan, np.float32) if logits_init is None
           else np.array(logits_init, np.float32, copy=True))
    st = pool.state()
    assert lib.qsa_oracle_scores_decode(DTYPES[dtype], _ptr(out), _ptr(q), _ptr(_i32(context_lengths)),
                                        ctypes.byref(st), B, max_blocks) == 0
    return out


def topk_expand_decode(logits, context_lengths, split_counters=None, num_kv_heads=2):
    """B3: outIdx [B, 2051] (and split_counters zeroed in place when given)."""
    lib = _load()
    lg = _f32(logits)
    B, maxb = lg.shape
    out = np.empty((B, INDEX_WIDTH), np.int32)
    scratch = np.empty(4 * max(maxb, 1), np.uint32)
    sc = 0 if split_counters is None else _ptr(split_counters)
    assert lib.qsa_oracle_topk_expand_decode(_ptr(out), _ptr(lg), _ptr(_i32(context_lengths)), sc,
                                             num_kv_heads, B, maxb, _ptr(scratch)) == 0
    return out
