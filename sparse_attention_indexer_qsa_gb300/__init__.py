"""GB300 (sm_103a) QSA sparse-attention indexer: K1a q-prep, K1b K-compress, K2 scores.

A thin ctypes binding over the C ABI in ``include/qsa_indexer.h``; every step of
the computation runs in the library's CUDA kernels.  The functions keep the C
names and argument order.  Array arguments are torch CUDA tensors (or raw
device addresses as ints, with ``dtype`` given); the stream defaults to torch's
current stream.  A non-zero status raises :class:`QsaError`.

There is no CPU fallback: if ``_build/libqsa_indexer.so`` is missing, every call
(and ``load()``) raises.  Build it with ``python -m sparse_attention_indexer_qsa_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

__all__ = [
    "QsaError", "QSA_BF16", "QSA_F16", "load", "lib", "qsa_abi_version", "qsa_last_error",
    "qsa_index_q_prep", "qsa_index_k_compress", "qsa_index_qk_prep", "qsa_index_scores",
    "qsa_index_scores_no_alloc", "qsa_index_ids_fill", "qsa_index_expand", "qsa_index_topk_expand",
    "qsa_index_scores_topk_expand", "PoolState", "pool_state", "qsa_index_k_compress_paged", "qsa_raw_k_tail_write_prefill",
    "qsa_indexer_pre_decode", "qsa_index_scores_decode", "qsa_topk_expand_decode",
    "qsa_indexer_decode_step", "qsa_device_fault_flags",
    "qsa_testing_index_scores_cuda_core", "qsa_testing_bounded_wait_probe", "qsa_testing_stream_yardstick",
    "qsa_testing_gather_yardstick", "qsa_testing_decode_step_histograms", "LIB_PATH",
]

QSA_BF16 = 0
QSA_F16 = 1
STATUS_NAMES = {0: "QSA_OK", -1: "QSA_E_NULL", -2: "QSA_E_SHAPE", -3: "QSA_E_RANGE",
                -4: "QSA_E_DTYPE", -5: "QSA_E_ALIGN", -6: "QSA_E_CUDA", -7: "QSA_E_DEVICE"}
EXPORTED = ["qsa_abi_version", "qsa_last_error", "qsa_index_q_prep", "qsa_index_k_compress",
            "qsa_index_qk_prep", "qsa_index_ids_fill", "qsa_index_expand", "qsa_index_topk_expand",
            "qsa_index_scores_topk_expand", "qsa_index_k_compress_paged", "qsa_raw_k_tail_write_prefill", "qsa_indexer_pre_decode",
            "qsa_index_scores_decode", "qsa_topk_expand_decode", "qsa_indexer_decode_step",
            "qsa_index_scores", "qsa_index_scores_no_alloc", "qsa_device_fault_flags",
            "qsa_testing_index_scores_cuda_core", "qsa_testing_bounded_wait_probe", "qsa_testing_stream_yardstick",
            "qsa_testing_gather_yardstick", "qsa_testing_decode_step_histograms"]


class QsaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class PoolState(ctypes.Structure):
    """qsa_pool_state_t: the paged indexer pool (device pointers, host struct)."""
    _fields_ = [("poolPtr", ctypes.c_void_p), ("pageTable", ctypes.c_void_p),
                ("maxPagesPerSeq", ctypes.c_int32), ("numPages", ctypes.c_int32),
                ("numKVHeads", ctypes.c_int32), ("poolHeadDim", ctypes.c_int32),
                ("headSize", ctypes.c_int32)]


def pool_state(pool, pageTable, numPages, numKVHeads=2, poolHeadDim=384, headSize=256) -> PoolState:
    """Describe a device pool [2*numPages, 128, numKVHeads, poolHeadDim] and its page table
    [B, 2, maxPagesPerSeq] (V ids offset by +numPages, -1 = unused)."""
    max_pages = pageTable.shape[-1] if hasattr(pageTable, "shape") else int(pageTable[1])
    return PoolState(_addr(pool), _addr(pageTable), int(max_pages), int(numPages), int(numKVHeads),
                     int(poolHeadDim), int(headSize))


_lib = None


def load():
    """Load the CUDA library (once).  Raises if it has not been built: no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run "
                          "`python -m sparse_attention_indexer_qsa_gb300.build` (nvcc, sm_103a)")
    L = ctypes.CDLL(LIB_PATH)
    p = ctypes.c_void_p
    i32 = ctypes.c_int32
    f32 = ctypes.c_float
    L.qsa_abi_version.argtypes = []
    L.qsa_abi_version.restype = ctypes.c_int
    L.qsa_last_error.argtypes = []
    L.qsa_last_error.restype = ctypes.c_char_p
    L.qsa_index_q_prep.argtypes = [ctypes.c_int, p, p, p, p, p, f32, i32, i32, p]
    L.qsa_index_q_prep.restype = ctypes.c_int
    L.qsa_index_k_compress.argtypes = [ctypes.c_int, p, p, p, p, p, f32, i32, i32, i32,
                                       i32, i32, i32, p]
    L.qsa_index_k_compress.restype = ctypes.c_int
    L.qsa_index_qk_prep.argtypes = [ctypes.c_int, p, p, p, p, p, p, p, f32, i32, i32, i32, p]
    L.qsa_index_qk_prep.restype = ctypes.c_int
    L.qsa_index_ids_fill.argtypes = [p, i32, i32, p]
    L.qsa_index_ids_fill.restype = ctypes.c_int
    L.qsa_index_expand.argtypes = [p, p, p, i32, i32, i32, i32, i32, p]
    L.qsa_index_expand.restype = ctypes.c_int
    L.qsa_index_topk_expand.argtypes = [p, p, p, i32, i32, i32, i32, i32, p]
    L.qsa_index_topk_expand.restype = ctypes.c_int
    L.qsa_index_scores_topk_expand.argtypes = [ctypes.c_int, p, p, p, p, i32, i32, i32, i32, i32, p]
    L.qsa_index_scores_topk_expand.restype = ctypes.c_int
    pp = ctypes.POINTER(PoolState)
    L.qsa_index_k_compress_paged.argtypes = [ctypes.c_int, p, p, p, p, p, f32, pp, i32, i32, i32, i32, i32, i32, p]
    L.qsa_index_k_compress_paged.restype = ctypes.c_int
    L.qsa_raw_k_tail_write_prefill.argtypes = [ctypes.c_int, p, p, pp, i32, i32, p]
    L.qsa_raw_k_tail_write_prefill.restype = ctypes.c_int
    L.qsa_indexer_pre_decode.argtypes = [ctypes.c_int, p, p, p, p, p, p, f32, pp, i32, p]
    L.qsa_indexer_pre_decode.restype = ctypes.c_int
    L.qsa_index_scores_decode.argtypes = [ctypes.c_int, p, p, p, pp, i32, i32, p]
    L.qsa_index_scores_decode.restype = ctypes.c_int
    L.qsa_topk_expand_decode.argtypes = [p, p, p, p, i32, i32, i32, p]
    L.qsa_topk_expand_decode.restype = ctypes.c_int
    L.qsa_indexer_decode_step.argtypes = [ctypes.c_int, p, p, p, p, p, p, p, p, f32, pp, p, i32, i32, i32, p]
    L.qsa_indexer_decode_step.restype = ctypes.c_int
    L.qsa_index_scores.argtypes = [ctypes.c_int, p, p, p, p, i32, i32, i32, i32, i32, p]
    L.qsa_index_scores.restype = ctypes.c_int
    L.qsa_index_scores_no_alloc.argtypes = list(L.qsa_index_scores.argtypes)
    L.qsa_index_scores_no_alloc.restype = ctypes.c_int
    L.qsa_testing_index_scores_cuda_core.argtypes = list(L.qsa_index_scores.argtypes)
    L.qsa_testing_index_scores_cuda_core.restype = ctypes.c_int
    L.qsa_testing_bounded_wait_probe.argtypes = [i32, p]
    L.qsa_testing_bounded_wait_probe.restype = ctypes.c_int
    L.qsa_testing_decode_step_histograms.argtypes = [i32, p]
    L.qsa_testing_decode_step_histograms.restype = ctypes.c_int
    i64 = ctypes.c_int64
    L.qsa_testing_stream_yardstick.argtypes = [p, p, i64, i32, i64, i64, i64, i32, p]
    L.qsa_testing_stream_yardstick.restype = ctypes.c_int
    L.qsa_testing_gather_yardstick.argtypes = [p, p, i64, i64, i64, i32, p]
    L.qsa_testing_gather_yardstick.restype = ctypes.c_int
    L.qsa_device_fault_flags.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, p]
    L.qsa_device_fault_flags.restype = ctypes.c_int
    _lib = L
    return L


def __getattr__(name):
    if name == "lib":
        return load()
    raise AttributeError(name)


def qsa_abi_version() -> int:
    return int(load().qsa_abi_version())


def qsa_last_error() -> str:
    return load().qsa_last_error().decode()


def _addr(x) -> int | None:
    """Device address of a tensor argument.  The C ABI takes dense row-major device
    arrays, so a host tensor (whose address a kernel would dereference as a device
    address) or a non-contiguous view (whose strides the kernels would ignore) is
    rejected here, before anything is enqueued.  Plain ints pass through as raw
    device addresses."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if getattr(x, "is_cuda", True) is False:
        raise ValueError(f"expected a CUDA tensor (a device array), got one on {x.device}")
    if hasattr(x, "is_contiguous") and not x.is_contiguous():
        raise ValueError("expected a contiguous tensor: the C ABI takes dense row-major arrays")
    return x.data_ptr()


def _dtype(dtype, *tensors) -> int:
    """The T code of a call: ``dtype`` if given, else the type of its bf16/fp16 tensors.
    Every bf16/fp16 tensor of a call must have that one type (bit-pattern tensors of
    other dtypes, and raw addresses, are taken as given)."""
    import torch
    seen = {QSA_BF16 if t.dtype == torch.bfloat16 else QSA_F16 for t in tensors
            if isinstance(t, torch.Tensor) and t.dtype in (torch.bfloat16, torch.float16)}
    if dtype is not None:
        code = {"bf16": QSA_BF16, "fp16": QSA_F16}[dtype] if isinstance(dtype, str) else int(dtype)
        if seen and seen != {code}:
            raise ValueError(f"dtype {dtype!r} does not match the tensors' element type")
        return code
    if len(seen) == 1:
        return seen.pop()
    if len(seen) > 1:
        raise ValueError("the tensors mix bf16 and fp16: every T array of a call has one type")
    raise ValueError("dtype not given and not inferable from the tensors")


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int):
    if status != 0:
        raise QsaError(status, qsa_last_error())


def qsa_index_q_prep(qNormed, indexQk, cosSin, contextLengths, wQ, rmsEps, batchSize, seqLen,
                     stream=None, dtype=None):
    """K1a: indexQk [B, S, 640] -> qNormed [B, S, 4, 128] (see include/qsa_indexer.h)."""
    _check(load().qsa_index_q_prep(_dtype(dtype, indexQk, qNormed, wQ), _addr(qNormed), _addr(indexQk),
                                _addr(cosSin), _addr(contextLengths), _addr(wQ), float(rmsEps),
                                int(batchSize), int(seqLen), _stream(stream)))


def qsa_index_k_compress(kbar, indexQk, cosSin, contextLengths, wK, rmsEps, batchSize, seqLen,
                         numBlocks, blockBegin, blockEnd, pastLen, stream=None, dtype=None):
    """K1b: rows [blockBegin, blockEnd) of kbar [B, numBlocks, 128] (see include/qsa_indexer.h)."""
    _check(load().qsa_index_k_compress(_dtype(dtype, indexQk, kbar, wK), _addr(kbar), _addr(indexQk),
                                    _addr(cosSin), _addr(contextLengths), _addr(wK), float(rmsEps),
                                    int(batchSize), int(seqLen), int(numBlocks), int(blockBegin),
                                    int(blockEnd), int(pastLen), _stream(stream)))


def qsa_index_qk_prep(qNormed, kbar, indexQk, cosSin, contextLengths, wQ, wK, rmsEps, batchSize,
                      seqLen, numBlocks, stream=None, dtype=None):
    """K1a + prefill K1b in one pass over indexQk (see include/qsa_indexer.h)."""
    _check(load().qsa_index_qk_prep(_dtype(dtype, indexQk, qNormed, kbar, wQ, wK), _addr(qNormed), _addr(kbar),
                                 _addr(indexQk), _addr(cosSin), _addr(contextLengths), _addr(wQ),
                                 _addr(wK), float(rmsEps), int(batchSize), int(seqLen), int(numBlocks),
                                 _stream(stream)))


def qsa_index_scores(logits, qNormed, kbar, contextLengths, batchSize, seqLen, numBlocks,
                     rowStart, numRows, stream=None, dtype=None):
    """K2: FP32 logits [numRows, numBlocks] on the tensor cores (see include/qsa_indexer.h)."""
    _check(load().qsa_index_scores(_dtype(dtype, qNormed, kbar), _addr(logits), _addr(qNormed),
                                _addr(kbar), _addr(contextLengths), int(batchSize), int(seqLen),
                                int(numBlocks), int(rowStart), int(numRows), _stream(stream)))


def qsa_index_ids_fill(ids, numRows, numBlocks, stream=None):
    """K3: ids[r, c] = c (see include/qsa_indexer.h)."""
    _check(load().qsa_index_ids_fill(_addr(ids), int(numRows), int(numBlocks), _stream(stream)))


def qsa_index_expand(outIdx, sortedIds, contextLengths, batchSize, seqLen, numBlocks, rowStart, numRows,
                     stream=None):
    """K4: sorted block ids -> 2051 token ids per row (see include/qsa_indexer.h)."""
    _check(load().qsa_index_expand(_addr(outIdx), _addr(sortedIds), _addr(contextLengths), int(batchSize),
                                int(seqLen), int(numBlocks), int(rowStart), int(numRows), _stream(stream)))


def qsa_index_topk_expand(outIdx, logits, contextLengths, batchSize, seqLen, numBlocks, rowStart, numRows,
                          stream=None):
    """Prefill selection in one kernel: radix top-512 + order + expand (see include/qsa_indexer.h)."""
    _check(load().qsa_index_topk_expand(_addr(outIdx), _addr(logits), _addr(contextLengths), int(batchSize),
                                     int(seqLen), int(numBlocks), int(rowStart), int(numRows), _stream(stream)))


def qsa_index_scores_topk_expand(outIdx, qNormed, kbar, contextLengths, batchSize, seqLen, numBlocks, rowStart,
                                 numRows, stream=None, dtype=None):
    """K2 fused with the top-512 selection + expand; no logits written (see include/qsa_indexer.h)."""
    _check(load().qsa_index_scores_topk_expand(_dtype(dtype, qNormed, kbar), _addr(outIdx), _addr(qNormed),
                                            _addr(kbar), _addr(contextLengths), int(batchSize), int(seqLen),
                                            int(numBlocks), int(rowStart), int(numRows), _stream(stream)))


def qsa_index_k_compress_paged(kbar, indexQk, cosSin, contextLengths, wK, rmsEps, pool: PoolState, batchSize,
                               seqLen, numBlocks, blockBegin, blockEnd, pastLen, stream=None, dtype=None):
    """K1b that also persists valid kbar rows to the pool V-tails (see include/qsa_indexer.h)."""
    _check(load().qsa_index_k_compress_paged(_dtype(dtype, indexQk, kbar, wK), _addr(kbar), _addr(indexQk),
                                          _addr(cosSin), _addr(contextLengths), _addr(wK), float(rmsEps),
                                          ctypes.byref(pool), int(batchSize), int(seqLen), int(numBlocks),
                                          int(blockBegin), int(blockEnd), int(pastLen), _stream(stream)))


def qsa_raw_k_tail_write_prefill(indexQk, contextLengths, pool: PoolState, batchSize, seqLen, stream=None,
                                 dtype=None):
    """Raw index-K of each sequence's trailing incomplete block -> pool K-tails."""
    _check(load().qsa_raw_k_tail_write_prefill(_dtype(dtype, indexQk), _addr(indexQk), _addr(contextLengths),
                                            ctypes.byref(pool), int(batchSize), int(seqLen), _stream(stream)))


def qsa_indexer_pre_decode(qNormed, indexQk, cosSin, contextLengths, wQ, wK, rmsEps, pool: PoolState, batchSize,
                           stream=None, dtype=None):
    """Decode pre-pass: q-prep of the new token + K-tail write or block compress."""
    _check(load().qsa_indexer_pre_decode(_dtype(dtype, indexQk, qNormed, wQ, wK), _addr(qNormed), _addr(indexQk),
                                      _addr(cosSin), _addr(contextLengths), _addr(wQ), _addr(wK), float(rmsEps),
                                      ctypes.byref(pool), int(batchSize), _stream(stream)))


def qsa_index_scores_decode(logits, qNormed, contextLengths, pool: PoolState, batchSize, maxBlocks, stream=None,
                            dtype=None):
    """Decode block logits from the pool V-tails (valid prefix [0, ctx/4) only)."""
    _check(load().qsa_index_scores_decode(_dtype(dtype, qNormed), _addr(logits), _addr(qNormed),
                                       _addr(contextLengths), ctypes.byref(pool), int(batchSize), int(maxBlocks),
                                       _stream(stream)))


def qsa_topk_expand_decode(outIdx, logits, contextLengths, splitCounters, numKVHeads, batchSize, maxBlocks,
                           stream=None):
    """Decode top-512 + expand (+ split-counter zeroing)."""
    _check(load().qsa_topk_expand_decode(_addr(outIdx), _addr(logits), _addr(contextLengths), _addr(splitCounters),
                                      int(numKVHeads), int(batchSize), int(maxBlocks), _stream(stream)))


def qsa_indexer_decode_step(outIdx, logits, qNormed, indexQk, cosSin, contextLengths, wQ, wK, rmsEps,
                            pool: PoolState, splitCounters, numKVHeads, batchSize, maxBlocks, stream=None,
                            dtype=None):
    """The decode step in one launch: pre-decode, paged scores, top-512 + expand."""
    _check(load().qsa_indexer_decode_step(_dtype(dtype, indexQk, qNormed, wQ, wK), _addr(outIdx), _addr(logits),
                                       _addr(qNormed), _addr(indexQk), _addr(cosSin), _addr(contextLengths),
                                       _addr(wQ), _addr(wK), float(rmsEps), ctypes.byref(pool),
                                       _addr(splitCounters), int(numKVHeads), int(batchSize), int(maxBlocks),
                                       _stream(stream)))


def qsa_index_scores_no_alloc(logits, qNormed, kbar, contextLengths, batchSize, seqLen, numBlocks,
                              rowStart, numRows, stream=None, dtype=None):
    """K2 with its scratch in one static device array: for callers that cannot allocate
    (see include/qsa_indexer.h; overlapping calls race)."""
    _check(load().qsa_index_scores_no_alloc(_dtype(dtype, qNormed, kbar), _addr(logits), _addr(qNormed),
                                         _addr(kbar), _addr(contextLengths), int(batchSize), int(seqLen),
                                         int(numBlocks), int(rowStart), int(numRows), _stream(stream)))


def qsa_testing_bounded_wait_probe(timeoutMs, stream=None):
    """A bounded wait that runs out on purpose (include/qsa_indexer_testing.h): sets a
    device fault bit after timeoutMs, faults nothing."""
    _check(load().qsa_testing_bounded_wait_probe(int(timeoutMs), _stream(stream)))


def qsa_testing_decode_step_histograms(add, stream=None):
    """Offset (add > 0) or zero (add = 0) the one-launch decode step's first-digit
    histograms (include/qsa_indexer_testing.h), to exercise its count check."""
    _check(load().qsa_testing_decode_step_histograms(int(add), _stream(stream)))


def qsa_testing_stream_yardstick(dst, src, units, rows, rowPitch, unitPitch, offset, nbytes, stream=None):
    """A plain streaming kernel with a K1 kernel's byte pattern (include/qsa_indexer_testing.h)."""
    _check(load().qsa_testing_stream_yardstick(_addr(dst), _addr(src), int(units), int(rows), int(rowPitch),
                                            int(unitPitch), int(offset), int(nbytes), _stream(stream)))


def qsa_testing_gather_yardstick(dst, src, units, unitPitch, offset, nbytes, stream=None):
    """A plain gathering kernel with the paged decode scoring's byte pattern
    (include/qsa_indexer_testing.h)."""
    _check(load().qsa_testing_gather_yardstick(_addr(dst), _addr(src), int(units), int(unitPitch), int(offset),
                                            int(nbytes), _stream(stream)))


def qsa_testing_index_scores_cuda_core(logits, qNormed, kbar, contextLengths, batchSize, seqLen,
                                       numBlocks, rowStart, numRows, stream=None, dtype=None):
    """K2 on CUDA cores (include/qsa_indexer_testing.h): a test-only cross-check."""
    _check(load().qsa_testing_index_scores_cuda_core(
        _dtype(dtype, qNormed, kbar), _addr(logits), _addr(qNormed), _addr(kbar),
        _addr(contextLengths), int(batchSize), int(seqLen), int(numBlocks), int(rowStart),
        int(numRows), _stream(stream)))


def qsa_device_fault_flags(clear: bool = True, stream=None) -> int:
    """Synchronise ``stream`` and return (and optionally clear) the device fault bits."""
    flags = ctypes.c_uint32(0)
    _check(load().qsa_device_fault_flags(ctypes.byref(flags), 1 if clear else 0, _stream(stream)))
    return int(flags.value)
