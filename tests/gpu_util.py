"""Device-side helpers for the GPU parity tests: uploads, red-zoned outputs, calls."""
from __future__ import annotations

import numpy as np
import torch

import sparse_attention_indexer_qsa_gb300 as qsa

RED = 256            # guard bytes on each side of every output (keeps 16-byte alignment)
RED_BYTE = 0xA5


def dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)          # T bit patterns travel as int16
    t = torch.from_numpy(a)
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def t_dtype(dtype: str):
    return {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]


class Guarded:
    """An output buffer with RED poisoned bytes before and after it."""

    def __init__(self, nbytes: int, fill: int | None = None, init: np.ndarray | None = None):
        self.nbytes = nbytes
        self.buf = torch.full((nbytes + 2 * RED,), RED_BYTE, dtype=torch.uint8, device="cuda")
        if init is not None:
            raw = np.ascontiguousarray(init).view(np.uint8).reshape(-1)
            assert raw.size == nbytes
            self.buf[RED:RED + nbytes].copy_(torch.from_numpy(raw))
        elif fill is not None:
            self.buf[RED:RED + nbytes].fill_(fill)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr() + RED

    def check_red(self):
        b = self.buf.cpu().numpy()
        assert np.all(b[:RED] == RED_BYTE), "write before the start of an output"
        assert np.all(b[RED + self.nbytes:] == RED_BYTE), "write past the end of an output"

    def numpy(self, dtype, shape) -> np.ndarray:
        torch.cuda.synchronize()
        self.check_red()
        return self.buf[RED:RED + self.nbytes].cpu().numpy().view(dtype).reshape(shape)


class DevWorkload:
    """A workloads.Workload uploaded to the device."""

    def __init__(self, wl):
        self.wl = wl
        self.dtype = wl.dtype
        self.index_qk = dev(wl.index_qk)
        self.cos_sin = dev(wl.cos_sin)
        self.ctx = dev(wl.context_lengths)
        self.w_q = dev(wl.w_q)
        self.w_k = dev(wl.w_k)


def q_prep(d: DevWorkload, index_qk=None, B=None, S=None) -> np.ndarray:
    wl = d.wl
    B = B or wl.B
    S = S or wl.S
    out = Guarded(B * S * 512 * 2)
    qsa.qsa_index_q_prep(out.ptr, index_qk if index_qk is not None else d.index_qk, d.cos_sin, d.ctx,
                         d.w_q, wl.eps, B, S, dtype=d.dtype)
    return out.numpy(np.uint16, (B, S, 4, 128))


def k_compress(d: DevWorkload, num_blocks, block_begin, block_end, past_len, index_qk=None,
               seq_len=None, kbar_init=None, sentinel=0x1234) -> np.ndarray:
    wl = d.wl
    S = seq_len or wl.S
    if kbar_init is None:
        kbar_init = np.full((wl.B, num_blocks, 128), sentinel, np.uint16)
    out = Guarded(wl.B * num_blocks * 128 * 2, init=kbar_init)
    qsa.qsa_index_k_compress(out.ptr, index_qk if index_qk is not None else d.index_qk, d.cos_sin,
                             d.ctx, d.w_k, wl.eps, wl.B, S, num_blocks, block_begin, block_end,
                             past_len, dtype=d.dtype)
    return out.numpy(np.uint16, (wl.B, num_blocks, 128))


def scores(dtype: str, q_dev, kbar_dev, ctx_dev, B, S, NB, row_start, num_rows,
           cuda_core=False) -> np.ndarray:
    out = Guarded(num_rows * NB * 4, fill=0x7F)
    fn = qsa.qsa_testing_index_scores_cuda_core if cuda_core else qsa.qsa_index_scores
    fn(out.ptr, q_dev, kbar_dev, ctx_dev, B, S, NB, row_start, num_rows, dtype=dtype)
    return out.numpy(np.float32, (num_rows, NB))


def assert_no_device_faults():
    assert qsa.qsa_device_fault_flags(clear=True) == 0
