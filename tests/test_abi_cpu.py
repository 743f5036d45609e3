"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
headers declare, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def qsa():
    from sparse_attention_indexer_qsa_gb300 import build as b
    b.build()
    import sparse_attention_indexer_qsa_gb300 as q
    return q


def declared_functions():
    names = set()
    for f in os.listdir(INCLUDE):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(INCLUDE, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?\w+\s*\*?\s*(qsa_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_headers_declare_the_entry_points():
    names = declared_functions()
    for n in ("qsa_index_q_prep", "qsa_index_k_compress", "qsa_index_scores", "qsa_last_error",
              "qsa_abi_version", "qsa_device_fault_flags"):
        assert n in names


def test_library_exports_every_declared_symbol(qsa):
    lib = qsa.load()
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", qsa.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    public = {s for s in exported if s.startswith("qsa_")}
    assert public == declared_functions(), public ^ declared_functions()
    assert qsa.qsa_abi_version() == 1


P = 0x1000  # a 16-byte aligned fake device address: never dereferenced on these paths


def test_null_dtype_shape_range_align_rejected(qsa):
    L = qsa.load()
    # null pointers
    assert L.qsa_index_q_prep(0, None, P, P, P, P, 1e-6, 1, 8, None) == -1
    assert L.qsa_index_k_compress(0, P, None, P, P, P, 1e-6, 1, 8, 2, 0, 2, 0, None) == -1
    assert L.qsa_index_scores(0, P, P, None, P, 1, 8, 2, 0, 8, None) == -1
    assert "null" in qsa.qsa_last_error()
    # dtype
    assert L.qsa_index_q_prep(7, P, P, P, P, P, 1e-6, 1, 8, None) == -4
    # shapes
    assert L.qsa_index_q_prep(0, P, P, P, P, P, 1e-6, 0, 8, None) == -2
    assert L.qsa_index_q_prep(0, P, P, P, P, P, 1e-6, 1, 0, None) == -2
    assert L.qsa_index_q_prep(0, P, P, P, P, P, 1e-6, 65536, 65536, None) == -2
    assert L.qsa_index_scores(0, P, P, P, P, 1, 9, 2, 0, 9, None) == -2       # NB < ceil(9/4)
    # ranges
    assert L.qsa_index_k_compress(0, P, P, P, P, P, 1e-6, 1, 8, 2, 1, 3, 0, None) == -3
    assert L.qsa_index_k_compress(0, P, P, P, P, P, 1e-6, 1, 8, 2, 2, 1, 0, None) == -3
    assert L.qsa_index_k_compress(0, P, P, P, P, P, 1e-6, 1, 8, 2, -1, 1, 0, None) == -3
    assert L.qsa_index_k_compress(0, P, P, P, P, P, 1e-6, 1, 8, 2, 0, 1, -4, None) == -3
    assert L.qsa_index_scores(0, P, P, P, P, 2, 8, 2, 10, 7, None) == -3
    assert L.qsa_index_scores(0, P, P, P, P, 2, 8, 2, -1, 1, None) == -3
    # alignment
    assert L.qsa_index_q_prep(0, P + 2, P, P, P, P, 1e-6, 1, 8, None) == -5
    assert L.qsa_index_k_compress(0, P, P, P + 8, P, P, 1e-6, 1, 8, 2, 0, 2, 0, None) == -5
    assert L.qsa_index_scores(0, P, P + 4, P, P, 1, 8, 2, 0, 8, None) == -5
    assert "aligned" in qsa.qsa_last_error()
    # the testing entry point validates the same way
    assert L.qsa_testing_index_scores_cuda_core(0, P, P, None, P, 1, 8, 2, 0, 8, None) == -1
    assert L.qsa_testing_bounded_wait_probe(0, None) == -3          # timeout out of range
    assert L.qsa_testing_bounded_wait_probe(10001, None) == -3


def test_empty_work_is_a_no_op(qsa):
    L = qsa.load()
    assert L.qsa_index_k_compress(0, P, P, P, P, P, 1e-6, 1, 8, 2, 1, 1, 0, None) == 0
    assert L.qsa_index_scores(0, P, P, P, P, 1, 8, 2, 8, 0, None) == 0
    assert qsa.qsa_last_error() == ""


def test_error_message_is_per_thread(qsa):
    import threading
    L = qsa.load()
    assert L.qsa_index_q_prep(0, None, P, P, P, P, 1e-6, 1, 8, None) == -1
    seen = []

    def other():
        seen.append(qsa.qsa_last_error())

    th = threading.Thread(target=other)
    th.start()
    th.join()
    assert seen == [""]
    assert "null" in qsa.qsa_last_error()


def test_binding_raises_with_status(qsa):
    with pytest.raises(qsa.QsaError) as e:
        qsa.qsa_index_k_compress(P, P, P, P, P, 1e-6, 1, 8, 2, 2, 1, 0, stream=0, dtype="bf16")
    assert e.value.status == -3
    assert "QSA_E_RANGE" in str(e.value)


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "sparse_attention_indexer_qsa_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".h", ".cuh")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "qsa_oracle" not in text, f


def test_binding_rejects_host_and_strided_tensors(qsa):
    """A host tensor's address is not a device address, and the kernels ignore strides:
    the binding refuses both before calling the library."""
    import torch
    host = torch.zeros((1, 8, 640), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        qsa.qsa_index_q_prep(host, host, host, host, host, 1e-6, 1, 8, stream=0)

    class StridedDeviceView:  # stands in for a non-contiguous CUDA tensor
        is_cuda = True

        def is_contiguous(self):
            return False

        def data_ptr(self):
            return P
    with pytest.raises(ValueError, match="contiguous"):
        qsa._addr(StridedDeviceView())
    assert qsa._addr(None) is None and qsa._addr(P) == P


def test_binding_dtype_must_match_the_tensors(qsa):
    """One T per call: bf16 and fp16 tensors are not mixed, and an explicit dtype agrees
    with them (checked before any address is taken)."""
    import torch
    bf = torch.zeros((1, 8, 640), dtype=torch.bfloat16)
    fp = torch.zeros((1, 8, 4, 128), dtype=torch.float16)
    bits = torch.zeros((128,), dtype=torch.int16)
    with pytest.raises(ValueError, match="mix"):
        qsa.qsa_index_q_prep(fp, bf, P, P, bits, 1e-6, 1, 8, stream=0)
    with pytest.raises(ValueError, match="does not match"):
        qsa.qsa_index_q_prep(P, bf, P, P, bits, 1e-6, 1, 8, stream=0, dtype="fp16")
    with pytest.raises(ValueError, match="inferable"):
        qsa.qsa_index_q_prep(P, P, P, P, bits, 1e-6, 1, 8, stream=0)
    assert qsa._dtype("fp16", bits, P) == qsa.QSA_F16      # bit-pattern tensors: dtype as given
    assert qsa._dtype(None, bits, bf) == qsa.QSA_BF16
