"""CPU checks of the C ABI: the library builds for sm_103a, loads without a
GPU, exports every function the public header declares, and rejects bad host
arguments before touching the device."""
import ctypes
import os
import re

import pytest

import long_context_compressed_13_b300 as lc
from long_context_compressed_13_b300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return lc.load_library()


def _declared_functions():
    names = []
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:lc_status|size_t|const char\s*\*|int32_t|uint64_t|void)\s*"
                             r"\*?\s*([A-Za-z_]\w*)\s*\(", text, flags=re.M):
            names.append(m.group(1))
    return names


def test_header_declares_the_method_calls():
    names = _declared_functions()
    for fn in ("csa_compress", "hca_compress", "lightning_index", "topk_select",
               "sparse_mqa_attn", "hca_dense_attn"):
        assert fn in names
    assert set(lc.ENTRY_POINTS) <= set(names)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {lc.LIB_PATH}").read()
    for name in _declared_functions():
        assert re.search(rf"\bT {name}$", out, flags=re.M), name


def test_library_has_no_libcuda_or_torch_dependency(lib):
    needed = os.popen(f"readelf -d {lc.LIB_PATH}").read()
    assert "libcuda.so" not in needed
    assert "torch" not in needed and "c10" not in needed


def test_host_only_helpers(lib):
    assert lib.lc_version().startswith(b"lcattn")
    assert lib.lc_status_string(0) == b"ok"
    assert b"argument" in lib.lc_status_string(1)
    assert isinstance(lib.lc_launch_count(), int)


def _batch(total_q=4, max_q=4, max_c=8, B=1, null=False):
    p = 0 if null else 0x1000
    return lc._LcBatch(B, p, p, p, p, p, total_q, max_q, max_c, max_c * B, 0)


def test_invalid_arguments_are_rejected_on_the_host(lib):
    launches_before = lib.lc_launch_count()
    P = ctypes.c_void_p(0x1000)
    N = None
    b = _batch()
    # compressors: null pointers, bad sizes, unsupported d
    assert lib.csa_compress(N, P, P, P, 16, 64, 4, lc.LC_F32, P, P, -1, N) == lc.LC_ERR_INVALID_ARG
    assert lib.csa_compress(P, P, N, P, 16, 64, 4, lc.LC_F32, P, P, -1, N) == lc.LC_ERR_INVALID_ARG
    assert lib.csa_compress(P, P, P, P, 16, 64, 4, lc.LC_F32, N, P, -1, N) == lc.LC_ERR_INVALID_ARG
    assert lib.csa_compress(P, P, P, P, -1, 64, 4, lc.LC_F32, P, P, -1, N) == lc.LC_ERR_INVALID_ARG
    assert lib.hca_compress(P, P, P, P, 16, 64, 0, lc.LC_F32, P, P, -1, N) == lc.LC_ERR_INVALID_ARG
    assert lib.csa_compress(P, P, P, P, 16, 96, 4, lc.LC_F32, P, P, -1, N) == lc.LC_ERR_UNSUPPORTED
    assert lib.csa_compress(P, P, P, P, 16, 64, 4, 7, P, P, -1, N) == lc.LC_ERR_INVALID_ARG
    # indexer: no output requested, missing batch arrays, bad head shape,
    # ld smaller than the widest sequence, missing workspace
    assert lib.lightning_index(P, P, P, ctypes.byref(b), 8, 64, 4, lc.LC_BF16, N, 0, 0, N, N, 0,
                               N, N) == lc.LC_ERR_INVALID_ARG
    nb = _batch(null=True)
    assert lib.lightning_index(P, P, P, ctypes.byref(nb), 8, 64, 4, lc.LC_BF16, P, 8, 0, N, N, 0,
                               N, N) == lc.LC_ERR_INVALID_ARG
    assert lib.lightning_index(P, P, P, ctypes.byref(b), 3, 64, 4, lc.LC_BF16, P, 8, 0, N, N, 0,
                               N, N) == lc.LC_ERR_UNSUPPORTED
    assert lib.lightning_index(P, P, P, ctypes.byref(b), 8, 48, 4, lc.LC_BF16, P, 8, 0, N, N, 0,
                               N, N) == lc.LC_ERR_UNSUPPORTED
    assert lib.lightning_index(P, P, P, ctypes.byref(b), 8, 64, 4, lc.LC_BF16, P, 7, 0, N, N, 0,
                               N, N) == lc.LC_ERR_INVALID_ARG
    assert lib.lightning_index(P, P, P, ctypes.byref(b), 8, 64, 4, lc.LC_BF16, N, 0, 16, P, N, 0,
                               N, N) == lc.LC_ERR_WORKSPACE
    # top-k: k out of range, ld too small
    assert lib.topk_select(P, 8, ctypes.byref(b), 4, 0, P, N, 0, N, N) == lc.LC_ERR_INVALID_ARG
    assert lib.topk_select(P, 8, ctypes.byref(b), 4, 5000, P, N, 0, N, N) == lc.LC_ERR_UNSUPPORTED
    assert lib.topk_select(P, 4, ctypes.byref(b), 4, 8, P, N, 0, N, N) == lc.LC_ERR_INVALID_ARG
    # attention: unsupported heads/dims, negative window, missing raw cache
    args = dict(scale=ctypes.c_float(0.125))
    assert lib.sparse_mqa_attn(P, P, P, P, 8, P, P, ctypes.byref(b), 12, 128, 4, 128,
                               args["scale"], N, 0, lc.LC_BF16, P, N, N, 0, N, N) == lc.LC_ERR_UNSUPPORTED
    assert lib.sparse_mqa_attn(P, P, P, P, 8, P, P, ctypes.byref(b), 64, 80, 4, 128,
                               args["scale"], N, 0, lc.LC_BF16, P, N, N, 0, N, N) == lc.LC_ERR_UNSUPPORTED
    assert lib.sparse_mqa_attn(P, P, P, P, 8, P, P, ctypes.byref(b), 64, 128, 4, -1,
                               args["scale"], N, 0, lc.LC_BF16, P, N, N, 0, N, N) == lc.LC_ERR_INVALID_ARG
    assert lib.sparse_mqa_attn(P, P, P, P, 8, N, N, ctypes.byref(b), 64, 128, 4, 16,
                               args["scale"], N, 0, lc.LC_BF16, P, N, N, 0, N, N) == lc.LC_ERR_INVALID_ARG
    assert lib.hca_dense_attn(P, P, P, P, P, ctypes.byref(b), 64, 128, 128, 128,
                              ctypes.c_float(0.0), N, 0, lc.LC_BF16, P, N, N, 0,
                              N, N) == lc.LC_ERR_INVALID_ARG
    assert lib.hca_dense_attn(N, P, P, P, P, ctypes.byref(b), 64, 128, 128, 128,
                              args["scale"], N, 0, lc.LC_BF16, P, N, N, 0, N, N) == lc.LC_ERR_INVALID_ARG
    # RoPE arguments: a negative position other than -1, a rope flag other than 0/1
    assert lib.csa_compress(P, P, P, P, 16, 64, 4, lc.LC_F32, P, P, -2, N) == lc.LC_ERR_INVALID_ARG
    assert lib.rope_rotate(P, 4, 1, 128, -1, 0, lc.LC_BF16, N) == lc.LC_ERR_INVALID_ARG
    assert lib.rope_rotate(P, 4, 1, 96, 0, 0, lc.LC_BF16, N) == lc.LC_ERR_UNSUPPORTED
    assert lib.hca_dense_attn(P, P, P, P, P, ctypes.byref(b), 64, 128, 128, 128,
                              args["scale"], N, 2, lc.LC_BF16, P, N, N, 0, N,
                              N) == lc.LC_ERR_INVALID_ARG
    assert lib.token_gated_compress(P, P, 16, 48, 4, lc.LC_F32, P, -1, N) == lc.LC_ERR_UNSUPPORTED
    # decode state: ring shorter than a block, missing indexer buffers
    Lbad = lc._LcDecodeLayer(2, 2, 128, 4, 0, 0, 16, *([0x1000] * 10))
    assert lib.decode_append(ctypes.byref(Lbad), P, P, N, P, P, N, lc.LC_BF16, N,
                             N) == lc.LC_ERR_INVALID_ARG
    Lidx = lc._LcDecodeLayer(2, 8, 128, 4, 8, 64, 16, 0x1000, 0x1000, 0x1000, 0, 0x1000, 0x1000,
                             0, 0x1000, 0x1000, 0x1000)
    assert lib.decode_append(ctypes.byref(Lidx), P, P, P, P, P, P, lc.LC_BF16, N,
                             N) == lc.LC_ERR_INVALID_ARG
    # MX quantizer and indexer: size not a multiple of 32, unknown format,
    # misaligned codes, unsupported head shape
    assert lib.mx_quantize(P, 48, lc.LC_MXFP8, lc.LC_BF16, P, P, N) == lc.LC_ERR_INVALID_ARG
    assert lib.mx_quantize(P, 64, 6, lc.LC_BF16, P, P, N) == lc.LC_ERR_INVALID_ARG
    assert lib.mx_quantize(P, 64, lc.LC_MXFP4, lc.LC_BF16, N, P, N) == lc.LC_ERR_INVALID_ARG
    A = ctypes.c_void_p(0x1008)
    assert lib.lightning_index_mx(6, P, P, P, P, P, ctypes.byref(b), 8, 64, 4, P, 8, 0, N, N, 0,
                                  N, N) == lc.LC_ERR_INVALID_ARG
    assert lib.lightning_index_mx(lc.LC_MXFP4, P, P, P, A, P, ctypes.byref(b), 8, 64, 4, P, 8, 0,
                                  N, N, 0, N, N) == lc.LC_ERR_INVALID_ARG
    assert lib.lightning_index_mx(lc.LC_MXFP8, P, P, P, P, P, ctypes.byref(b), 8, 32, 4, P, 8, 0,
                                  N, N, 0, N, N) == lc.LC_ERR_UNSUPPORTED
    assert lib.lightning_index_mx(lc.LC_MXFP8, P, P, P, P, P, ctypes.byref(b), 8, 64, 4, N, 0, 16,
                                  P, N, 0, N, N) == lc.LC_ERR_WORKSPACE
    # nothing above reached a kernel
    assert lib.lc_launch_count() == launches_before


def test_workspace_size_covers_materialised_scores(lib):
    b = _batch(total_q=64, max_q=1, max_c=65536, B=64)
    n = lib.lc_workspace_size(lc.LC_OP_LIGHTNING_INDEX, ctypes.byref(b), 0, 0, 8, 64, 1024)
    assert n >= 64 * 65536 * 4 and n % 256 == 0
    assert lib.lc_workspace_size(lc.LC_OP_TOPK_SELECT, ctypes.byref(b), 0, 0, 0, 0, 16) == 0


def test_workspace_is_bounded_without_the_score_matrix(lib):
    # the 1M-context chunk (4096 rows x 262144 entries: a 4 GiB score matrix)
    # fits in 512 MiB, for the fused tensor-core plan and for any other path
    b = _batch(total_q=4096, max_q=4096, max_c=262144)
    for HI, dI in ((8, 64), (2, 64), (4, 32)):
        n = lib.lc_workspace_size(lc.LC_OP_LIGHTNING_INDEX, ctypes.byref(b), 0, 0, HI, dI, 1024)
        assert 0 < n <= 512 << 20, (HI, dI, n)
    # a score matrix that fits in the chunk bound is kept whole
    small = _batch(total_q=300, max_q=300, max_c=1000)
    n = lib.lc_workspace_size(lc.LC_OP_LIGHTNING_INDEX, ctypes.byref(small), 0, 0, 2, 64, 32)
    assert n >= 300 * 1000 * 4


def test_binding_fails_loudly_without_a_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    K = torch.zeros(8, 64)
    with pytest.raises(ValueError, match="CUDA tensor"):
        lc.csa_compress(K, K, torch.zeros(4, 64), m=4)
