"""The index + top-k entry point that allocates nothing.

Some callers cannot allocate device memory: a host program whose device
memory belongs to another runtime's pool, or a latency-critical loop where
cudaMalloc/cudaFree could synchronise the device.  For them the library keeps
the score matrix of the fused index + top-k in a fixed array of its own.  This
test calls that entry point through the C ABI twice in a row and checks that
its selection equals, bit for bit, the one of lightning_index with a caller
workspace (the top-k tolerance of every other test).  The file name makes
pytest collect it last.
"""
import ctypes

import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


def _noalloc_fn(lib):
    fn = lib.lightning_index_topk_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    import long_context_compressed_13_b300 as lc
    fn.argtypes = [vp, vp, vp, ctypes.POINTER(lc._LcBatch), i32, i32, i32, i32, i32, vp, vp, vp]
    fn.restype = i32
    return fn


def test_no_alloc_index_topk_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import long_context_compressed_13_b300 as lc
    from long_context_compressed_13_b300 import _build
    _build.build()
    lib = lc.load_library()
    fn = _noalloc_fn(lib)
    stream = torch.cuda.current_stream().cuda_stream

    cases = [
        # decode-shaped ragged batch (streaming launch shape), then a
        # prefill-shaped one with a narrower score matrix: the second call
        # reuses the array the first one filled
        wl.csa_decode(B=6, ctx_lo=4000, ctx_hi=40000, H=8, d=64, HI=8, dI=64, m=4, k=256, W=16,
                      dtype="bf16", seed=61),
        wl.csa_layer(T=1536, H=8, d=64, HI=4, dI=32, m=4, k=32, W=16, dtype="f32", seed=62),
    ]
    for L in cases:
        k = L["k"]
        b = lc.DeviceBatch.from_workload(L["batch"])
        qI, w, kI = L["qI"].cuda(), L["w"].cuda(), L["kI"].cuda()
        _, ref = lc.lightning_index(qI, w, kI, b, L["m"], scores=False, k=k, topk=True)
        out = torch.full((b.total_q, k), -7, dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        cb = b.c_struct()
        HI, dI = qI.shape[1], qI.shape[2]
        dt = lc.LC_F32 if qI.dtype == torch.float32 else lc.LC_BF16
        st = fn(qI.data_ptr(), w.data_ptr(), kI.data_ptr(), ctypes.byref(cb), HI, dI, L["m"], dt,
                k, out.data_ptr(), err.data_ptr(), stream)
        assert st == lc.LC_OK, lib.lc_status_string(st)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(out, ref)

    # a score matrix larger than the fixed array is refused, with no launch
    big = lc.DeviceBatch.from_host([0, 1024], [10 ** 7], [0, 1 << 20], [0, 0], [0])
    before = lib.lc_launch_count()
    out = torch.empty((1024, 8), dtype=torch.int32, device="cuda")
    st = fn(qI.data_ptr(), w.data_ptr(), kI.data_ptr(), ctypes.byref(big.c_struct()), HI, dI, 4,
            dt, 8, out.data_ptr(), None, stream)
    assert st == lc.LC_ERR_WORKSPACE
    assert lib.lc_launch_count() == before
