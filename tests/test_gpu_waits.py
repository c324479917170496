"""The bounded waits of the tensor-core kernels, made to run out without a
fault.

Every mbarrier wait in the tensor-core kernels gives up after a limit, marks
the CTA as aborted, raises LC_DEVERR_TIMEOUT, waits (again bounded) for its
own copies in flight and still frees its tensor memory.  The library's test
hook lc_debug_stall makes the MMA issuer of a chosen kernel first wait on a
barrier that nothing completes (before any MMA is issued), with a limit of
about a millisecond.  Each test checks that the call then reports the
timeout bit, and that the next normal call on the same context is correct:
had a CTA kept its tensor memory, the next kernel's allocation on that SM
would never succeed.  With LC_DEBUG_SYNC=1 (a fresh process) the timeout
comes back as the call's status, LC_ERR_TIMEOUT.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu
STALL_CLOCKS = 2_000_000  # about 1 ms at 2 GHz
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import long_context_compressed_13_b300 as m
    from long_context_compressed_13_b300 import _build
    _build.build()
    m.load_library()
    yield m
    m.debug_stall(0, 0)


def _bf16(x):
    return torch.from_numpy(x).to(torch.bfloat16)


def _hca_case():
    L = wl.hca_layer(T=600, H=64, d=128, m=8, W=32, dtype="bf16", seed=51)
    Kc, Vc = _bf16(oracle.compress(L["K"], L["G"], 8)), _bf16(oracle.compress(L["V"], L["G"], 8))
    return L, Kc, Vc


def _run_hca(lc, L, Kc, Vc, err):
    b = lc.DeviceBatch.from_workload(L["batch"])
    return lc.hca_dense_attn(L["Q"].cuda(), Kc.cuda(), Vc.cuda(), L["K"].cuda(), L["V"].cuda(), b,
                             8, 32, L["scale"], dev_err=err)


def test_hca_wait_runs_out_then_next_call_is_exact(lc):
    L, Kc, Vc = _hca_case()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lc.debug_stall(lc.LC_STALL_HCA_TC, STALL_CLOCKS)
    _run_hca(lc, L, Kc, Vc, err)
    torch.cuda.synchronize()
    assert lc.last_kernel() == "k_hca_tc"
    assert int(err.item()) & lc.LC_DEVERR_TIMEOUT
    lc.debug_stall(0, 0)
    err.zero_()
    O, _ = _run_hca(lc, L, Kc, Vc, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    tpos = np.arange(600)
    rO, _ = oracle.hca_attn(L["Q"], Kc, Vc, 8, L["K"], L["V"], 0, tpos, 32, L["scale"])
    np.testing.assert_allclose(O.double().cpu().numpy(), rO, rtol=0, atol=2e-2)


def test_sparse_wait_runs_out_then_next_call_is_exact(lc):
    T, m, k, W = 600, 4, 32, 32
    L = wl.csa_layer(T=T, H=64, d=128, HI=4, dI=32, m=m, k=k, W=W, dtype="bf16", seed=52)
    Kc, Vc = _bf16(oracle.compress(L["K"], L["G"], m)), _bf16(oracle.compress(L["V"], L["G"], m))
    tpos = np.arange(T)
    sel = oracle.topk(np.random.default_rng(1).standard_normal((T, T // m)), (tpos + 1) // m, k)
    b = lc.DeviceBatch.from_workload(L["batch"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (L["Q"].cuda(), Kc.cuda(), Vc.cuda(), torch.from_numpy(sel).cuda(), L["K"].cuda(),
            L["V"].cuda(), b, m, W, L["scale"])
    lc.debug_stall(lc.LC_STALL_SPARSE_TC, STALL_CLOCKS)
    lc.sparse_mqa_attn(*args, dev_err=err)
    torch.cuda.synchronize()
    assert lc.last_kernel() == "k_sparse_tc"
    assert int(err.item()) & lc.LC_DEVERR_TIMEOUT
    lc.debug_stall(0, 0)
    err.zero_()
    O, _ = lc.sparse_mqa_attn(*args, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rO, _ = oracle.sparse_attn(L["Q"], Kc, Vc, sel, L["K"], L["V"], 0, tpos, W, L["scale"])
    np.testing.assert_allclose(O.double().cpu().numpy(), rO, rtol=0, atol=2e-2)


def test_indexer_wait_runs_out_then_next_call_is_exact(lc):
    L = wl.csa_layer(T=2048, H=8, d=64, HI=8, dI=64, m=4, k=16, W=16, dtype="bf16", seed=53)
    b = lc.DeviceBatch.from_workload(L["batch"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qI, w, kI = L["qI"].cuda(), L["w"].cuda(), L["kI"].cuda()
    lc.debug_stall(lc.LC_STALL_INDEX_TC, STALL_CLOCKS)
    lc.lightning_index(qI, w, kI, b, 4, scores=True, dev_err=err)
    torch.cuda.synchronize()
    assert lc.last_kernel() == "k_index_tc<materialize>"
    assert int(err.item()) & lc.LC_DEVERR_TIMEOUT
    lc.debug_stall(0, 0)
    err.zero_()
    sc, _ = lc.lightning_index(qI, w, kI, b, 4, scores=True, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.index(L["qI"], L["w"], L["kI"], np.arange(2048), 4)
    got = sc.double().cpu().numpy()
    vis = np.isfinite(ref)
    assert np.array_equal(np.isneginf(got), ~vis)
    np.testing.assert_allclose(got[vis], ref[vis], rtol=1e-5, atol=1e-3)


_DEBUG_SYNC_SCRIPT = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import long_context_compressed_13_b300 as lc
import workloads as wl
L = wl.hca_layer(T=600, H=64, d=128, m=8, W=32, dtype="bf16", seed=51)
dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in L.items()}
b = lc.DeviceBatch.from_workload(L["batch"])
Kc, Vc = lc.hca_compress(dev["K"], dev["V"], dev["G"], m=8)
err = torch.zeros(1, dtype=torch.int32, device="cuda")
lc.debug_stall(lc.LC_STALL_HCA_TC, 2_000_000)
try:
    lc.hca_dense_attn(dev["Q"], Kc, Vc, dev["K"], dev["V"], b, 8, 32, L["scale"], dev_err=err)
    print("no error")
except lc.LCError as e:
    print("status", e.status)
lc.debug_stall(0, 0)
err.zero_()
lc.hca_dense_attn(dev["Q"], Kc, Vc, dev["K"], dev["V"], b, 8, 32, L["scale"], dev_err=err)
print("then ok", int(err.item()))
"""


def test_debug_sync_reports_the_timeout_status(lc):
    env = dict(os.environ, LC_DEBUG_SYNC="1")
    out = subprocess.run([sys.executable, "-c", _DEBUG_SYNC_SCRIPT, ROOT], env=env,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    assert f"status {lc.LC_ERR_TIMEOUT}" in out.stdout, out.stdout
    assert "then ok 0" in out.stdout, out.stdout
