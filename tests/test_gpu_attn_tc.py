"""GPU parity of the tensor-core attention kernels (bf16, head dim 128)
against the CPU oracle: CSA sparse attention over rows gathered with TMA
tile::gather4 (ragged batches, padding slots anywhere, k not a multiple of the
64-key tile, H below 128) and its device-side error flags.  Bar: max-abs 2e-2
on O and on lse."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module")
def lc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import long_context_compressed_13_b300 as m
    from long_context_compressed_13_b300 import _build
    _build.build()
    m.load_library()
    return m


def f64(x):
    return x.detach().to("cpu").double().numpy()


def bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(x).to(torch.bfloat16)


def _case(H, m, k, W, T, seed, q_from=0):
    L = wl.csa_layer(T=T, H=H, d=128, HI=4, dI=32, m=m, k=k, W=W, dtype="bf16", seed=seed,
                     q_from=q_from)
    Kc = bf16(oracle.compress(L["K"], L["G"], m))
    Vc = bf16(oracle.compress(L["V"], L["G"], m))
    return L, Kc, Vc


def _compare(O, lse, rO, rl):
    np.testing.assert_allclose(f64(O), rO, rtol=0, atol=TOL)
    g = f64(lse)
    assert np.array_equal(np.isneginf(g), np.isneginf(rl))
    fin = np.isfinite(rl)
    np.testing.assert_allclose(g[fin], rl[fin], rtol=0, atol=TOL)


@pytest.mark.parametrize("H,m,k,W,T,q_from", [
    (128, 4, 1024, 128, 6000, 5700),   # the 1M setting's head count, k and window
    (128, 4, 100, 128, 1500, 0),       # k not a multiple of 64, early rows padded
    (64, 4, 512, 128, 3000, 2500),     # H below 128: rows 64..127 of the tile idle
    (32, 8, 70, 0, 900, 300),          # no window
])
def test_sparse_tc(lc, H, m, k, W, T, q_from):
    L, Kc, Vc = _case(H, m, k, W, T, seed=81, q_from=q_from)
    tpos = np.array(L["batch"].positions())
    rng = np.random.default_rng(5)
    sel = oracle.topk(rng.standard_normal((len(tpos), T // m)), (tpos + 1) // m, k)
    b = lc.DeviceBatch.from_workload(L["batch"])
    O, lse = lc.sparse_mqa_attn(L["Q"].cuda(), Kc.cuda(), Vc.cuda(), torch.from_numpy(sel).cuda(),
                                L["K"].cuda(), L["V"].cuda(), b, m, W, L["scale"])
    torch.cuda.synchronize()
    rO, rl = oracle.sparse_attn(L["Q"], Kc, Vc, sel, L["K"], L["V"], 0, tpos, W, L["scale"])
    _compare(O, lse, rO, rl)


def test_sparse_tc_padding_anywhere_and_repeats(lc):
    # user-supplied selections: -1 slots in the middle, repeated entries
    # (each occurrence counts), unsorted order
    H, m, k, W, T = 128, 4, 96, 32, 800
    L, Kc, Vc = _case(H, m, k, W, T, seed=82)
    tpos = np.array(L["batch"].positions())
    rng = np.random.default_rng(6)
    sel = np.full((T, k), -1, dtype=np.int32)
    for r in range(T):
        nv = (r + 1) // m
        if nv:
            sel[r] = rng.integers(0, nv, k)
        sel[r, rng.random(k) < 0.3] = -1
    b = lc.DeviceBatch.from_workload(L["batch"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    O, lse = lc.sparse_mqa_attn(L["Q"].cuda(), Kc.cuda(), Vc.cuda(), torch.from_numpy(sel).cuda(),
                                L["K"].cuda(), L["V"].cuda(), b, m, W, L["scale"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rO, rl = oracle.sparse_attn(L["Q"], Kc, Vc, sel, L["K"], L["V"], 0, tpos, W, L["scale"])
    _compare(O, lse, rO, rl)


def test_sparse_tc_ragged_decode(lc):
    D = wl.csa_decode(B=7, ctx_lo=300, ctx_hi=5000, H=128, d=128, HI=8, dI=64, m=4, k=256,
                      W=128, dtype="bf16", seed=83)
    bt = D["batch"]
    b = lc.DeviceBatch.from_workload(bt)
    rng = np.random.default_rng(7)
    sels = []
    for s in range(bt.B):
        nv = bt.cu_c[s + 1] - bt.cu_c[s]
        sels.append(oracle.topk(rng.standard_normal((1, nv)), [nv], 256)[0])
    sel = np.stack(sels).astype(np.int32)
    O, lse = lc.sparse_mqa_attn(D["Q"].cuda(), D["Kc"].cuda(), D["Vc"].cuda(),
                                torch.from_numpy(sel).cuda(), D["Kraw"].cuda(), D["Vraw"].cuda(),
                                b, 4, 128, D["scale"])
    torch.cuda.synchronize()
    for s in range(bt.B):
        c0, c1, r0, r1 = bt.cu_c[s], bt.cu_c[s + 1], bt.cu_raw[s], bt.cu_raw[s + 1]
        rO, rl = oracle.sparse_attn(D["Q"][s:s + 1], D["Kc"][c0:c1], D["Vc"][c0:c1], sel[s:s + 1],
                                    D["Kraw"][r0:r1], D["Vraw"][r0:r1], bt.raw_pos0[s],
                                    [bt.q_pos0[s]], 128, D["scale"])
        _compare(O[s:s + 1], lse[s:s + 1], rO, rl)


def test_sparse_tc_flags_bad_indices(lc):
    H, m, k, W, T = 128, 4, 64, 16, 256
    L, Kc, Vc = _case(H, m, k, W, T, seed=84)
    sel = torch.full((T, k), -1, dtype=torch.int32)
    sel[100, 3] = 10 ** 6     # beyond the stored entries
    sel[40, 0] = 30           # stored, not visible from t=40 (n_vis = 10)
    sel[200, 0] = 7           # fine
    b = lc.DeviceBatch.from_workload(L["batch"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    O, _ = lc.sparse_mqa_attn(L["Q"].cuda(), Kc.cuda(), Vc.cuda(), sel.cuda(), L["K"].cuda(),
                              L["V"].cuda(), b, m, W, L["scale"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lc.LC_DEVERR_INDEX
    assert torch.isfinite(O.float()).all()
    # the flagged slots are skipped: rows 40 and 100 see only their window
    tpos = np.arange(T)
    clean = sel.numpy().copy()
    clean[100, 3] = -1
    clean[40, 0] = -1
    rO, _ = oracle.sparse_attn(L["Q"], Kc, Vc, clean, L["K"], L["V"], 0, tpos, W, L["scale"])
    np.testing.assert_allclose(f64(O), rO, rtol=0, atol=TOL)
