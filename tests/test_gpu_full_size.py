"""Parity at the full benchmarked sizes, in the launch configuration the
benchmark times, on sampled outputs the oracle computes one by one.

- layer_pair_1m: 1,048,576-token context, last 4096 positions queried; CSA
  (m=4, indexer 8x64 over 262,144 entries, top-k 1024, window 128) and HCA
  (m'=128, window 128), 128 heads x 128.  The step is the benchmark's own.
  266 sampled query rows are checked against the oracle: the fused top-k
  (equal, or different only inside the near-tie band of selection_check),
  CSA attention (rows whose
  selection equals the oracle's) and HCA attention, both within the bf16
  tolerance; sampled compressed entries of the chunk within one bf16 ulp.
- csa_decode: 64 sequences with contexts ~U[65536, 262144]; every sequence
  is checked the same way.
- csa_prefill (T=32768, 64 heads, k=512) and hca_prefill (T=131072, 64
  heads, m'=128): the benchmark's steps, 256+ sampled rows each, checked
  the same way.

The oracle builds its own compressed caches from the raw inputs (rounded to
bf16, the stored type) and never reads a value the CUDA path produced.
"""
import numpy as np
import pytest
import torch

import oracle
from selection_check import check_selection

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module")
def lc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import long_context_compressed_13_b300 as m
    m.load_library()
    return m


def _bf16_round(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def _check_rows(gsel, I, nvis, k):
    """Selections equal the oracle's, or differ only inside the near-tie
    band (selection_check).  Returns (oracle selection, identical-row mask)."""
    return check_selection(gsel, I, nvis, k)


def test_layer_pair_1m_sampled(lc):
    import bench
    wk = bench.LayerPair(lc, "cuda")
    wk.step()
    torch.cuda.synchronize()
    assert int(wk.err.item()) == 0
    P = wk.P
    c, h = P["csa"], P["hca"]
    Pc = {"csa": {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in c.items()},
          "hca": {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in h.items()}}
    st, raw, kI64 = bench._oracle_state(Pc, wk.q0, wk.ctx, wk.m_c, wk.m_h, wk.W)
    Kc, Vc = _bf16_round(st["Kc"]), _bf16_round(st["Vc"])
    Kh, Vh = _bf16_round(st["Kh"]), _bf16_round(st["Vh"])

    # compressed entries written by the timed step (the chunk's entries)
    rng = np.random.default_rng(11)
    for name, gpu, ref, m in (("csa K", wk.Kc, Kc, wk.m_c), ("csa V", wk.Vc, Vc, wk.m_c),
                              ("hca K", wk.Kh, Kh, wk.m_h), ("hca V", wk.Vh, Vh, wk.m_h)):
        lo = wk.q0 // m
        ents = np.unique(np.concatenate([[lo, ref.shape[0] - 1],
                                         rng.integers(lo, ref.shape[0], 30)]))
        got = gpu[torch.from_numpy(ents).cuda()].double().cpu().numpy()
        ulp = np.abs(ref[ents]) * 2.0 ** -7 + 1e-30
        assert np.all(np.abs(got - ref[ents]) <= ulp), name

    # 256+ query rows over the chunk: its first and last rows, the edges of
    # the 128-row tiles of the indexer and the HCA CTAs, and seeded rows
    fixed = [0, 1, 127, 128, 255, 256, 2047, 2048, 4094, 4095]
    rest = np.setdiff1d(np.arange(wk.chunk), fixed)
    rows = np.unique(np.concatenate([fixed, rng.choice(rest, 256, replace=False)]))
    t = (wk.q0 + rows).astype(np.int64)
    I = oracle.index(c["qI"][rows].cpu(), c["w"][rows].cpu(), kI64, t, wk.m_c)
    gsel = wk.sel[torch.from_numpy(rows).cuda()].cpu().numpy()
    rsel, same = _check_rows(gsel, I, (t + 1) // wk.m_c, wk.k)
    del I
    assert same.mean() >= 0.95

    rO, rl = oracle.sparse_attn(c["Q"][rows].cpu(), Kc, Vc, rsel, raw["csa_K"], raw["csa_V"],
                                raw["pos0"], t, wk.W, c["scale"])
    gO = wk.O_csa[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    np.testing.assert_allclose(gO[same], rO[same], rtol=0, atol=TOL)
    gl = wk.lse_csa[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    np.testing.assert_allclose(gl[same], rl[same], rtol=0, atol=TOL)

    rOh, rlh = oracle.hca_attn(h["Q"][rows].cpu(), Kh, Vh, wk.m_h, raw["hca_K"], raw["hca_V"],
                               raw["pos0"], t, wk.W, h["scale"])
    gOh = wk.O_hca[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    np.testing.assert_allclose(gOh, rOh, rtol=0, atol=TOL)
    glh = wk.lse_hca[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    np.testing.assert_allclose(glh, rlh, rtol=0, atol=TOL)


def test_csa_decode_sampled(lc):
    import bench
    wk = bench.Decode(lc, "cuda")
    wk.step()
    torch.cuda.synchronize()
    assert int(wk.err.item()) == 0
    D = wk.D
    bt = D["batch"]
    gsel_all = wk.sel.cpu().numpy()
    gO_all = wk.O.double().cpu().numpy()
    gl_all = wk.lse.double().cpu().numpy()
    # every sequence of the batch
    for s in range(D["B"]):
        c0, c1, r0, r1 = bt.cu_c[s], bt.cu_c[s + 1], bt.cu_raw[s], bt.cu_raw[s + 1]
        t = np.array([bt.q_pos0[s]], dtype=np.int64)
        I = oracle.index(D["qI"][s:s + 1].cpu(), D["w"][s:s + 1].cpu(), D["kI"][c0:c1].cpu(), t,
                         wk.m)
        rsel, same = _check_rows(gsel_all[s:s + 1], I, (t + 1) // wk.m, wk.k)
        if not same[0]:
            continue
        rO, rl = oracle.sparse_attn(D["Q"][s:s + 1].cpu(), D["Kc"][c0:c1].cpu(),
                                    D["Vc"][c0:c1].cpu(), rsel, D["Kraw"][r0:r1].cpu(),
                                    D["Vraw"][r0:r1].cpu(), bt.raw_pos0[s], t, wk.W, D["scale"])
        np.testing.assert_allclose(gO_all[s:s + 1], rO, rtol=0, atol=TOL)
        np.testing.assert_allclose(gl_all[s:s + 1], rl, rtol=0, atol=TOL)


def _sample_rows(T, n, rng, fixed):
    fixed = np.array(sorted(set(int(x) for x in fixed if 0 <= x < T)), dtype=np.int64)
    rest = np.setdiff1d(np.arange(T), fixed)
    return np.unique(np.concatenate([fixed, rng.choice(rest, n, replace=False)]))


def _check_entries(name, gpu, ref, rng):
    ents = np.unique(np.concatenate([[0, ref.shape[0] - 1], rng.integers(0, ref.shape[0], 64)]))
    got = gpu[torch.from_numpy(ents).cuda()].double().cpu().numpy()
    ulp = np.abs(ref[ents]) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(got - ref[ents]) <= ulp), name


def test_csa_prefill_32k_sampled(lc):
    """CSA prefill, T = 32,768, 64 heads x 128, indexer 8 x 64 over 8192
    entries, top-k 512, window 128: the benchmark's step, 256+ sampled rows."""
    import bench
    wk = bench.CsaPrefill(lc, "cuda")
    for _ in range(3):  # repeated steps reuse the workspace, as the benchmark does
        wk.step()
    torch.cuda.synchronize()
    assert int(wk.err.item()) == 0
    L = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in wk.L.items()}
    rng = np.random.default_rng(21)
    Kc = _bf16_round(oracle.compress(L["K"], L["G"], wk.m))
    Vc = _bf16_round(oracle.compress(L["V"], L["G"], wk.m))
    _check_entries("Kc", wk.Kc, Kc, rng)
    _check_entries("Vc", wk.Vc, Vc, rng)
    # the first rows (no entry visible), rows around the first entries and the
    # point where n_vis passes k, tile edges of the indexer, the last rows
    fixed = [0, 1, 2, 3, 4, 127, 128, 2047, 2048, 2051, 4095, 4096, 16383, 16384, 32766, 32767]
    rows = _sample_rows(wk.T, 256, rng, fixed)
    t = rows.astype(np.int64)
    I = oracle.index(L["qI"][rows], L["w"][rows], L["kI"], t, wk.m)
    gsel = wk.sel[torch.from_numpy(rows).cuda()].cpu().numpy()
    rsel, same = _check_rows(gsel, I, (t + 1) // wk.m, wk.k)
    assert same.mean() >= 0.95
    rO, rl = oracle.sparse_attn(L["Q"][rows], Kc, Vc, rsel, L["K"], L["V"], 0, t, wk.W,
                                L["scale"])
    gO = wk.O[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    gl = wk.lse[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    np.testing.assert_allclose(gO[same], rO[same], rtol=0, atol=TOL)
    np.testing.assert_allclose(gl[same], rl[same], rtol=0, atol=TOL)


def test_hca_prefill_128k_sampled(lc):
    """HCA prefill, T = 131,072, 64 heads x 128, m' = 128 (1024 entries),
    window 128: the benchmark's step, 256+ sampled rows."""
    import bench
    wk = bench.HcaPrefill(lc, "cuda")
    wk.step()
    torch.cuda.synchronize()
    assert int(wk.err.item()) == 0
    L = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in wk.L.items()}
    rng = np.random.default_rng(22)
    Kc = _bf16_round(oracle.compress(L["K"], L["G"], wk.m))
    Vc = _bf16_round(oracle.compress(L["V"], L["G"], wk.m))
    _check_entries("Kc", wk.Kc, Kc, rng)
    _check_entries("Vc", wk.Vc, Vc, rng)
    # rows before the first entry, around entry boundaries, CTA edges (4
    # tokens of 64 heads per CTA) and the last rows
    fixed = [0, 1, 3, 4, 126, 127, 128, 255, 256, 257, 16383, 16384, 65535, 65536,
             131068, 131071]
    rows = _sample_rows(wk.T, 256, rng, fixed)
    rO, rl = oracle.hca_attn(L["Q"][rows], Kc, Vc, wk.m, L["K"], L["V"], 0,
                             rows.astype(np.int64), wk.W, L["scale"])
    gO = wk.O[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    gl = wk.lse[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    np.testing.assert_allclose(gO, rO, rtol=0, atol=TOL)
    np.testing.assert_allclose(gl, rl, rtol=0, atol=TOL)
