"""GPU parity of every step against the CPU oracle, through the C ABI.

Inputs are drawn by ``workloads`` on the CPU and copied to the device, so both
sides read identical values.  Bars:
  - compressed entries: fp32 within 1e-5; bf16 a faithful rounding of the
    fp64 value (within one bf16 ulp);
  - indexer scores: within a derived fp32 accumulation bound; invisible
    entries exactly -inf;
  - top-k: bit-exact on identical score tensors;
  - attention: max-abs 1e-4 (fp32 inputs) and 2e-2 (bf16 inputs);
  - fused index + top-k: rows whose selection differs from the oracle's are
    allowed only where the oracle's gap between its k-th and (k+1)-th score
    is below 1e-5.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from selection_check import check_row, check_selection

pytestmark = pytest.mark.gpu

TOL_ATTN = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module")
def lc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import long_context_compressed_13_b300 as m
    from long_context_compressed_13_b300 import _build
    _build.build()
    m.load_library()
    return m


def dev(x):
    return x.to("cuda")


def f64(x):
    return x.detach().to("cpu").double().numpy()


def cast(x: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(x).to(wl.DTYPES[dtype])


def assert_faithful_bf16(got: torch.Tensor, exact: np.ndarray):
    g = f64(got)
    tol = np.abs(exact) * 2.0 ** -7 + 1e-30
    bad = np.abs(g - exact) > tol
    assert not bad.any(), f"{bad.sum()} entries off by more than one bf16 ulp"


# ------------------------------------------------------------- compressors

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("m,T,d", [(4, 2048, 64), (4, 1027, 128), (128, 4096 + 77, 128),
                                   (128, 100, 64), (4, 3, 64), (1, 65, 64)])
def test_compress(lc, dtype, m, T, d):
    g = wl._gen(11, "cpu")
    K, V = wl.normal(g, (T, d), dtype, "cpu"), wl.normal(g, (T, d), dtype, "cpu")
    GK, GV = wl.normal(g, (m, d), "f32", "cpu"), wl.normal(g, (m, d), "f32", "cpu")
    fn = lc.csa_compress if m < 128 else lc.hca_compress
    Kc, Vc = fn(dev(K), dev(V), dev(GK), dev(GV), m=m)
    torch.cuda.synchronize()
    assert Kc.shape == (T // m, d)
    for got, X, G in ((Kc, K, GK), (Vc, V, GV)):
        exact = oracle.compress(X, G, m)
        if dtype == "f32":
            np.testing.assert_allclose(f64(got), exact, rtol=0, atol=1e-5)
        else:
            assert_faithful_bf16(got, exact)


# ----------------------------------------------------------------- indexer

def _index_bound(qI, w, kI, tpos, m):
    """Rigorous bound on an fp32 evaluation of the score: gamma_n times the
    sum of |terms|, n = dI + HI + 2 rounding steps."""
    q, k, ww = f64(qI), f64(kI), f64(w)
    absdot = np.einsum("rhe,jhe->rjh", np.abs(q), np.abs(k))
    mag = np.einsum("rh,rjh->rj", np.abs(ww), absdot)
    n = q.shape[2] + q.shape[1] + 2
    u = 2.0 ** -24
    return mag * (n * u / (1 - n * u)) + 1e-30


@pytest.mark.parametrize("dtype,HI,dI,T,m", [("f32", 4, 32, 2048, 4), ("bf16", 8, 64, 1536, 4),
                                             ("bf16", 8, 64, 700, 8)])
def test_index_scores(lc, dtype, HI, dI, T, m):
    L = wl.csa_layer(T=T, H=8, d=64, HI=HI, dI=dI, m=m, k=16, W=16, dtype=dtype, seed=5)
    b = lc.DeviceBatch.from_workload(L["batch"])
    tpos = np.array(L["batch"].positions())
    sc, _ = lc.lightning_index(dev(L["qI"]), dev(L["w"]), dev(L["kI"]), b, m)
    torch.cuda.synchronize()
    ref = oracle.index(L["qI"], L["w"], L["kI"], tpos, m)
    got = sc.cpu().double().numpy()
    vis = np.isfinite(ref)
    assert np.array_equal(np.isneginf(got), ~vis)
    bound = _index_bound(L["qI"], L["w"], L["kI"], tpos, m)
    assert np.all(np.abs(got[vis] - ref[vis]) <= bound[vis])


def test_index_scan_ragged_decode(lc):
    # few rows per sequence: the streaming (decode) launch shape
    D = wl.csa_decode(B=5, ctx_lo=37, ctx_hi=3000, H=8, d=64, HI=8, dI=64, m=4, k=64, W=16,
                      dtype="bf16", seed=9)
    b = lc.DeviceBatch.from_workload(D["batch"])
    sc, sel = lc.lightning_index(dev(D["qI"]), dev(D["w"]), dev(D["kI"]), b, 4, k=64, topk=True)
    torch.cuda.synchronize()
    got, gsel = sc.cpu().double().numpy(), sel.cpu().numpy()
    bt = D["batch"]
    for s in range(bt.B):
        c0, c1 = bt.cu_c[s], bt.cu_c[s + 1]
        t = bt.q_pos0[s]
        ref = oracle.index(D["qI"][s:s + 1], D["w"][s:s + 1], D["kI"][c0:c1], [t], 4)
        nv = c1 - c0
        assert np.all(np.isneginf(got[s, nv:]))
        bound = _index_bound(D["qI"][s:s + 1], D["w"][s:s + 1], D["kI"][c0:c1], [t], 4)
        assert np.all(np.abs(got[s, :nv] - ref[0]) <= bound[0])
        osel = oracle.topk(ref, [nv], 64)[0]
        check_row(gsel[s], osel, ref[0], nv, 64, label=f"sequence {s}")


@pytest.mark.parametrize("HI", [4, 8])
def test_index_stream_long_rows(lc, HI):
    # decode rows long enough to be split across several CTAs of the
    # streaming indexer (1024+ entries each), both head counts it serves
    D = wl.csa_decode(B=3, ctx_lo=9000, ctx_hi=24000, H=8, d=64, HI=HI, dI=64, m=4, k=128, W=16,
                      dtype="bf16", seed=19)
    b = lc.DeviceBatch.from_workload(D["batch"])
    sc, sel = lc.lightning_index(dev(D["qI"]), dev(D["w"]), dev(D["kI"]), b, 4, k=128, topk=True)
    torch.cuda.synchronize()
    got, gsel = sc.cpu().double().numpy(), sel.cpu().numpy()
    bt = D["batch"]
    for s in range(bt.B):
        c0, c1 = bt.cu_c[s], bt.cu_c[s + 1]
        t = bt.q_pos0[s]
        nv = c1 - c0
        assert nv > 2048
        ref = oracle.index(D["qI"][s:s + 1], D["w"][s:s + 1], D["kI"][c0:c1], [t], 4)
        assert np.all(np.isneginf(got[s, nv:]))
        bound = _index_bound(D["qI"][s:s + 1], D["w"][s:s + 1], D["kI"][c0:c1], [t], 4)
        assert np.all(np.abs(got[s, :nv] - ref[0]) <= bound[0])
        osel = oracle.topk(ref, [nv], 128)[0]
        check_row(gsel[s], osel, ref[0], nv, 128, label=f"sequence {s}")


# ------------------------------------------------------------------- top-k

def _score_rows(kind, Nq, ld, seed):
    g = torch.Generator().manual_seed(seed)
    if kind == "normal":
        return torch.randn(Nq, ld, generator=g)
    if kind == "ties":
        return torch.randint(0, 4, (Nq, ld), generator=g).float()
    if kind == "zeros":  # ReLU-style exact zeros with mixed signs
        x = torch.randint(0, 3, (Nq, ld), generator=g).float() - 1.0
        x = torch.where(x < 0, torch.zeros_like(x), x)
        sign = torch.randint(0, 2, (Nq, ld), generator=g).bool()
        return torch.where((x == 0) & sign, -torch.zeros_like(x), x)
    if kind == "wide":  # magnitudes across many binades, both signs
        e = torch.randint(-60, 60, (Nq, ld), generator=g).float()
        s = torch.randint(0, 2, (Nq, ld), generator=g).float() * 2 - 1
        return s * torch.exp2(e) * (1 + torch.rand(Nq, ld, generator=g))
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["normal", "ties", "zeros", "wide"])
@pytest.mark.parametrize("k,m,ld,Nq,t0", [
    (1, 4, 300, 64, 900), (32, 4, 512, 200, 0), (512, 4, 8192, 48, 20000),
    (1024, 4, 3000, 40, 9000), (4096, 1, 6000, 8, 5990), (7, 128, 40, 30, 4000),
    # at most 296 rows of 4096+ entries: one 8-CTA cluster per row
    (1024, 4, 65536, 64, 200000),   # ~50000 visible entries, slices staged in shared memory
    (2048, 4, 9000, 100, 30000),    # slices of ~940 entries
    (4096, 4, 20000, 20, 70000),
    (64, 1, 140000, 16, 139990),    # slices of 17500 > 16384 entries: read from global memory
    (4090, 1, 4100, 24, 4080),      # rows of 4081..4100 entries, some with n_vis <= k
])
def test_topk_bit_exact(lc, kind, k, m, ld, Nq, t0):
    S = _score_rows(kind, Nq, ld, seed=k + ld)
    nvis = np.minimum((np.arange(t0, t0 + Nq) + 1) // m, ld)
    Tc = int(nvis.max())
    batch = wl.single(T_raw=0, q_pos0=t0, Nq=Nq, Tc=Tc)
    b = lc.DeviceBatch.from_workload(batch)
    got = lc.topk_select(dev(S), b, m, k).cpu().numpy()
    torch.cuda.synchronize()
    ref = oracle.topk(S.double().numpy(), nvis, k)
    assert np.array_equal(got, ref)


# --------------------------------------------------------------- attention

def _attn_case(dtype, H, d, m, k, W, T, seed, q_from=0):
    L = wl.csa_layer(T=T, H=H, d=d, HI=4, dI=32, m=m, k=k, W=W, dtype=dtype, seed=seed,
                     q_from=q_from)
    # compressed entries: the oracle's own compression, rounded to the dtype
    Kc = cast(oracle.compress(L["K"], L["G"], m), dtype)
    Vc = cast(oracle.compress(L["V"], L["G"], m), dtype)
    return L, Kc, Vc


@pytest.mark.parametrize("dtype,H,d,m,k,W,T", [
    ("f32", 8, 64, 4, 32, 64, 2048),
    ("bf16", 64, 128, 4, 64, 128, 1200),
    ("bf16", 16, 64, 4, 512, 0, 700),     # k > n_vis everywhere: -1 padding
    ("f32", 8, 128, 2, 5, 3, 300),
    ("bf16", 128, 128, 4, 16, 16, 160),
])
def test_sparse_attn(lc, dtype, H, d, m, k, W, T):
    L, Kc, Vc = _attn_case(dtype, H, d, m, k, W, T, seed=21)
    tpos = np.array(L["batch"].positions())
    rng = np.random.default_rng(3)
    sel = oracle.topk(rng.standard_normal((len(tpos), max(1, T // m))), (tpos + 1) // m, k)
    b = lc.DeviceBatch.from_workload(L["batch"])
    O, lse = lc.sparse_mqa_attn(dev(L["Q"]), dev(Kc), dev(Vc), dev(torch.from_numpy(sel)),
                                dev(L["K"]), dev(L["V"]), b, m, W, L["scale"])
    torch.cuda.synchronize()
    rO, rl = oracle.sparse_attn(L["Q"], Kc, Vc, sel, L["K"], L["V"], 0, tpos, W, L["scale"])
    tol = TOL_ATTN[dtype]
    np.testing.assert_allclose(f64(O), rO, rtol=0, atol=tol)
    g = f64(lse)
    assert np.array_equal(np.isneginf(g), np.isneginf(rl))
    fin = np.isfinite(rl)
    np.testing.assert_allclose(g[fin], rl[fin], rtol=0, atol=tol)


@pytest.mark.parametrize("dtype,H,d,m,W,T,q_from", [
    ("f32", 8, 64, 128, 128, 1000, 0),
    ("bf16", 64, 128, 128, 128, 2100, 0),
    ("bf16", 64, 128, 4, 0, 300, 0),
    ("f32", 16, 128, 1, 0, 90, 0),        # m'=1, W=0: plain causal attention
    ("bf16", 128, 128, 128, 128, 8192 + 300, 8192 - 200),
    ("bf16", 64, 128, 128, 128, 301, 0),   # last CTA holds 64 of 128 rows
    ("bf16", 32, 128, 16, 48, 700, 100),   # 4 tokens per tile, window crosses tiles
    ("bf16", 128, 128, 128, 0, 1000, 0),   # no window: rows t < 127 see nothing
])
def test_hca_attn(lc, dtype, H, d, m, W, T, q_from):
    L = wl.hca_layer(T=T, H=H, d=d, m=m, W=W, dtype=dtype, seed=31, q_from=q_from)
    Kc = cast(oracle.compress(L["K"], L["G"], m), dtype)
    Vc = cast(oracle.compress(L["V"], L["G"], m), dtype)
    tpos = np.array(L["batch"].positions())
    b = lc.DeviceBatch.from_workload(L["batch"])
    O, lse = lc.hca_dense_attn(dev(L["Q"]), dev(Kc), dev(Vc), dev(L["K"]), dev(L["V"]), b, m, W,
                               L["scale"])
    torch.cuda.synchronize()
    rO, rl = oracle.hca_attn(L["Q"], Kc, Vc, m, L["K"], L["V"], 0, tpos, W, L["scale"])
    tol = TOL_ATTN[dtype]
    np.testing.assert_allclose(f64(O), rO, rtol=0, atol=tol)
    fin = np.isfinite(rl)
    assert np.array_equal(np.isneginf(f64(lse)), ~fin)
    np.testing.assert_allclose(f64(lse)[fin], rl[fin], rtol=0, atol=tol)


@pytest.mark.parametrize("H", [64, 128])
def test_hca_attn_ragged(lc, H):
    # one ragged batch: row tiles of each sequence end part-way, a sequence
    # without query rows, one whose window starts before its first query, one
    # with a single compressed entry; every sequence against the oracle alone
    m, W, dtype = 128, 128, "bf16"
    seqs = [(2100, 0), (301, 0), (8192 + 300, 8192 - 200), (700, 650), (500, 500), (257, 200)]
    parts = [wl.hca_layer(T=T, H=H, d=128, m=m, W=W, dtype=dtype, seed=95 + i, q_from=q)
             for i, (T, q) in enumerate(seqs)]
    for L in parts:
        L["Kc"] = cast(oracle.compress(L["K"], L["G"], m), dtype)
        L["Vc"] = cast(oracle.compress(L["V"], L["G"], m), dtype)
    R = wl.ragged(parts, ["Q", "K", "V", "Kc", "Vc"])
    bt = R["batch"]
    b = lc.DeviceBatch.from_workload(bt)
    O, lse = lc.hca_dense_attn(dev(R["Q"]), dev(R["Kc"]), dev(R["Vc"]), dev(R["K"]), dev(R["V"]),
                               b, m, W, parts[0]["scale"])
    torch.cuda.synchronize()
    assert lc.last_kernel() == "k_hca_tc"
    gO, gl = f64(O), f64(lse)
    tol = TOL_ATTN[dtype]
    for s, L in enumerate(parts):
        tpos = np.array(L["batch"].positions())
        if len(tpos) == 0:
            continue
        rO, rl = oracle.hca_attn(L["Q"], L["Kc"], L["Vc"], m, L["K"], L["V"], 0, tpos, W,
                                 L["scale"])
        q0, q1 = bt.cu_q[s], bt.cu_q[s + 1]
        np.testing.assert_allclose(gO[q0:q1], rO, rtol=0, atol=tol, err_msg=f"sequence {s}")
        fin = np.isfinite(rl)
        assert np.array_equal(np.isneginf(gl[q0:q1]), ~fin)
        np.testing.assert_allclose(gl[q0:q1][fin], rl[fin], rtol=0, atol=tol)


# ------------------------------------------------------- attention sink

def _sinks(H, seed):
    """Per-head sink logits: head 0 has none (-inf), head 1 one that takes
    almost all of the attention, the rest moderate."""
    s = np.random.default_rng(seed).normal(0.0, 2.0, H)
    s[0] = -np.inf
    s[1] = 40.0
    return s.astype(np.float32)


@pytest.mark.parametrize("kind,dtype,H,d,W,T", [
    ("sparse", "f32", 8, 64, 64, 900),      # SIMT path
    ("sparse", "bf16", 64, 128, 128, 1200),  # tensor-core path
    ("hca", "f32", 8, 64, 64, 1000),
    ("hca", "bf16", 64, 128, 128, 2100),
    ("hca", "bf16", 128, 128, 0, 1000),      # no window: rows t < 127 see only the sink
])
def test_attention_sink(lc, kind, dtype, H, d, W, T):
    sink = _sinks(H, 5)
    sink_d = dev(torch.from_numpy(sink))
    if kind == "sparse":
        m, k = 4, 64
        L, Kc, Vc = _attn_case(dtype, H, d, m, k, W, T, seed=41)
        tpos = np.array(L["batch"].positions())
        sel = oracle.topk(np.random.default_rng(4).standard_normal((len(tpos), T // m)),
                          (tpos + 1) // m, k)
        b = lc.DeviceBatch.from_workload(L["batch"])
        O, lse = lc.sparse_mqa_attn(dev(L["Q"]), dev(Kc), dev(Vc), dev(torch.from_numpy(sel)),
                                    dev(L["K"]), dev(L["V"]), b, m, W, L["scale"], sink=sink_d)
        rO, rl = oracle.sparse_attn(L["Q"], Kc, Vc, sel, L["K"], L["V"], 0, tpos, W, L["scale"],
                                    sink=sink)
    else:
        m = 128
        L = wl.hca_layer(T=T, H=H, d=d, m=m, W=W, dtype=dtype, seed=42)
        Kc = cast(oracle.compress(L["K"], L["G"], m), dtype)
        Vc = cast(oracle.compress(L["V"], L["G"], m), dtype)
        tpos = np.array(L["batch"].positions())
        b = lc.DeviceBatch.from_workload(L["batch"])
        O, lse = lc.hca_dense_attn(dev(L["Q"]), dev(Kc), dev(Vc), dev(L["K"]), dev(L["V"]), b,
                                   m, W, L["scale"], sink=sink_d)
        rO, rl = oracle.hca_attn(L["Q"], Kc, Vc, m, L["K"], L["V"], 0, tpos, W, L["scale"],
                                 sink=sink)
    torch.cuda.synchronize()
    # the path that ran: tensor cores for bf16 with d = 128, SIMT otherwise
    want = ("k_sparse_tc" if kind == "sparse" else "k_hca_tc") if dtype == "bf16" else "k_attn_simt"
    assert lc.last_kernel() == want
    tol = TOL_ATTN[dtype]
    np.testing.assert_allclose(f64(O), rO, rtol=0, atol=tol)
    g, fin = f64(lse), np.isfinite(rl)
    assert np.array_equal(np.isneginf(g), np.isneginf(rl))
    np.testing.assert_allclose(g[fin], rl[fin], rtol=0, atol=tol)
    assert np.abs(f64(O)[:, 1]).max() < 1e-6  # the dominant sink leaves almost nothing


@pytest.mark.parametrize("kind,dtype,H,d", [("sparse", "bf16", 64, 128), ("hca", "bf16", 64, 128),
                                            ("sparse", "f32", 8, 64)])
def test_unusable_sink_is_flagged(lc, kind, dtype, H, d):
    """A NaN or +inf sink logit is flagged (LC_DEVERR_SINK) and that head is
    computed without a sink; the other heads keep theirs.  A sink tensor of
    the wrong length is refused by the binding."""
    T, W, m = 600, 64, 4
    sink = _sinks(H, 6)
    sink[2] = np.nan
    sink[3] = np.inf
    clean = sink.copy()
    clean[2] = clean[3] = -np.inf
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if kind == "sparse":
        L, Kc, Vc = _attn_case(dtype, H, d, m, 32, W, T, seed=44)
        tpos = np.array(L["batch"].positions())
        sel = oracle.topk(np.random.default_rng(5).standard_normal((len(tpos), T // m)),
                          (tpos + 1) // m, 32)
        b = lc.DeviceBatch.from_workload(L["batch"])
        args = (dev(L["Q"]), dev(Kc), dev(Vc), dev(torch.from_numpy(sel)), dev(L["K"]),
                dev(L["V"]), b, m, W, L["scale"])
        O, lse = lc.sparse_mqa_attn(*args, sink=dev(torch.from_numpy(sink)), dev_err=err)
        rO, rl = oracle.sparse_attn(L["Q"], Kc, Vc, sel, L["K"], L["V"], 0, tpos, W, L["scale"],
                                    sink=clean)
        with pytest.raises(ValueError, match="one fp32 logit per head"):
            lc.sparse_mqa_attn(*args, sink=dev(torch.zeros(H - 1)))
    else:
        L = wl.hca_layer(T=T, H=H, d=d, m=m, W=W, dtype=dtype, seed=45)
        Kc = cast(oracle.compress(L["K"], L["G"], m), dtype)
        Vc = cast(oracle.compress(L["V"], L["G"], m), dtype)
        tpos = np.array(L["batch"].positions())
        b = lc.DeviceBatch.from_workload(L["batch"])
        O, lse = lc.hca_dense_attn(dev(L["Q"]), dev(Kc), dev(Vc), dev(L["K"]), dev(L["V"]), b,
                                   m, W, L["scale"], sink=dev(torch.from_numpy(sink)), dev_err=err)
        rO, rl = oracle.hca_attn(L["Q"], Kc, Vc, m, L["K"], L["V"], 0, tpos, W, L["scale"],
                                 sink=clean)
    torch.cuda.synchronize()
    assert int(err.item()) == lc.LC_DEVERR_SINK
    tol = TOL_ATTN[dtype]
    np.testing.assert_allclose(f64(O), rO, rtol=0, atol=tol)
    fin = np.isfinite(rl)
    np.testing.assert_allclose(f64(lse)[fin], rl[fin], rtol=0, atol=tol)


# -------------------------------------------------------------- end to end

def test_csa_tiny_end_to_end(lc):
    """The tiny fp32 setting (T=2048, 8 heads x 64, indexer 4 x 32, k=32,
    W=64, seed 0) through compress -> index + top-k -> attention."""
    L = wl.CONFIGS["csa_tiny"]()
    m, k, W = L["m"], L["k"], L["W"]
    b = lc.DeviceBatch.from_workload(L["batch"])
    tpos = np.array(L["batch"].positions())
    Kc, Vc = lc.csa_compress(dev(L["K"]), dev(L["V"]), dev(L["G"]), m=m)
    _, sel = lc.lightning_index(dev(L["qI"]), dev(L["w"]), dev(L["kI"]), b, m, scores=False,
                                k=k, topk=True)
    O, lse = lc.sparse_mqa_attn(dev(L["Q"]), Kc, Vc, sel, dev(L["K"]), dev(L["V"]), b, m, W,
                                L["scale"])
    torch.cuda.synchronize()
    # oracle pipeline on the same inputs
    rKc = cast(oracle.compress(L["K"], L["G"], m), "f32")
    rVc = cast(oracle.compress(L["V"], L["G"], m), "f32")
    I = oracle.index(L["qI"], L["w"], L["kI"], tpos, m)
    nvis = (tpos + 1) // m
    rsel = oracle.topk(I, nvis, k)
    rO, rl = oracle.sparse_attn(L["Q"], rKc, rVc, rsel, L["K"], L["V"], 0, tpos, W, L["scale"])
    gsel = sel.cpu().numpy()
    _, same = check_selection(gsel, I, nvis, k)
    differ = ~same
    np.testing.assert_allclose(f64(O)[same], rO[same], rtol=0, atol=TOL_ATTN["f32"])
    print(f"excused selection mismatches: {differ.sum()} of {len(differ)} rows")


def test_hca_tc_short_raw_cache_is_flagged(lc):
    # raw cache holding positions 200.. only: windows reaching below 200 are
    # cut there and flagged; rows whose window lies inside it are exact
    L = wl.hca_layer(T=400, H=64, d=128, m=8, W=32, dtype="bf16", seed=43)
    Kc = cast(oracle.compress(L["K"], L["G"], 8), "bf16")
    Vc = cast(oracle.compress(L["V"], L["G"], 8), "bf16")
    batch = wl.Batch(cu_q=[0, 400], q_pos0=[0], cu_c=[0, 50], cu_raw=[0, 200], raw_pos0=[200])
    b = lc.DeviceBatch.from_workload(batch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    O, _ = lc.hca_dense_attn(dev(L["Q"]), dev(Kc), dev(Vc), dev(L["K"][200:]), dev(L["V"][200:]),
                             b, 8, 32, L["scale"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lc.LC_DEVERR_WINDOW
    rows = np.arange(231, 400)
    rO, _ = oracle.hca_attn(L["Q"][rows], Kc, Vc, 8, L["K"][200:], L["V"][200:], 200, rows, 32,
                            L["scale"])
    np.testing.assert_allclose(f64(O)[rows], rO, rtol=0, atol=TOL_ATTN["bf16"])


def test_device_errors_are_flagged_not_trapped(lc):
    L, Kc, Vc = _attn_case("bf16", 8, 64, 4, 4, 4, 64, seed=41)
    b = lc.DeviceBatch.from_workload(L["batch"])
    Nq = L["Q"].shape[0]
    sel = torch.full((Nq, 4), -1, dtype=torch.int32)
    sel[10, 0] = 999          # beyond the stored entries
    sel[12, 1] = 5            # stored, but not visible from t=12 (n_vis = 3)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    O, _ = lc.sparse_mqa_attn(dev(L["Q"]), dev(Kc), dev(Vc), dev(sel), dev(L["K"]), dev(L["V"]),
                              b, 4, 4, L["scale"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lc.LC_DEVERR_INDEX
    assert torch.isfinite(O.float()).all()
    # a raw cache that does not hold the window's positions
    err.zero_()
    short = wl.single(T_raw=8, q_pos0=0, Nq=Nq, Tc=Nq // 4)
    bs = lc.DeviceBatch.from_workload(short)
    lc.hca_dense_attn(dev(L["Q"]), dev(Kc), dev(Vc), dev(L["K"][:8]), dev(L["V"][:8]), bs, 4, 4,
                      L["scale"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lc.LC_DEVERR_WINDOW
