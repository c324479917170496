"""GPU parity of partial RoPE ("DeepSeek-V4 技术解析…", §1.1, engineering
details: RoPE on the last 64 dimensions, inverse RoPE on the core-attention
output) against the CPU oracle.

The GPU pipeline starts from unrotated tokens like the oracle's: the
compressors rotate each entry at its last token's position (rope_pos0), the
window cache is rotated with rope_rotate, and the attention kernels rotate Q
at t and the output back at t.  Bars: rotated rows as `close` states;
attention fp32 1e-4 and bf16 2e-2, where in the bf16 setting the oracle's
rotated q, k and v are bf16 values (the operands the method multiplies)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "bf16": 2e-2}


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


def close(got, ref, dtype, what, unrot):
    """Rotated values: fp32 within 1e-5; bf16 within one bf16 ulp of the exact
    rotation plus an absolute 1e-5 x the pair's magnitude (the fp32 rotation
    before the rounding cancels where the result is small, and the angle at
    positions near 5e9 carries about 1e-6 rad)."""
    g = f64(got)
    u = np.abs(np.asarray(unrot, dtype=np.float64))
    pair = np.maximum(u, u.reshape(*u.shape[:-1], -1, 2)[..., ::-1].reshape(u.shape))
    if dtype == "f32":
        bad = np.abs(g - ref) > 1e-5 * np.maximum(pair, 1.0)
    else:
        bad = np.abs(g - ref) > np.abs(ref) * 2.0 ** -7 + 1e-5 * pair + 1e-30
    assert not bad.any(), f"{what}: {bad.sum()} values outside the bound"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape,pos0", [((300, 128), 0), ((77, 4, 64), 1048500),
                                        ((1000, 2, 128), 5_000_000_000)])
def test_rope_rotate(lc, dtype, shape, pos0):
    g = wl._gen(91, "cpu")
    X = wl.normal(g, shape, dtype, "cpu")
    pos = pos0 + np.arange(shape[0])
    Y = lc.rope_rotate(X.cuda(), pos0)
    torch.cuda.synchronize()
    assert lc.last_kernel() == "k_rope_rows"
    close(Y, oracle.rope(X, pos), dtype, "rotate", f64(X))
    # and back
    Z = lc.rope_rotate(Y.clone(), pos0, inverse=True)
    torch.cuda.synchronize()
    close(Z, oracle.rope(f64(Y), pos, inverse=True), dtype, "rotate back", f64(Y))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind,m,T,d,pos0", [("csa", 4, 1030, 128, 0), ("csa", 4, 512, 64, 4096),
                                             ("hca", 128, 4096 + 5, 128, 1 << 20),
                                             ("tok", 4, 999, 128, 77), ("tok", 128, 1024, 64, 0)])
def test_compress_with_rope(lc, dtype, kind, m, T, d, pos0):
    g = wl._gen(92, "cpu")
    K, V = wl.normal(g, (T, d), dtype, "cpu"), wl.normal(g, (T, d), dtype, "cpu")
    ep = oracle.entry_positions(pos0, T // m, m)
    if kind == "tok":
        Z = wl.normal(g, (T, d), "f32", "cpu") * 2
        got = lc.token_gated_compress(K.cuda(), Z.cuda(), m, rope_pos0=pos0)
        torch.cuda.synchronize()
        ent = oracle.compress_tok(K, Z, m)
        close(got, oracle.rope(ent, ep), dtype, "token-gated entries", ent)
        return
    G = wl.normal(g, (m, d), "f32", "cpu")
    fn = lc.csa_compress if kind == "csa" else lc.hca_compress
    Kc, Vc = fn(K.cuda(), V.cuda(), G.cuda(), m=m, rope_pos0=pos0)
    torch.cuda.synchronize()
    eK, eV = oracle.compress(K, G, m), oracle.compress(V, G, m)
    close(Kc, oracle.rope(eK, ep), dtype, "K entries", eK)
    close(Vc, oracle.rope(eV, ep), dtype, "V entries", eV)


def _rotated_caches(lc, L, m, dev):
    """The GPU side: entries rotated by the compressor, window tokens by
    rope_rotate (both from position 0)."""
    fn = lc.csa_compress if m < 32 else lc.hca_compress
    Kc, Vc = fn(dev["K"], dev["V"], dev["G"], m=m, rope_pos0=0)
    Kr = lc.rope_rotate(dev["K"].clone(), 0)
    Vr = lc.rope_rotate(dev["V"].clone(), 0)
    return Kc, Vc, Kr, Vr


@pytest.mark.parametrize("dtype,H,d,k,W,T,q_from", [
    ("bf16", 64, 128, 64, 128, 1500, 200),    # tensor-core path
    ("bf16", 128, 128, 32, 16, 700, 0),
    ("f32", 8, 64, 32, 64, 900, 100),         # SIMT paths
    ("f32", 16, 128, 16, 8, 400, 0),
])
def test_sparse_attn_with_rope(lc, dtype, H, d, k, W, T, q_from):
    m = 4
    L = wl.csa_layer(T=T, H=H, d=d, HI=4, dI=32, m=m, k=k, W=W, dtype=dtype, seed=93,
                     q_from=q_from)
    dev = {n: (v.cuda() if torch.is_tensor(v) else v) for n, v in L.items()}
    tpos = np.array(L["batch"].positions())
    sel = oracle.topk(np.random.default_rng(7).standard_normal((len(tpos), T // m)),
                      (tpos + 1) // m, k)
    b = lc.DeviceBatch.from_workload(L["batch"])
    Kc, Vc, Kr, Vr = _rotated_caches(lc, L, m, dev)
    O, lse = lc.sparse_mqa_attn(dev["Q"], Kc, Vc, torch.from_numpy(sel).cuda(), Kr, Vr, b, m, W,
                                L["scale"], rope=True)
    torch.cuda.synchronize()
    want = "k_sparse_tc" if dtype == "bf16" else "k_attn_simt"
    assert lc.last_kernel() == want
    rKc, rVc = oracle.compress(L["K"], L["G"], m), oracle.compress(L["V"], L["G"], m)
    op = "bf16" if dtype == "bf16" else None
    rO, rl = oracle.sparse_attn_rope(L["Q"], rKc, rVc, sel, L["K"], L["V"], 0, tpos, W,
                                     L["scale"], m, operand_dtype=op)
    np.testing.assert_allclose(f64(O), rO, rtol=0, atol=TOL[dtype])
    fin = np.isfinite(rl)
    np.testing.assert_allclose(f64(lse)[fin], rl[fin], rtol=0, atol=TOL[dtype])


@pytest.mark.parametrize("dtype,H,d,m,W,T,q_from", [
    ("bf16", 64, 128, 128, 128, 2300, 0),     # tensor-core path
    ("bf16", 128, 128, 16, 40, 900, 300),
    ("bf16", 8, 128, 128, 128, 1100, 0),      # 32 tokens per CTA
    ("f32", 8, 64, 128, 64, 1000, 0),         # SIMT path
])
def test_hca_attn_with_rope(lc, dtype, H, d, m, W, T, q_from):
    L = wl.hca_layer(T=T, H=H, d=d, m=m, W=W, dtype=dtype, seed=94, q_from=q_from)
    dev = {n: (v.cuda() if torch.is_tensor(v) else v) for n, v in L.items()}
    tpos = np.array(L["batch"].positions())
    b = lc.DeviceBatch.from_workload(L["batch"])
    Kc, Vc, Kr, Vr = _rotated_caches(lc, L, m, dev)
    O, lse = lc.hca_dense_attn(dev["Q"], Kc, Vc, Kr, Vr, b, m, W, L["scale"], rope=True)
    torch.cuda.synchronize()
    want = "k_hca_tc" if dtype == "bf16" else "k_attn_simt"
    assert lc.last_kernel() == want
    rKc, rVc = oracle.compress(L["K"], L["G"], m), oracle.compress(L["V"], L["G"], m)
    op = "bf16" if dtype == "bf16" else None
    rO, rl = oracle.hca_attn_rope(L["Q"], rKc, rVc, m, L["K"], L["V"], 0, tpos, W, L["scale"],
                                  operand_dtype=op)
    np.testing.assert_allclose(f64(O), rO, rtol=0, atol=TOL[dtype])
    fin = np.isfinite(rl)
    np.testing.assert_allclose(f64(lse)[fin], rl[fin], rtol=0, atol=TOL[dtype])


def test_hca_with_rope_at_a_million_positions(lc):
    """Queries near position 2^20 (angles up to ~1e6 rad): the last 256
    positions of a 1,048,576-token sequence, HCA m' = 128, 128 heads."""
    T, m, W, H, d = 1 << 20, 128, 128, 128, 128
    q_from = T - 256
    L = wl.hca_layer(T=T, H=H, d=d, m=m, W=W, dtype="bf16", seed=95, q_from=q_from)
    dev = {n: (v.cuda() if torch.is_tensor(v) else v) for n, v in L.items()}
    b = lc.DeviceBatch.from_workload(L["batch"])
    Kc, Vc = lc.hca_compress(dev["K"], dev["V"], dev["G"], m=m, rope_pos0=0)
    # the window cache: the last W + 256 tokens, rotated at their positions
    lo = q_from - W
    Kr = lc.rope_rotate(dev["K"][lo:].clone(), lo)
    Vr = lc.rope_rotate(dev["V"][lo:].clone(), lo)
    bw = lc.DeviceBatch.from_host([0, 256], [q_from], [0, T // m], [0, T - lo], [lo])
    O, _ = lc.hca_dense_attn(dev["Q"], Kc, Vc, Kr, Vr, bw, m, W, L["scale"], rope=True)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 100, 254, 255])
    tpos = q_from + rows
    rKc = oracle.compress(L["K"], L["G"], m)
    rVc = oracle.compress(L["V"], L["G"], m)
    rO, _ = oracle.hca_attn_rope(L["Q"][rows], rKc, rVc, m, L["K"][lo:], L["V"][lo:], lo, tpos,
                                 W, L["scale"], operand_dtype="bf16")
    np.testing.assert_allclose(f64(O)[rows], rO, rtol=0, atol=TOL["bf16"])
