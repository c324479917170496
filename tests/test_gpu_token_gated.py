"""GPU parity of the token-gated compressor (each token brings its own gate
logits, "DeepSeek-V4 技术解析…", §1.1, CSA paragraph) and of a CSA layer
whose K, V and indexer keys all go through it, against the CPU oracle.

Bars: compressed entries fp32 within 1e-5, bf16 a faithful rounding of the
fp64 value (one bf16 ulp); end to end, the fused top-k equal to the
oracle's or different only inside the near-tie band (selection_check) and
attention within 2e-2 (bf16)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from selection_check import check_selection

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("m,T,shape", [(4, 2051, (64,)), (4, 1024, (8, 64)), (128, 4096 + 77, (128,)),
                                       (7, 300, (32,)), (1, 65, (128,)), (16, 5, (64,)),
                                       (4096, 8192, (32,))])
def test_token_gated_compress(lc, dtype, m, T, shape):
    g = wl._gen(13, "cpu")
    X = wl.normal(g, (T, *shape), dtype, "cpu")
    Z = wl.normal(g, (T, *shape), "f32", "cpu") * 3
    got = lc.token_gated_compress(X.cuda(), Z.cuda(), m)
    torch.cuda.synchronize()
    assert lc.last_kernel() == "k_compress_tok" or T // m == 0
    assert got.shape == (T // m, *shape)
    d = int(np.prod(shape))
    ref = oracle.compress_tok(X.reshape(T, d), Z.reshape(T, d), m).reshape(T // m, *shape)
    g64 = f64(got)
    if dtype == "f32":
        np.testing.assert_allclose(g64, ref, rtol=1e-5, atol=1e-6)
    else:
        tol = np.abs(ref) * 2.0 ** -7 + 1e-30
        assert np.all(np.abs(g64 - ref) <= tol)


def test_token_gated_csa_layer_end_to_end(lc):
    """K, V and the indexer keys compressed with per-token gates, then the
    fused index + top-k and the tensor-core CSA attention."""
    T, m, k, W = 4096, 4, 64, 128
    L = wl.csa_layer_token_gated(T=T, H=64, d=128, HI=8, dI=64, m=m, k=k, W=W, dtype="bf16",
                                 seed=81, q_from=3072)
    dev = {n: (v.cuda() if torch.is_tensor(v) else v) for n, v in L.items()}
    b = lc.DeviceBatch.from_workload(L["batch"])
    Kc = lc.token_gated_compress(dev["K"], dev["ZK"], m)
    Vc = lc.token_gated_compress(dev["V"], dev["ZV"], m)
    kI = lc.token_gated_compress(dev["kI_tok"], dev["ZI"], m)
    torch.cuda.synchronize()
    tpos = np.array(L["batch"].positions())
    rKc = oracle.compress_tok(L["K"], L["ZK"], m)
    rVc = oracle.compress_tok(L["V"], L["ZV"], m)
    rkI = oracle.compress_tok(L["kI_tok"].reshape(T, -1), L["ZI"].reshape(T, -1), m)
    # the stored (bf16) entries are faithful roundings of the oracle's
    for got, ref in ((Kc, rKc), (Vc, rVc), (kI.reshape(T // m, -1), rkI)):
        assert np.all(np.abs(f64(got) - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)
    # Two faithful roundings may differ by one ulp, and the selection is not
    # continuous in the keys, so the indexer reads the oracle's rounded keys
    # (the attention absorbs one-ulp differences of Kc/Vc within its tolerance).
    bf = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    rkI_b = bf(rkI).reshape(T // m, 8, 64)
    _, sel = lc.lightning_index(dev["qI"], dev["w"], rkI_b.cuda(), b, m, scores=False, k=k,
                                topk=True)
    O, lse = lc.sparse_mqa_attn(dev["Q"], Kc, Vc, sel, dev["K"], dev["V"], b, m, W, L["scale"])
    torch.cuda.synchronize()
    I = oracle.index(L["qI"], L["w"], rkI_b, tpos, m)
    rsel, same = check_selection(sel.cpu().numpy(), I, (tpos + 1) // m, k)
    assert same.mean() >= 0.95
    rO, rl = oracle.sparse_attn(L["Q"], bf(rKc), bf(rVc), rsel, L["K"], L["V"], 0, tpos, W,
                                L["scale"])
    np.testing.assert_allclose(f64(O)[same], rO[same], rtol=0, atol=2e-2)
    np.testing.assert_allclose(f64(lse)[same], rl[same], rtol=0, atol=2e-2)
