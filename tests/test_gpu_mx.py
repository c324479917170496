"""Low-precision indexer ("DeepSeek V4 详解…", §"mHC、Muon、FP4": FP4 in the CSA
indexer's QK path, the quantized selector keeps almost all of the exact
selection) against the oracle's MX quantizer and indexer, through the C ABI.

- mx_quantize: codes and scales bit-exact against oracle.mx_quantize (both
  decide every code in exact arithmetic: the block scale is a power of two,
  the element rounding is round-to-nearest-even), MXFP8 and MXFP4, fp32 and
  bf16 inputs, with zero blocks, saturating blocks, tie values, values in the
  elements' subnormal range and negative values that round to zero;
- lightning_index_mx: scores within the fp32 accumulation bound of the
  oracle's score of the dequantized q and k; invisible entries exactly -inf;
- the fused top-k of those scores: equal to the oracle's selection on its own
  quantized scores, or different only inside the near-tie band;
- recall of the quantized selection against the exact (unquantized) oracle
  selection, reported and held above a floor measured for these synthetic
  inputs (unit-normal keys leave many near-ties at the k-th score, so the
  recall is below what a trained indexer reaches).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from selection_check import check_selection

pytestmark = pytest.mark.gpu
FMTS = [8, 4]
RECALL_FLOOR = {8: 0.90, 4: 0.75}


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


def _packed(codes: np.ndarray, fmt: int) -> np.ndarray:
    """Oracle codes in the library's byte layout (E2M1: two per byte, the
    even-indexed value in the low nibble)."""
    c = codes.reshape(-1).astype(np.uint8)
    if fmt == 8:
        return c
    return (c[0::2] & 15) | ((c[1::2] & 15) << 4)


def _special_values(n_blocks: int, rng) -> np.ndarray:
    X = rng.standard_normal((n_blocks, 32)) * 2.0 ** rng.integers(-20, 20, (n_blocks, 1))
    X[0] = 0.0                                    # all-zero block
    X[1, :4] = [500.0, -479.0, 3.0, -0.0]         # saturates to 448 (MXFP8)
    X[2, :] = 0.0
    X[2, :8] = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]  # E2M1 ties at unit scale
    X[3, :] = 0.0
    X[3, :6] = [448.0, 1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, -2.0 ** -12]  # E4M3 ties
    X[4, :] = 1e-3
    X[4, 0] = 7.9                                 # tiny values round to zero
    X[4, 1] = -1e-3                               # negative value that rounds to -0
    return X


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_mx_quantize_bit_exact(lc, fmt, dtype):
    rng = np.random.default_rng(7)
    X = torch.from_numpy(_special_values(2048 + 5, rng)).to(wl.DTYPES[dtype])
    codes, scales = lc.mx_quantize(X.cuda(), fmt)
    torch.cuda.synchronize()
    rc, rs, _ = oracle.mx_quantize(X.double().numpy(), fmt)
    np.testing.assert_array_equal(scales.cpu().numpy().reshape(-1), rs)
    got = codes.cpu().numpy().reshape(-1)
    np.testing.assert_array_equal(got, _packed(rc, fmt))


def _layer(HI, seed, B=6, lo=3000, hi=9000, k=256):
    return wl.csa_decode(B=B, ctx_lo=lo, ctx_hi=hi, H=8, d=64, HI=HI, dI=64, m=4, k=k, W=16,
                         dtype="bf16", seed=seed)


def _index_bound(q, w, k, tpos, m):
    """fp32 evaluation bound of the score (as the bf16 indexer's parity
    test): gamma_n times the sum of |terms|, n = dI + HI + 2."""
    absdot = np.einsum("rhe,jhe->rjh", np.abs(q), np.abs(k))
    mag = np.einsum("rh,rjh->rj", np.abs(w), absdot)
    n = q.shape[2] + q.shape[1] + 2
    u = 2.0 ** -24
    return mag * (n * u / (1 - n * u)) + 1e-30


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("HI", [8, 4])
def test_mx_index_scores_and_selection(lc, fmt, HI):
    D = _layer(HI, seed=31 + HI + fmt)
    bt = D["batch"]
    b = lc.DeviceBatch.from_workload(bt)
    qc, qs = lc.mx_quantize(D["qI"].cuda(), fmt)
    kc, ks = lc.mx_quantize(D["kI"].cuda(), fmt)
    k = D["k"]
    sc, sel = lc.lightning_index_mx(fmt, qc, qs, D["w"].cuda(), kc, ks, b, 4, k=k, topk=True)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, sel2 = lc.lightning_index_mx(fmt, qc, qs, D["w"].cuda(), kc, ks, b, 4, scores=False, k=k,
                                    topk=True, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(sel, sel2)
    got, gsel = sc.cpu().double().numpy(), sel.cpu().numpy()
    _, _, qd = oracle.mx_quantize(D["qI"], fmt)
    _, _, kd = oracle.mx_quantize(D["kI"], fmt)
    w = D["w"].double().numpy()
    recalls = []
    for s in range(bt.B):
        c0, c1 = bt.cu_c[s], bt.cu_c[s + 1]
        t = np.array([bt.q_pos0[s]])
        I = oracle.index(qd[s:s + 1], w[s:s + 1], kd[c0:c1], t, 4)
        vis = np.isfinite(I[0])
        row = got[s, :c1 - c0]
        assert np.array_equal(np.isneginf(row), ~vis)
        bound = _index_bound(qd[s:s + 1], w[s:s + 1], kd[c0:c1], t, 4)[0]
        assert np.all(np.abs(row[vis] - I[0][vis]) <= bound[vis]), f"sequence {s}"
        nv = [(bt.q_pos0[s] + 1) // 4]
        check_selection(gsel[s:s + 1], I, nv, k)
        # recall against the exact selector of the unquantized inputs
        Ie = oracle.index(D["qI"][s:s + 1], D["w"][s:s + 1], D["kI"][c0:c1], t, 4)
        ref = oracle.topk(Ie, nv, k)[0]
        recalls.append(len(np.intersect1d(ref[ref >= 0], gsel[s][gsel[s] >= 0])) / min(k, nv[0]))
    print(f"MXFP{fmt} HI={HI}: recall {np.mean(recalls):.4f} (min {np.min(recalls):.4f})")
    assert np.mean(recalls) >= RECALL_FLOOR[fmt]


def test_mx_index_rejects_bad_arguments(lc):
    D = _layer(8, seed=3, B=2)
    b = lc.DeviceBatch.from_workload(D["batch"])
    qc, qs = lc.mx_quantize(D["qI"].cuda(), 8)
    kc, ks = lc.mx_quantize(D["kI"].cuda(), 8)
    with pytest.raises(lc.LCError) as e:
        lc.lightning_index_mx(5, qc, qs, D["w"].cuda(), kc, ks, b, 4)
    assert e.value.status == 1
    with pytest.raises(lc.LCError) as e:  # misaligned key codes
        lc.lightning_index_mx(8, qc, qs, D["w"].cuda(), kc.view(-1)[1:1 + kc.numel() - 16],
                              ks, b, 4)
    assert e.value.status == 1


def test_mx_index_in_row_chunks(lc):
    D = _layer(8, seed=5, B=9)
    b = lc.DeviceBatch.from_workload(D["batch"])
    qc, qs = lc.mx_quantize(D["qI"].cuda(), 4)
    kc, ks = lc.mx_quantize(D["kI"].cuda(), 4)
    row = 4 * b.max_c
    out = []
    for nbytes in (9 * row, 2 * row + 3):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        _, sel = lc.lightning_index_mx(4, qc, qs, D["w"].cuda(), kc, ks, b, 4, scores=False,
                                       k=D["k"], topk=True, ws=ws)
        out.append(sel)
    torch.cuda.synchronize()
    assert torch.equal(out[0], out[1])
