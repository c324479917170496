"""GPU parity of the tensor-core Lightning Indexer and of its fused exact
top-k (sampled threshold -> candidate filter -> exact selection -> per-row
fallback) against the CPU oracle.

Bars: scores within a rigorous fp32 accumulation bound, invisible entries
exactly -inf; fused selections equal the oracle's, or differ from it only
inside the near-tie band at the k-th boundary (selection_check: boundary gap
below 1e-5, every kept entry within 1e-5 below the oracle's k-th score,
every left-out entry within 1e-5 above it)."""
import math

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


def _bound(qI, w, kI):
    q, k, ww = f64(qI), f64(kI), f64(w)
    mag = np.einsum("rh,rjh->rj", np.abs(ww), np.einsum("rhe,jhe->rjh", np.abs(q), np.abs(k)))
    n = q.shape[2] + q.shape[1] + 2
    u = 2.0 ** -24
    return mag * (n * u / (1 - n * u)) + 1e-30


def _check_selection(gsel, I, nvis, k):
    """gsel: GPU top-k; I: oracle scores.  Returns the number of excused rows."""
    _, same = check_selection(gsel, I, nvis, k)
    return int((~same).sum())


@pytest.mark.parametrize("HI,T,m,q_from", [(8, 2048, 4, 0), (4, 2304, 4, 100), (8, 1400, 8, 0)])
def test_tc_scores(lc, HI, T, m, q_from):
    L = wl.csa_layer(T=T, H=8, d=64, HI=HI, dI=64, m=m, k=16, W=16, dtype="bf16", seed=71,
                     q_from=q_from)
    b = lc.DeviceBatch.from_workload(L["batch"])
    tpos = np.array(L["batch"].positions())
    ld = b.max_c + 12  # columns past the stored entries are -inf too
    sc = torch.full((b.total_q, ld), 7.0, device="cuda")
    lc.lightning_index(L["qI"].cuda(), L["w"].cuda(), L["kI"].cuda(), b, m, scores=sc)
    torch.cuda.synchronize()
    ref = oracle.index(L["qI"], L["w"], L["kI"], tpos, m)
    got = sc.cpu().double().numpy()
    assert np.all(np.isneginf(got[:, b.max_c:]))
    got = got[:, : b.max_c]
    vis = np.isfinite(ref)
    assert np.array_equal(np.isneginf(got), ~vis)
    bound = _bound(L["qI"], L["w"], L["kI"])
    err = np.abs(got[vis] - ref[vis])
    assert np.all(err <= bound[vis]), f"max err {err.max()}"


@pytest.mark.parametrize("k,T,q_from", [(64, 4096, 0), (32, 2048, 1000), (512, 16384, 12000)])
def test_fused_topk_prefill(lc, k, T, q_from):
    L = wl.csa_layer(T=T, H=8, d=64, HI=8, dI=64, m=4, k=k, W=16, dtype="bf16", seed=72,
                     q_from=q_from)
    b = lc.DeviceBatch.from_workload(L["batch"])
    tpos = np.array(L["batch"].positions())
    _, sel = lc.lightning_index(L["qI"].cuda(), L["w"].cuda(), L["kI"].cuda(), b, 4,
                                scores=False, k=k, topk=True)
    torch.cuda.synchronize()
    I = oracle.index(L["qI"], L["w"], L["kI"], tpos, 4)
    n = _check_selection(sel.cpu().numpy(), I, (tpos + 1) // 4, k)
    print(f"excused rows: {n} of {len(tpos)}")


def test_fused_topk_long_rows_sampled(lc):
    # 32768 entries per row: the sampled threshold uses every 32nd entry
    T, k = 131072, 64
    L = wl.csa_layer(T=T, H=8, d=64, HI=8, dI=64, m=4, k=k, W=16, dtype="bf16", seed=73,
                     q_from=T - 256)
    b = lc.DeviceBatch.from_workload(L["batch"])
    tpos = np.array(L["batch"].positions())
    _, sel = lc.lightning_index(L["qI"].cuda(), L["w"].cuda(), L["kI"].cuda(), b, 4,
                                scores=False, k=k, topk=True)
    torch.cuda.synchronize()
    I = oracle.index(L["qI"], L["w"], L["kI"], tpos, 4)
    _check_selection(sel.cpu().numpy(), I, (tpos + 1) // 4, k)


def test_fused_topk_skewed_rows_overflow(lc):
    # every row's best entries sit in one 1024-entry range (keys scaled by 4,
    # head weights made non-negative), inside one 2048-entry CTA column of the
    # candidate pass: about 640 candidates per row against 256 private slots,
    # so most of them go through the row's shared overflow region
    T, k = 131072, 64
    L = wl.csa_layer(T=T, H=8, d=64, HI=8, dI=64, m=4, k=k, W=16, dtype="bf16", seed=75,
                     q_from=T - 256)
    w = L["w"].abs()
    kI = L["kI"].clone()
    kI[4096:5120] = kI[4096:5120] * 4
    b = lc.DeviceBatch.from_workload(L["batch"])
    tpos = np.array(L["batch"].positions())
    _, sel = lc.lightning_index(L["qI"].cuda(), w.cuda(), kI.cuda(), b, 4, scores=False, k=k,
                                topk=True)
    torch.cuda.synchronize()
    I = oracle.index(L["qI"], w, kI, tpos, 4)
    gsel = sel.cpu().numpy()
    _check_selection(gsel, I, (tpos + 1) // 4, k)
    assert np.mean((gsel >= 4096) & (gsel < 5120)) > 0.9  # the skew is what was tested


def test_fused_topk_ties_take_the_fallback(lc):
    # rows with all-zero indexer queries or head weights score every entry 0:
    # the candidate list overflows and the exact fallback keeps the lowest
    # indices; the other rows go through the candidate path
    T, k = 16384, 128
    L = wl.csa_layer(T=T, H=8, d=64, HI=8, dI=64, m=4, k=k, W=16, dtype="bf16", seed=74,
                     q_from=T - 512)
    qI, w = L["qI"].clone(), L["w"].clone()
    qI[5:9] = 0
    w[100:103] = 0
    qI[200, :, :] = -qI[200, :, :].abs()  # some heads positive, some negative per entry
    b = lc.DeviceBatch.from_workload(L["batch"])
    tpos = np.array(L["batch"].positions())
    _, sel = lc.lightning_index(qI.cuda(), w.cuda(), L["kI"].cuda(), b, 4, scores=False, k=k,
                                topk=True)
    torch.cuda.synchronize()
    I = oracle.index(qI, w, L["kI"], tpos, 4)
    gsel = sel.cpu().numpy()
    for r in list(range(5, 9)) + [100, 101, 102]:
        assert gsel[r].tolist() == list(range(k))
    _check_selection(gsel, I, (tpos + 1) // 4, k)


def test_fused_topk_rows_past_the_warp_bitmaps(lc):
    # 40960 entries per row: more than the warp-per-row pick's bitmaps hold,
    # so the CTA-per-row pick runs; rows with all-zero scores fail the
    # candidate check and go through the fallback's recomputed rows
    T, k = 163840, 256
    L = wl.csa_layer(T=T, H=8, d=64, HI=8, dI=64, m=4, k=k, W=16, dtype="bf16", seed=76,
                     q_from=T - 192)
    qI, w = L["qI"].clone(), L["w"].clone()
    qI[3] = 0
    w[150] = 0
    b = lc.DeviceBatch.from_workload(L["batch"])
    tpos = np.array(L["batch"].positions())
    _, sel = lc.lightning_index(qI.cuda(), w.cuda(), L["kI"].cuda(), b, 4, scores=False, k=k,
                                topk=True)
    torch.cuda.synchronize()
    assert lc.last_kernel() == "k_topk_fallback"
    I = oracle.index(qI, w, L["kI"], tpos, 4)
    gsel = sel.cpu().numpy()
    for r in (3, 150):
        assert gsel[r].tolist() == list(range(k))
    _check_selection(gsel, I, (tpos + 1) // 4, k)


@pytest.mark.parametrize("dtype,HI,dI", [("f32", 4, 32), ("bf16", 2, 64)])
def test_fused_topk_in_row_chunks_equals_one_pass(lc, dtype, HI, dI):
    # without the tensor-core plan the fused call keeps the scores of as many
    # rows as the workspace holds and selects them chunk by chunk: the result
    # is the one of a workspace that holds every row
    T, k = 4096, 32
    L = wl.csa_layer(T=T, H=8, d=64, HI=HI, dI=dI, m=4, k=k, W=16, dtype=dtype, seed=77,
                     q_from=T - 300)
    b = lc.DeviceBatch.from_workload(L["batch"])
    qI, w, kI = L["qI"].cuda(), L["w"].cuda(), L["kI"].cuda()
    row = 4 * b.max_c
    full = torch.empty(300 * row, dtype=torch.uint8, device="cuda")
    small = torch.empty(7 * row + 5, dtype=torch.uint8, device="cuda")  # 7 rows at a time
    _, a = lc.lightning_index(qI, w, kI, b, 4, scores=False, k=k, topk=True, ws=full)
    _, c = lc.lightning_index(qI, w, kI, b, 4, scores=False, k=k, topk=True, ws=small)
    torch.cuda.synchronize()
    assert torch.equal(a, c)
    tpos = np.array(L["batch"].positions())
    I = oracle.index(L["qI"], L["w"], L["kI"], tpos, 4)
    _check_selection(c.cpu().numpy(), I, (tpos + 1) // 4, k)


# ---------------------------------------------------- ragged batches

# (T, q_from) per sequence: sequence-local row tiles that end part-way, a
# sequence of five rows, one without query rows, entries that start at
# offsets which are not multiples of any tile or sampling stride
RAGGED_SEQS = [(1400, 0), (3000, 2900), (700, 695), (2048, 2048), (2500, 2300)]


@pytest.mark.parametrize("HI", [8, 4])
def test_tc_scores_ragged(lc, HI):
    parts = [wl.csa_layer(T=T, H=8, d=64, HI=HI, dI=64, m=4, k=16, W=16, dtype="bf16",
                          seed=80 + i, q_from=q) for i, (T, q) in enumerate(RAGGED_SEQS)]
    R = wl.ragged(parts, ["qI", "w", "kI"])
    bt = R["batch"]
    b = lc.DeviceBatch.from_workload(bt)
    ld = b.max_c + 12
    sc = torch.full((b.total_q, ld), 7.0, device="cuda")
    lc.lightning_index(R["qI"].cuda(), R["w"].cuda(), R["kI"].cuda(), b, 4, scores=sc)
    torch.cuda.synchronize()
    assert lc.last_kernel() == "k_index_tc<materialize>"
    got = sc.cpu().double().numpy()
    for s, L in enumerate(parts):
        rows = got[bt.cu_q[s]:bt.cu_q[s + 1]]
        Tc = bt.cu_c[s + 1] - bt.cu_c[s]
        assert np.all(np.isneginf(rows[:, Tc:])), f"sequence {s}"
        tpos = np.array(L["batch"].positions())
        if len(tpos) == 0:
            continue
        ref = oracle.index(L["qI"], L["w"], L["kI"], tpos, 4)
        rows = rows[:, :Tc]
        vis = np.isfinite(ref)
        assert np.array_equal(np.isneginf(rows), ~vis), f"sequence {s}"
        bound = _bound(L["qI"], L["w"], L["kI"])
        assert np.all(np.abs(rows[vis] - ref[vis]) <= bound[vis]), f"sequence {s}"


@pytest.mark.parametrize("long_T", [32768, 140000])
def test_fused_topk_ragged(lc, long_T):
    # one batch of sequences of very different lengths.  The sampled threshold
    # reads every s-th entry of each sequence from that sequence's own first
    # entry (s = 32 here, and sequence starts that are not multiples of it);
    # rows of the short sequences hold k or fewer visible entries; sequence 1's
    # rows see 4000 tied best entries, more than the candidate capacity, which
    # the fallback settles from that sequence's own keys (the lowest indices).
    # long_T = 140000 gives rows past the warp pick's bitmaps: the CTA-per-row
    # pick runs for every row.
    k = 64
    seqs = [(long_T, long_T - 40), (20000, 19900), (777, 700), (300, 0), (5001, 4990)]
    parts = [wl.csa_layer(T=T, H=8, d=64, HI=8, dI=64, m=4, k=k, W=16, dtype="bf16",
                          seed=90 + i, q_from=q) for i, (T, q) in enumerate(seqs)]
    parts[1]["qI"] = parts[1]["qI"].abs()
    parts[1]["kI"] = parts[1]["kI"].clone()
    parts[1]["kI"][:4000] = 3.0
    R = wl.ragged(parts, ["qI", "w", "kI"])
    bt = R["batch"]
    b = lc.DeviceBatch.from_workload(bt)
    _, sel = lc.lightning_index(R["qI"].cuda(), R["w"].cuda(), R["kI"].cuda(), b, 4,
                                scores=False, k=k, topk=True)
    torch.cuda.synchronize()
    assert lc.last_kernel() == "k_topk_fallback"
    gsel = sel.cpu().numpy()
    for s, L in enumerate(parts):
        g = gsel[bt.cu_q[s]:bt.cu_q[s + 1]]
        tpos = np.array(L["batch"].positions())
        I = oracle.index(L["qI"], L["w"], L["kI"], tpos, 4)
        if s == 1:
            assert all(r.tolist() == list(range(k)) for r in g)
        _check_selection(g, I, (tpos + 1) // 4, k)
