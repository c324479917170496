"""Incremental decode state ("DeepSeek V4 详解…", §"第二刀": a classical cache of
compressed entries plus a per-request state cache holding the window and the
open block's tail), against the one-shot oracle run on each request's whole
token history.

Three requests start at positions 5, 126 and 300 and take 140 decode steps,
so each closes several CSA blocks (m = 4) and at least one HCA block
(m' = 128).  The state before the first step is built with the library's
compressors (tested elsewhere) and plain copies into the ring.  Checked:
after the last step the classical caches against the oracle's compression of
each history (faithful bf16), the ring rows and batch arrays exactly; at
every step the fused index + top-k (equal to the oracle's or inside its
near-tie band), CSA and HCA attention within 2e-2 (bf16)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from selection_check import check_selection

pytestmark = pytest.mark.gpu
TOL = 2e-2
B, R, d, H, m, mh, HI, dI, K_TOP, W = 3, 128, 128, 16, 4, 128, 8, 64, 32, 128
CAP_C, CAP_H = 256, 8
START = [5, 126, 300]
STEPS = 140


@pytest.fixture(scope="module")
def lc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import long_context_compressed_13_b300 as mod
    from long_context_compressed_13_b300 import _build
    _build.build()
    mod.load_library()
    return mod


def f64(x):
    return x.detach().to("cpu").double().numpy()


def faithful(got, exact, mag, m):
    """A bf16 rounding of a value computed in fp32: one bf16 ulp plus the fp32
    accumulation bound of an m-term weighted sum, gamma * sum_p w_p |x_p|
    (mag, the pooling of |x| with the same gates)."""
    u = 2.0 ** -24
    gamma = (m + 2) * u / (1 - (m + 2) * u)
    return np.all(np.abs(f64(got) - exact) <= np.abs(exact) * 2.0 ** -7 + gamma * mag + 1e-30)


def _draw(seed):
    g = wl._gen(seed, "cpu")
    n = max(START) + STEPS
    dr = lambda *s: wl.normal(g, s, "bf16", "cpu")
    S = {"K": dr(B, n, d), "V": dr(B, n, d), "kI": dr(B, n, HI, dI), "Kh": dr(B, n, d),
         "Vh": dr(B, n, d), "G": wl.normal(g, (m, d), "f32", "cpu"),
         "Gh": wl.normal(g, (mh, d), "f32", "cpu"), "Q": dr(B, STEPS, H, d),
         "Qh": dr(B, STEPS, H, d), "qI": dr(B, STEPS, HI, dI),
         "w": wl.uniform(g, (B, STEPS, HI), "f32", "cpu")}
    return S


def _init_layer(lc, L, K, V, G, kI=None, GI=None):
    """Request b holds positions 0 .. START[b]-1: entries from the library's
    compressors, the ring and the open block's indexer keys copied in."""
    for b, s in enumerate(START):
        Kb, Vb = K[b, :s].cuda(), V[b, :s].cuda()
        n = s // L.m
        fn = lc.csa_compress if L.m < 32 else lc.hca_compress
        fn(Kb, Vb, G.cuda(), m=L.m, Kc=L.Kc[b * L.cap:b * L.cap + n],
           Vc=L.Vc[b * L.cap:b * L.cap + n])
        if kI is not None:
            Z = GI.reshape(L.m, -1).repeat(s // L.m + 1, 1)[:s].contiguous()
            lc.token_gated_compress(kI[b, :s].reshape(s, -1).cuda(), Z.cuda(), L.m,
                                    Xc=L.kI[b * L.cap:b * L.cap + n].view(n, -1))
            for p in range(s - s % L.m, s):
                L.kI_ring[b * L.m + p % L.m] = kI[b, p].cuda()
        for p in range(max(0, s - L.R), s):
            r = b * 2 * L.R + p % L.R
            for rr in (r, r + L.R):
                L.Kring[rr] = K[b, p].cuda()
                L.Vring[rr] = V[b, p].cuda()
        L.n_tok[b] = s


def _run(lc, seed, GI, check_steps):
    S = _draw(seed)
    csa = lc.DecodeLayer(B, R, d, m, CAP_C, HI, dI)
    hca = lc.DecodeLayer(B, R, d, mh, CAP_H)
    _init_layer(lc, csa, S["K"], S["V"], S["G"], S["kI"], GI)
    _init_layer(lc, hca, S["Kh"], S["Vh"], S["Gh"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    GIc = GI.reshape(m, -1).cuda()
    scale = 1.0 / np.sqrt(d)
    for i in range(STEPS):
        pos = [s + i for s in START]
        take = lambda name: torch.stack([S[name][b, pos[b]] for b in range(B)]).cuda()
        lc.decode_append(csa, take("K"), take("V"), S["G"].cuda(), kI_new=take("kI"), G_I=GIc,
                         dev_err=err)
        lc.decode_append(hca, take("Kh"), take("Vh"), S["Gh"].cuda(), dev_err=err)
        if not check_steps:
            continue
        Q, Qh, qI, w = (S[n][:, i].contiguous().cuda() for n in ("Q", "Qh", "qI", "w"))
        _, sel = lc.lightning_index(qI, w, csa.kI, csa.batch, m, scores=False, k=K_TOP, topk=True,
                                    dev_err=err)
        O, _ = lc.sparse_mqa_attn(Q, csa.Kc, csa.Vc, sel, csa.Kring, csa.Vring, csa.batch, m, W,
                                  scale, dev_err=err)
        Oh, _ = lc.hca_dense_attn(Qh, hca.Kc, hca.Vc, hca.Kring, hca.Vring, hca.batch, mh, W,
                                  scale, dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"step {i}: device error {int(err.item())}"
        gsel, gO, gOh = sel.cpu().numpy(), f64(O), f64(Oh)
        for b in range(B):
            t = pos[b]
            Kt, Vt, kIt = S["K"][b, :t + 1], S["V"][b, :t + 1], S["kI"][b, :t + 1]
            Kc = f64(torch.from_numpy(oracle.compress(Kt, S["G"], m)).to(torch.bfloat16))
            Vc = f64(torch.from_numpy(oracle.compress(Vt, S["G"], m)).to(torch.bfloat16))
            kIc = torch.from_numpy(oracle.compress(kIt.reshape(t + 1, -1), GI.reshape(m, -1),
                                                   m)).to(torch.bfloat16).reshape(-1, HI, dI)
            I = oracle.index(S["qI"][b, i:i + 1], S["w"][b, i:i + 1], kIc, [t], m)
            rsel, same = check_selection(gsel[b:b + 1], I, [(t + 1) // m], K_TOP)
            lo = max(0, t - W + 1)
            if same[0]:
                rO, _ = oracle.sparse_attn(S["Q"][b, i:i + 1], Kc, Vc, rsel, Kt[lo:], Vt[lo:], lo,
                                           [t], W, scale)
                np.testing.assert_allclose(gO[b:b + 1], rO, rtol=0, atol=TOL,
                                           err_msg=f"step {i} request {b}")
            Kht, Vht = S["Kh"][b, :t + 1], S["Vh"][b, :t + 1]
            Khc = f64(torch.from_numpy(oracle.compress(Kht, S["Gh"], mh)).to(torch.bfloat16))
            Vhc = f64(torch.from_numpy(oracle.compress(Vht, S["Gh"], mh)).to(torch.bfloat16))
            rOh, _ = oracle.hca_attn(S["Qh"][b, i:i + 1], Khc, Vhc, mh, Kht[lo:], Vht[lo:], lo,
                                     [t], W, scale)
            np.testing.assert_allclose(gOh[b:b + 1], rOh, rtol=0, atol=TOL,
                                       err_msg=f"HCA step {i} request {b}")
    torch.cuda.synchronize()
    return S, csa, hca, err


def test_decode_state_caches_after_steps(lc):
    g = wl._gen(201, "cpu")
    GI = wl.normal(g, (m, HI, dI), "f32", "cpu")
    S, csa, hca, err = _run(lc, 202, GI, check_steps=False)
    assert int(err.item()) == 0
    for b, s in enumerate(START):
        t = s + STEPS  # tokens held
        assert int(csa.n_tok[b]) == t and int(hca.n_tok[b]) == t
        # batch arrays point at the newest token and the ring's oldest position
        lo = max(0, t - R)
        assert int(csa.q_pos0[b]) == t - 1 and int(csa.raw_pos0[b]) == lo
        assert int(csa.cu_raw[b]) == b * 2 * R + lo % R
        # classical caches: every entry of the history
        for L, Kn, Vn, G in ((csa, "K", "V", S["G"]), (hca, "Kh", "Vh", S["Gh"])):
            n = t // L.m
            for cache, name in ((L.Kc, Kn), (L.Vc, Vn)):
                X = S[name][b, :t]
                assert faithful(cache[b * L.cap:b * L.cap + n], oracle.compress(X, G, L.m),
                                oracle.compress(X.abs(), G, L.m), L.m), (name, b)
            # ring: row of position p holds the token, in both mirror slots
            for p in range(t - R, t):
                r = b * 2 * R + p % R
                assert torch.equal(L.Kring[r].cpu(), S[Kn][b, p])
                assert torch.equal(L.Kring[r + R].cpu(), S[Kn][b, p])
        n = t // m
        X = S["kI"][b, :t].reshape(t, -1)
        kIc = oracle.compress(X, GI.reshape(m, -1), m)
        assert faithful(csa.kI[b * CAP_C:b * CAP_C + n].reshape(n, -1), kIc,
                        oracle.compress(X.abs(), GI.reshape(m, -1), m), m)
        for p in range(t - t % m, t):
            assert torch.equal(csa.kI_ring[b * m + p % m].cpu(), S["kI"][b, p])


def test_decode_state_steps_match_the_oracle(lc):
    # one dominant indexer gate (each entry's indexer key is exactly one of its
    # tokens'): both sides then hold the same indexer keys bit for bit
    GI = torch.zeros(m, HI, dI)
    GI[2] = 60.0
    _run(lc, 203, GI, check_steps=True)


def test_decode_append_refuses_a_full_cache(lc):
    L = lc.DecodeLayer(1, 8, 64, 4, 2)  # room for 2 entries (8 tokens)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    G = torch.zeros(4, 64, device="cuda")
    x = torch.ones(1, 64, dtype=torch.bfloat16, device="cuda")
    for _ in range(12):
        lc.decode_append(L, x, x, G, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == lc.LC_DEVERR_BATCH  # the third block had no room
    assert int(L.n_tok[0]) == 12
