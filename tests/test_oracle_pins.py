"""Pins for the CPU oracle: each test checks the oracle against something
other than itself -- a worked example printed or hand-derived from the
pages, a closed form, an invariant of the mathematics, or brute force on
tiny inputs written independently here with numpy.

Sources: Quant VideoGen notes (papernotes.org): "core tension" (quantiser),
"overall framework" (dequant S*X_INT + C_i, BF16 centroids),
"Semantic-Aware Smoothing", "Progressive Residual Quantization" (stages,
error falls with stages), "algorithm-system co-design" (packed INT2).
The 2-bit quantisation trap (cloud.baidu.com), section 2 (toy quantiser,
"rounding error at most half a scale").  QuantWM write-up (loncent.com),
QSAC and PSAC (top-8 eigenvectors of the history-query second moment).
"""
import math
import os

import numpy as np
import pytest

from video_diffusion_kv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "p1_worked_example.txt")


def _cases():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition(" ")
        if key == "case":
            cur = {"name": val}
            cases.append(cur)
        else:
            cur[key] = val.split()
    return cases


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_worked_example(orc, case):
    bits, mode = int(case["bits"][0]), int(case["mode"][0])
    x = np.zeros(64, np.float32)
    x[:8] = [float(v) for v in case["input"]]
    s, q, rh = orc.quant_group(x, bits=bits, mode=mode)
    assert orc.f16_bits_to_f32(s) == float(case["scale"][0])
    want_q = np.zeros(64, np.int32)
    want_q[:8] = [int(v) for v in case["codes"]]
    np.testing.assert_array_equal(q, want_q)
    want_x = np.zeros(64, np.float32)
    want_x[:8] = [float(v) for v in case["dequant"]]
    np.testing.assert_array_equal(rh, want_x)
    packed = orc.pack_row(q, bits)
    np.testing.assert_array_equal(packed, np.array([int(b, 16) for b in case["bytes"]], np.uint8))
    np.testing.assert_array_equal(orc.unpack_row(packed, 64, bits), q)


@pytest.mark.parametrize("bits,mode,G", [(2, 0, 32), (2, 0, 64), (4, 0, 32), (4, 0, 64), (2, 1, 64)])
def test_rounding_error_bound(orc, bits, mode, G):
    """|r - r_hat| <= S'/2 for every element the clamp does not touch
    (the page's 'rounding error at most half a scale'); the element with
    |r| = amax maps to +-qmax in the QVG form, so nothing is clipped there."""
    rng = np.random.default_rng(1)
    qmax = (1 << (bits - 1)) - 1
    for trial in range(400):
        r = (rng.standard_normal(G) * 10.0 ** rng.uniform(-3, 1.5)).astype(np.float32)
        if trial % 7 == 0:
            r[rng.integers(0, G)] *= 300.0
        s, q, rh = orc.quant_group(r, bits=bits, mode=mode)
        Sp = float(orc.f16_bits_to_f32(s))
        S = float(np.float32(np.abs(r).max()) / np.float32(qmax if mode == 0 else 2))
        assert abs(Sp - S) <= S * 2.0 ** -11 + 6e-8
        assert q.min() >= -(1 << (bits - 1)) and q.max() <= qmax
        unclipped = np.abs(r / np.float32(Sp)) < qmax + 0.5
        err = np.abs(r.astype(np.float64) - rh.astype(np.float64))
        tol = Sp / 2 * (1 + 2.0 ** -22) + 1e-30
        assert np.all(err[unclipped] <= tol)
        if mode == 0:
            assert unclipped.all()
            k = int(np.argmax(np.abs(r)))
            assert abs(q[k]) == qmax
        np.testing.assert_array_equal(rh, np.float32(Sp) * q.astype(np.float32))


def test_scale_saturates_at_fp16_max(orc):
    """A scale beyond fp16 range is stored as 65504 and the codes clip."""
    r = np.zeros(32, np.float32)
    r[0], r[1] = 2.0e5, -1.0e5
    s, q, rh = orc.quant_group(r, bits=2, mode=0)
    assert orc.f16_bits_to_f32(s) == 65504.0
    assert q[0] == 1 and q[1] == -2 and not q[2:].any()  # 2e5/65504 -> 3 clips to 1; -1e5/65504 -> -2


def test_zero_group(orc):
    s, q, rh = orc.quant_group(np.zeros(32, np.float32), bits=2, mode=0)
    assert s == 0 and not q.any() and not rh.any()


def test_pack_roundtrip(orc):
    rng = np.random.default_rng(2)
    for bits in (2, 4):
        for d in (64, 128):
            q = rng.integers(-(1 << (bits - 1)), 1 << (bits - 1), size=d).astype(np.int32)
            b = orc.pack_row(q, bits)
            assert b.size == d * bits // 8
            np.testing.assert_array_equal(orc.unpack_row(b, d, bits), q)
            # element j lives at bit (j*bits) % 8 of byte (j*bits)//8
            j = 5
            u = (int(b[(j * bits) // 8]) >> ((j * bits) % 8)) & ((1 << bits) - 1)
            assert u - (1 << (bits - 1)) == q[j]


def test_init_picks(orc):
    for N, C in [(256, 16), (4680, 256), (300, 300), (2640, 256)]:
        idx = orc.init_picks(N, C, seed=5, chunk=3, head=1, stage=0)
        assert len(set(idx.tolist())) == C
        assert idx.min() >= 0 and idx.max() < N
        # one pick per stratum: idx_c = floor(t), t in [c N / C, (c+1) N / C)
        lo = np.floor(np.arange(C) * N / C)
        hi = (np.arange(C) + 1) * N / C
        assert np.all(idx >= lo) and np.all(idx < hi)
    a = orc.init_picks(4680, 256, 1, 0, 0, 0)
    b = orc.init_picks(4680, 256, 2, 0, 0, 0)
    c = orc.init_picks(4680, 256, 1, 0, 1, 0)
    assert (a != b).any() and (a != c).any()


def _brute_assign(g, cent, w):
    diff = g[:, None, :].astype(np.float64) - cent[None, :, :].astype(np.float64)
    dist = (diff * diff * w[None, None, :].astype(np.float64)).sum(-1)
    return dist


def test_assign_brute_force(orc):
    rng = np.random.default_rng(3)
    g = synth.bf16_values(rng.standard_normal((50, 16)).astype(np.float32))
    cent = synth.bf16_values(rng.standard_normal((7, 16)).astype(np.float32))
    for w in (None, rng.uniform(0.1, 3.0, 16).astype(np.float32)):
        ids, b1, b2, den = orc.assign(g, cent, w)
        ww = np.ones(16, np.float32) if w is None else w
        dist = _brute_assign(g, cent, ww)
        np.testing.assert_array_equal(ids, dist.argmin(1))
        srt = np.sort(dist, 1)
        np.testing.assert_allclose(b1, srt[:, 0], rtol=1e-12)
        np.testing.assert_allclose(b2, srt[:, 1], rtol=1e-12)
        want_den = (g.astype(np.float64) ** 2 * ww).sum(1) + (cent[ids].astype(np.float64) ** 2 * ww).sum(1)
        np.testing.assert_allclose(den, want_den, rtol=1e-12)
    # exact tie between two identical centroids goes to the lower index
    cent2 = np.concatenate([cent[:3], cent[1:2]], 0)
    ids, *_ = orc.assign(cent2[3:4], cent2)
    assert ids[0] == 1


def test_update_is_member_mean(orc):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((40, 8)).astype(np.float32)
    ids = rng.integers(0, 5, 40).astype(np.int32)
    ids[ids == 3] = 2  # cluster 3 empty
    prev = synth.bf16_values(rng.standard_normal((5, 8)).astype(np.float32))
    cent, mean, cnt = orc.update(x, ids, prev)
    for c in range(5):
        m = x[ids == c].astype(np.float64)
        assert cnt[c] == len(m)
        if len(m):
            np.testing.assert_allclose(mean[c], m.mean(0), rtol=1e-6, atol=1e-7)
            np.testing.assert_array_equal(cent[c], synth.bf16_values(mean[c]))
        else:
            np.testing.assert_array_equal(cent[c], prev[c])


def test_lloyd_monotone(orc):
    """Textbook Lloyd property: the assignment step and the exact-mean update
    never raise the (weighted) inertia; with bf16-stored centroids the
    trajectory may rise by no more than the rounding term."""
    w = synth.WORKLOADS["tiny"]
    x = synth.chunk_kv(w, 0, 0, synth.KIND_K)[:, 0, :]
    for weights in (None, np.random.default_rng(5).uniform(0.2, 2.0, w.d).astype(np.float32)):
        idx = orc.init_picks(x.shape[0], 16, 0, 0, 0, 0)
        cent = x[idx].copy()
        ids, *_ = orc.assign(x, cent, weights)
        J = orc.inertia(x, cent, ids, weights)
        for _ in range(10):
            new_cent, mean, cnt = orc.update(x, ids, cent)
            J_mean = orc.inertia(x, mean, ids, weights)
            assert J_mean <= J * (1 + 1e-12)
            J_rounded = orc.inertia(x, new_cent, ids, weights)
            ww = np.ones(w.d) if weights is None else weights.astype(np.float64)
            slack = float((cnt[:, None] * ww[None, :] * (new_cent.astype(np.float64) - mean) ** 2).sum())
            assert J_rounded <= J_mean + slack * (1 + 1e-9) + 1e-8 * J_mean  # fp32-held mean leaves a tiny cross term
            new_ids, *_ = orc.assign(x, new_cent, weights)
            J_next = orc.inertia(x, new_cent, new_ids, weights)
            assert J_next <= J_rounded * (1 + 1e-12)
            cent, ids, J = new_cent, new_ids, J_next


def test_c_equals_n_zero_residual(orc):
    """Every token its own centroid: zero residual, all codes 0, X_hat == X."""
    w = synth.WORKLOADS["tiny"]
    x = synth.chunk_kv(w, 1, 0, synth.KIND_V)[:64]
    out = orc.compress_chunk(x, C=64, L=1, bits=2, group=32, iters=3)
    np.testing.assert_array_equal(out["xhat"], x)
    assert np.all(out["scales"] == 0)
    assert np.all(out["codes"] == 0xAA)      # offset-binary code of q = 0
    assert not out["resid"].any()


def test_rtn_is_groupwise_quantiser(orc):
    """C = 0: no centroid; every group of every token quantised directly."""
    x = synth.chunk_kv(synth.WORKLOADS["tiny"], 2, 1, synth.KIND_K)[:32]
    out = orc.compress_chunk(x, C=0, L=1, bits=2, group=32, iters=0)
    for n in range(4):
        for h in range(2):
            for g in range(2):
                s, q, rh = orc.quant_group(x[n, h, 32 * g:32 * g + 32], 2, 0)
                assert out["scales"][0, h, n, g] == s
                np.testing.assert_array_equal(out["xhat"][n, h, 32 * g:32 * g + 32], rh)


def _rel_err(x, xh):
    return float(np.linalg.norm((x - xh).astype(np.float64)) / np.linalg.norm(x.astype(np.float64)))


@pytest.mark.parametrize("bits,stages", [(2, 3), (4, 2)])
def test_stages_reduce_error(orc, bits, stages):
    """Progressive residual quantisation: the reconstruction error does not
    grow with the number of stages, and X_hat is the sum of the per-stage
    dequantised values (rebuilt from the stored layout)."""
    w = synth.WORKLOADS["qvgpro"]
    for kind in (synth.KIND_K, synth.KIND_V):
        for chunk in range(2):
            x = synth.chunk_kv(w, 0, chunk, kind)
            errs = []
            for L in range(1, stages + 1):
                out = orc.compress_chunk(x, C=16, L=L, bits=bits, group=32, iters=10,
                                         seed=7, chunk=chunk)
                rebuilt = orc.decompress(out["codes"], out["scales"], out["ids"], out["cent"],
                                         16, bits, 32)
                np.testing.assert_array_equal(rebuilt, out["xhat"])
                np.testing.assert_allclose(out["resid"], x - out["xhat"], atol=1e-3 * np.abs(x).max())
                errs.append(_rel_err(x, out["xhat"]))
            assert all(b <= a * (1 + 1e-6) for a, b in zip(errs, errs[1:])), errs


def test_smoothing_beats_rtn(orc):
    """Subtracting the k-means centroid before quantising lowers the error
    against plain per-group quantisation, for K and for V."""
    w = synth.WORKLOADS["tiny"]
    for kind in (synth.KIND_K, synth.KIND_V):
        x = synth.chunk_kv(w, 3, 0, kind)
        qvg = orc.compress_chunk(x, C=16, L=1, bits=2, group=32, iters=10)
        rtn = orc.compress_chunk(x, C=0, L=1, bits=2, group=32, iters=0)
        assert _rel_err(x, qvg["xhat"]) < 0.7 * _rel_err(x, rtn["xhat"])


def test_given_centroids_no_iters(orc):
    """With centroids supplied and zero Lloyd iterations the ids are the
    brute-force argmin and the stored centroids are the given ones."""
    w = synth.WORKLOADS["tiny"]
    x = synth.chunk_kv(w, 4, 0, synth.KIND_K)
    rng = np.random.default_rng(6)
    cent_in = synth.bf16_values(rng.standard_normal((1, 2, 16, 64)).astype(np.float32))
    out = orc.compress_chunk(x, C=16, L=1, bits=2, group=32, iters=0, cent_in=cent_in)
    for h in range(2):
        dist = _brute_assign(x[:, h], cent_in[0, h], np.ones(64, np.float32))
        np.testing.assert_array_equal(out["ids"][0, h], dist.argmin(1))
        np.testing.assert_array_equal(orc.bf16_bits_to_f32(out["cent"][0, h]), cent_in[0, h])


def _np_attention(q, k, v, scale):
    logits = (q.astype(np.float64) @ k.T.astype(np.float64)) * scale
    e = np.exp(logits - logits.max(-1, keepdims=True))
    p = e / e.sum(-1, keepdims=True)
    return p @ v.astype(np.float64), np.log(e.sum(-1)) + logits.max(-1)


def test_attention_brute_force(orc):
    rng = np.random.default_rng(7)
    for Nq, Nk, H, Hq in [(3, 5, 1, 1), (8, 8, 2, 4), (1, 1, 1, 1)]:
        d = 16
        q = rng.standard_normal((Nq, Hq, d)).astype(np.float32)
        k = rng.standard_normal((Nk, H, d)).astype(np.float32)
        v = rng.standard_normal((Nk, H, d)).astype(np.float32)
        out, lse, am = orc.attention(q, k, v)
        for hq in range(Hq):
            h = hq // (Hq // H)
            o, l = _np_attention(q[:, hq], k[:, h], v[:, h], 1 / math.sqrt(d))
            np.testing.assert_allclose(out[:, hq], o, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(lse[hq], l, rtol=1e-12)
            np.testing.assert_array_equal(am[hq], (q[:, hq] @ k[:, h].T).argmax(-1))
        if Nk == 1:
            np.testing.assert_allclose(out[:, 0], np.repeat(v[:, 0], Nq, 0))


def test_top1_brute_force_ties_and_gqa(orc):
    """orc_top1 (the oracle side of the top-1 shift rate, QuantWM write-up,
    results: the share of queries whose most-attended history token moves)
    against numpy's argmax of q.k, which returns the first of equal maxima.
    Small-integer operands make every dot product exact, so planted
    duplicate keys give exact ties that must go to the lowest index; query
    heads read KV head hq // (Hq / H) (GQA with Hq = 2H and 4H), and the KV
    heads differ, so a wrong head map fails."""
    rng = np.random.default_rng(11)
    for Nq, Nk, H, Hq in [(7, 9, 2, 4), (5, 13, 1, 4), (6, 6, 3, 3)]:
        d = 8
        q = rng.integers(-3, 4, (Nq, Hq, d)).astype(np.float32)
        k = rng.integers(-3, 4, (Nk, H, d)).astype(np.float32)
        k[Nk - 1] = k[1]          # a duplicate of key 1 (tie goes to 1)
        k[Nk - 2] = k[0]          # and of key 0
        q[0] = 0.0                # all logits 0: the tie goes to slot 0
        am = orc.top1(q, k)
        assert am.shape == (Hq, Nq)
        for hq in range(Hq):
            h = hq // (Hq // H)
            ref = (q[:, hq].astype(np.float64) @ k[:, h].T.astype(np.float64)).argmax(-1)
            np.testing.assert_array_equal(am[hq], ref)
        assert (am[:, 0] == 0).all()
        # top1 agrees with the full attention's argmax (another route)
        _, _, am2 = orc.attention(q, k, k)
        np.testing.assert_array_equal(am, am2)
    # the shift rate: 0 for the same cache; each query whose best key changes counts once
    q = rng.standard_normal((40, 2, 16)).astype(np.float32)
    k = rng.standard_normal((30, 2, 16)).astype(np.float32)
    assert orc.shift_rate(q, k, k) == 0.0
    base = orc.top1(q, k)
    k2 = k.copy()
    k2[base[0, 0], 0] = -k2[base[0, 0], 0]  # the best key of query 0, head 0, flips sign
    moved = (orc.top1(q, k2) != base)
    assert moved[0, 0]
    assert orc.shift_rate(q, k, k2) == pytest.approx(moved.mean())


def test_attention_exact_when_lossless(orc):
    """C = N makes the compressed cache exact, so attention over it equals
    attention over the bf16 cache."""
    w = synth.WORKLOADS["tiny"]
    k = synth.chunk_kv(w, 5, 0, synth.KIND_K)[:48]
    v = synth.chunk_kv(w, 5, 0, synth.KIND_V)[:48]
    q = synth.queries(w, 5, 1)[:16]
    kc = orc.compress_chunk(k, C=48, L=1, bits=2, group=32, iters=2)
    vc = orc.compress_chunk(v, C=48, L=1, bits=2, group=32, iters=2)
    a, _, _ = orc.attention(q, kc["xhat"], vc["xhat"])
    b, _, _ = orc.attention(q, k, v)
    np.testing.assert_array_equal(a, b)


def test_attention_ar_is_the_lse_merge(orc):
    """Attention over [cache; current chunk] equals the two partial
    attentions merged by their log-sum-exps,
    O = (e^{l1} O1 + e^{l2} O2) / (e^{l1} + e^{l2}), lse = log(e^{l1} + e^{l2}):
    a softmax identity, here computed by a different route (two separate
    softmaxes).  An empty cache reduces to plain attention over the chunk."""
    rng = np.random.default_rng(21)
    Nq, Hq, H, d, Nc, Ncur = 6, 4, 2, 16, 9, 5
    q = rng.standard_normal((Nq, Hq, d)).astype(np.float32)
    kh = rng.standard_normal((Nc, H, d)).astype(np.float32)
    vh = rng.standard_normal((Nc, H, d)).astype(np.float32)
    kr = rng.standard_normal((Ncur, H, d)).astype(np.float32)
    vr = rng.standard_normal((Ncur, H, d)).astype(np.float32)
    slots = np.array([0, 1, 2, 3, 128, 129, 130, 256, 257])
    out, lse, top = orc.attention_ar(q, kh, vh, kr, vr, slots, 384)
    o1, l1, a1 = orc.attention(q, kh, vh)
    o2, l2, a2 = orc.attention(q, kr, vr)
    m = np.maximum(l1, l2)
    w1, w2 = np.exp(l1 - m), np.exp(l2 - m)
    ref = (w1.T[:, :, None] * o1 + w2.T[:, :, None] * o2) / (w1 + w2).T[:, :, None]
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, m + np.log(w1 + w2), rtol=1e-12)
    # top-1: the larger of the two partial maxima, numbered by slot
    for hq in range(Hq):
        h = hq // (Hq // H)
        s1 = (q[:, hq].astype(np.float64) @ kh[:, h].T.astype(np.float64)).max(-1)
        s2 = (q[:, hq].astype(np.float64) @ kr[:, h].T.astype(np.float64)).max(-1)
        want = np.where(s2 > s1, 384 + a2[hq], slots[a1[hq]])
        np.testing.assert_array_equal(top[hq], want)
    # first chunk: no cache
    o0, l0, t0 = orc.attention_ar(q, kh[:0], vh[:0], kr, vr, slots[:0], 0)
    np.testing.assert_array_equal(o0, o2)
    np.testing.assert_array_equal(t0, a2)


def test_query_stats(orc):
    rng = np.random.default_rng(8)
    q = rng.standard_normal((30, 4, 8)).astype(np.float32)
    M, cnt = orc.query_stats(q, H=2)
    assert cnt == 60
    for h in range(2):
        qs = q[:, 2 * h:2 * h + 2].reshape(-1, 8).astype(np.float64)
        np.testing.assert_allclose(M[h], qs.T @ qs, rtol=1e-12)
    M2, cnt2 = orc.query_stats(q, H=2, M=M, count=cnt)
    np.testing.assert_allclose(M2, 2 * M, rtol=1e-12)
    assert cnt2 == 120


def test_jacobi_planted_and_library(orc):
    """Exact planted spectrum (closed form) and agreement with LAPACK."""
    w = synth.WORKLOADS["quantwm"]
    U = synth.planted_basis(w, 0)[0]
    lam, s2 = synth.planted_spectrum(w.d)
    M = (U * lam) @ U.T + s2 * np.eye(w.d)
    ev, vec, sweeps = orc.jacobi(M)
    assert sweeps < 100
    np.testing.assert_allclose(ev[:8], lam + s2, rtol=1e-10)
    np.testing.assert_allclose(ev[8:], s2, rtol=1e-10)
    # subspace of the top 8 equals the planted one
    proj = vec[:, :8].T @ U
    sv = np.linalg.svd(proj, compute_uv=False)
    assert np.all(np.arccos(np.clip(sv, -1, 1)) < 1e-6)
    np.testing.assert_allclose(vec.T @ vec, np.eye(w.d), atol=1e-10)
    # energy fraction closed form: (0.7 d + 8 s2) / d
    Ub, eig, frac = orc.psac_basis(M[None] * 10.0, 10, 8)
    assert abs(frac[0] - (0.7 * w.d + 8 * s2) / w.d) < 1e-10
    rng = np.random.default_rng(9)
    A = rng.standard_normal((24, 24))
    A = A + A.T
    ev, vec, _ = orc.jacobi(A)
    ref = np.linalg.eigvalsh(A)[::-1]
    np.testing.assert_allclose(ev, ref, atol=1e-10)
    np.testing.assert_allclose(A @ vec, vec * ev[None, :], atol=1e-9)
    big = np.abs(vec).argmax(0)
    assert np.all(vec[big, np.arange(24)] > 0)


def test_psac_basis_from_queries(orc):
    """On planted history queries the top-8 eigenvectors recover the planted
    directions and hold about 71.9% of the energy (the page: >71%)."""
    w = synth.WORKLOADS["quantwm"]
    q = synth.history_queries(w, 0)[:, :2]
    M, cnt = orc.query_stats(q, H=2)
    U, eig, frac = orc.psac_basis(M, cnt, 8)
    Up = synth.planted_basis(w, 0)
    for h in range(2):
        np.testing.assert_allclose(U[h].T @ U[h], np.eye(8), atol=1e-10)
        Mn = M[h] / cnt
        np.testing.assert_allclose(np.einsum("dk,de,ek->k", U[h], Mn, U[h]), eig[h], rtol=1e-9)
        np.testing.assert_allclose(frac[h], eig[h].sum() / np.trace(Mn), rtol=1e-12)
        assert 0.69 < frac[h] < 0.75
        sv = np.linalg.svd(U[h].T @ Up[h], compute_uv=False)
        assert sv.min() > 0.95


def test_psac_encode(orc):
    """INT8 projection codes: |P - S'q| <= S'/2, and decoding adds P_hat U^T,
    which removes the part of the key error inside span(U)."""
    rng = np.random.default_rng(10)
    d, r = 64, 8
    U, _ = np.linalg.qr(rng.standard_normal((d, r)))
    U = U.astype(np.float32)
    for _ in range(50):
        E = (rng.standard_normal(d) * rng.uniform(0.01, 10)).astype(np.float32)
        p, s = orc.psac_encode_token(E, U)
        Sp = float(orc.f16_bits_to_f32(s))
        P = E.astype(np.float64) @ U.astype(np.float64)
        assert np.all(np.abs(P - Sp * p) <= Sp / 2 * (1 + 1e-5) + 1e-6 * np.abs(P).max())
        corrected = E - (Sp * p.astype(np.float32)) @ U.T
        inside = np.linalg.norm(corrected.astype(np.float64) @ U)
        assert inside <= np.sqrt(r) * Sp / 2 * 1.01 + 1e-6
    # compress with PSAC: the stored codes are those of the final residual
    w = synth.WORKLOADS["tiny"]
    x = synth.chunk_kv(w, 6, 0, synth.KIND_K)[:64]
    Ub = np.stack([U, U]).astype(np.float32)
    out = orc.compress_chunk(x, C=16, L=1, bits=2, group=32, iters=3, psac_U=Ub)
    for n in (0, 17, 63):
        p, s = orc.psac_encode_token(out["resid"][n, 1], Ub[1])
        np.testing.assert_array_equal(out["psac_p"][1, n], p)
        assert out["psac_s"][1, n] == s
    rebuilt = orc.decompress(out["codes"], out["scales"], out["ids"], out["cent"], 16, 2, 32,
                             psac_p=out["psac_p"], psac_s=out["psac_s"], psac_U=Ub)
    e0 = np.linalg.norm((x - out["xhat"]).astype(np.float64) @ U)
    e1 = np.linalg.norm((x - rebuilt).astype(np.float64) @ U)
    assert e1 < 0.1 * e0


# ---------------------------------------------------------------- outlier split

def test_outlier_split_hand_example(orc):
    """G = 8, INT2 (q in [-2, 1], S = amax / 1).  |r| sorted is
    [0, .25, .5, .5, .75, 1, 1, 12]; the 99th percentile sits at position
    0.99 * 7 = 6.93, T = 1 + 0.93 * (12 - 1) = 11.23, so only 12.0 (channel
    3) is split off.  The remaining amax is 1, S = 1, and round-half-even
    gives codes [0, -1, 0, 0, -1, 0, 1, 0]; 12.0 is kept as fp16 0x4A00."""
    r = np.array([0.5, -1.0, 0.25, 12.0, -0.75, 0.0, 1.0, -0.5], np.float32)
    s, q, rh, ov, oi = orc.quant_group_outlier(r, bits=2)
    assert s == 0x3C00 and oi == 3 and ov == 0x4A00
    np.testing.assert_array_equal(q, [0, -1, 0, 0, -1, 0, 1, 0])
    np.testing.assert_array_equal(rh, [0, -1, 0, 12.0, -1, 0, 1, 0])
    # without the split the outlier sets the step: S = 12, every small value -> 0
    s0, q0, _ = orc.quant_group(r, bits=2)
    assert s0 == 0x4A00 and np.count_nonzero(q0) == 1


@pytest.mark.parametrize("G", [8, 16, 32, 64])
def test_outlier_split_is_the_p99_exceedance(orc, G):
    """The split-off channel is exactly the set {j : |r_j| > P99(|r|)} of
    numpy's percentile (linear interpolation), on random groups with and
    without a planted outlier and with ties at the top (no split)."""
    rng = np.random.default_rng(40 + G)
    for t in range(300):
        r = rng.standard_normal(G).astype(np.float32)
        if t % 3 == 0:
            r[rng.integers(G)] *= 50.0
        if t % 7 == 0:  # a tie for the largest magnitude: nothing is split off
            i, j = rng.choice(G, 2, replace=False)
            r[i] = np.float32(2 * np.abs(r).max())
            r[j] = -r[i]
        a = np.abs(r.astype(np.float64))
        want = np.nonzero(a > np.percentile(a, 99))[0]
        s, q, rh, ov, oi = orc.quant_group_outlier(r, bits=2)
        assert len(want) <= 1
        if t % 7 == 0:
            assert len(want) == 0
        if len(want):
            assert oi == want[0]
            assert rh[oi] == orc.f16_bits_to_f32(np.array([ov], np.uint16))[0]
            assert abs(rh[oi] - r[oi]) <= 2 ** -11 * abs(r[oi])
            rest = np.delete(r, oi)
        else:
            assert oi == 0xFF and ov == 0
            rest = r
        # the scale is the plain quantiser's on the remaining values
        S = orc.f16_bits_to_f32(np.array([s], np.uint16))[0]
        assert S == orc.f16_bits_to_f32(np.array([orc.quant_group(rest, bits=2)[0]], np.uint16))[0]
        keep = np.arange(G) != (oi if oi != 0xFF else -1)
        # unclipped kept values are within half a step
        inside = keep & (np.abs(r) <= S)
        assert np.all(np.abs(r[inside] - rh[inside]) <= S / 2)


def test_outlier_split_refuses_large_groups(orc):
    with pytest.raises(ValueError):
        orc.quant_group_outlier(np.ones(128, np.float32))


def test_outlier_split_lowers_error_and_rebuilds(orc):
    """On synthetic K and V with token-varying outlier channels (x50 K,
    x300 V) the split lowers the reconstruction error of QVG and of RTN; the
    stored layout (codes, scales, side list) rebuilds X_hat exactly; at most
    one value per group is split off."""
    w = synth.WORKLOADS["tiny"]
    for kind in (synth.KIND_K, synth.KIND_V):
        x = synth.chunk_kv(w, 11, 0, kind)
        for C in (16, 0):
            base = orc.compress_chunk(x, C=C, L=1, bits=2, group=32, iters=10 if C else 0)
            out = orc.compress_chunk(x, C=C, L=1, bits=2, group=32, iters=10 if C else 0, outlier=True)
            np.testing.assert_array_equal(out["ids"], base["ids"])  # clustering is unchanged
            assert _rel_err(x, out["xhat"]) < _rel_err(x, base["xhat"])
            rebuilt = orc.decompress(out["codes"], out["scales"], out["ids"], out["cent"], C, 2, 32,
                                     outl_val=out["outl_val"], outl_idx=out["outl_idx"])
            np.testing.assert_array_equal(rebuilt, out["xhat"])
            oi = out["outl_idx"]
            assert np.all((oi < 32) | (oi == 0xFF))
            assert np.all(out["outl_val"][oi == 0xFF] == 0)
    # two stages: the second stage splits its own residual's outliers
    x = synth.chunk_kv(w, 11, 1, synth.KIND_V)
    one = orc.compress_chunk(x, C=16, L=1, bits=2, group=32, iters=10, outlier=True)
    two = orc.compress_chunk(x, C=16, L=2, bits=2, group=32, iters=10, outlier=True)
    rebuilt = orc.decompress(two["codes"], two["scales"], two["ids"], two["cent"], 16, 2, 32,
                             outl_val=two["outl_val"], outl_idx=two["outl_idx"])
    np.testing.assert_array_equal(rebuilt, two["xhat"])
    assert _rel_err(x, two["xhat"]) <= _rel_err(x, one["xhat"])
