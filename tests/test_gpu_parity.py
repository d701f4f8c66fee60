"""GPU-vs-oracle parity through the C ABI, on the seeded synthetic workloads.

Bars (the arithmetic behind them is in the helpers and below):
  - cluster ids: equal to the oracle's fp64 argmin over the same centroids,
    except near ties (relative score gap < 1e-5), which must stay < 0.01 %;
  - codes and fp16 scales: bit-exact wherever the ids agree (the quantiser is
    a chain of correctly rounded fp32 operations on both sides);
  - k-means initialisation: bit-exact centroids;
  - one Lloyd update from the same assignment: every bf16 centroid within
    1 ulp of the oracle's (fp32 vs fp64 sums round differently);
  - reconstruction from the same bytes: bit-exact (same fp32 operation
    order), PSAC correction within 1e-3 of max|X|;
  - attention: max|dO| / max|O_oracle| <= 2e-3 per head, oracle in fp64 on
    the reconstruction of the same compressed cache.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import video_diffusion_kv_gb300 as qvg
from video_diffusion_kv_gb300 import synth

from _helpers import (ATTN_TOL, NEAR_TIE_RATE, assignment_mismatches, bf16_ulp_diff,
                      chunk_arrays, chunk_slice, host_cache, lse_tolerance, oracle_rebuild, stage_abs_rebuild,
                      to_dev)

pytestmark = pytest.mark.gpu
NT = 16  # oracle threads


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


W = synth.WORKLOADS
# 2 heads of d = 128, chunks of one 16 x 20 frame (320 tokens: two and a half tiles)
W128 = synth.Workload("d128_small", H=2, d=128, frame_hw=(16, 20), frames_per_chunk=1, n_chunks=2, dist="ar1",
                      C=16, L=2, bits=2, group=128, iters=6, Hq=2, Nq=320)
CASES = {
    "tiny": (W["tiny"], qvg.Params(C=16, L=1, bits=2, group=32, iters=10, seed=3), 4),
    "pro_int2_L3": (W["qvgpro"], qvg.Params(C=16, L=3, bits=2, group=32, iters=10, seed=4), 2),
    "pro_int4_L2": (W["qvgpro"], qvg.Params(C=16, L=2, bits=4, group=32, iters=10, seed=5), 2),
    "page1_scale": (W["tiny"], qvg.Params(C=16, L=1, bits=2, group=32, iters=10, scale_mode=1, seed=6), 2),
    "rtn": (W["tiny"], qvg.Params(C=0, L=1, bits=2, group=32, iters=0), 2),
    "longcat": (W["longcat"], qvg.Params(C=256, L=1, bits=2, group=64, iters=8, seed=7), 2),
    # outlier split (fp16 side list of each group's value above its P99)
    "tiny_outlier": (W["tiny"], qvg.Params(C=16, L=1, bits=2, group=32, iters=10, seed=24, flags=qvg.QVG_OUTLIER), 2),
    "pro_outlier_L2": (W["qvgpro"], qvg.Params(C=16, L=2, bits=2, group=32, iters=10, seed=25, flags=qvg.QVG_OUTLIER), 2),
    "rtn_outlier_g8": (W["tiny"], qvg.Params(C=0, L=1, bits=4, group=8, iters=0, flags=qvg.QVG_OUTLIER), 2),
    "tiny_outlier_g16": (W["tiny"], qvg.Params(C=16, L=1, bits=2, group=16, iters=10, seed=27, flags=qvg.QVG_OUTLIER), 2),
    "longcat_outlier": (W["longcat"], qvg.Params(C=256, L=1, bits=2, group=64, iters=8, seed=26, flags=qvg.QVG_OUTLIER), 2),
    # groups wider than the 32 channels one lane of the quantiser holds: the
    # group statistics are combined across 2 (d = 64, G = 64) or 4 (d = 128,
    # G = 128) lanes of a row, with and without the outlier split
    "tiny_g64_int4": (W["tiny"], qvg.Params(C=16, L=1, bits=4, group=64, iters=10, seed=28), 2),
    "tiny_outlier_g64_L2": (W["tiny"], qvg.Params(C=16, L=2, bits=2, group=64, iters=10, seed=29,
                                                  flags=qvg.QVG_OUTLIER), 2),
    "d128_g128_L2": (W128, qvg.Params(C=16, L=2, bits=2, group=128, iters=6, seed=30), 2),
}
OUTL = lambda p: bool(p.flags & qvg.QVG_OUTLIER)


def _new_cache(w, p, n_chunks, N=None):
    N = N or w.N
    cap = n_chunks * (-(-N // 128) * 128)
    return qvg.CompressedKV(p, w.H, w.d, cap, n_chunks)


def _check_against_fed_oracle(x, hc, p, k, w=None, psac_U=None):
    """The oracle, fed the GPU's stored centroids with zero Lloyd iterations,
    must reproduce the GPU's ids (modulo near ties) and, on rows whose ids
    agree at every stage, its codes and scales bit for bit."""
    codes, scales, ids, cent = chunk_arrays(hc, p, k)
    cent_in = oracle.bf16_bits_to_f32(cent) if p.C > 0 else None
    o = oracle.compress_chunk(x, C=p.C, L=p.L, bits=p.bits, group=p.group, iters=0, mode=p.scale_mode,
                              seed=p.seed, chunk=k, qsac_w=w, psac_U=psac_U, cent_in=cent_in, outlier=OUTL(p),
                              nthreads=NT)
    N, H = x.shape[0], x.shape[1]
    ok_rows = np.ones((H, N), bool)
    total = near = 0
    stage_in = x.copy()
    for l in range(p.L):
        g = stage_in if l == 0 else synth.bf16_values(stage_in)
        if p.C > 0:
            for h in range(H):
                wh = None if w is None else w[h]
                rows = ok_rows[h]
                m, far = assignment_mismatches(g[rows, h], cent[l, h, :min(p.C, N)],
                                               ids[l, h][rows].astype(np.int32), wh)
                total += int(rows.sum())
                near += m
                assert far == 0, ("assignment mismatch outside near ties", l, h, far)
                ok_rows[h] &= ids[l, h] == o["ids"][l, h]
        sl = chunk_slice(hc, k)
        for h in range(H):
            np.testing.assert_array_equal(codes[l, h][ok_rows[h]], o["codes"][l, h][ok_rows[h]])
            np.testing.assert_array_equal(scales[l, h][ok_rows[h]], o["scales"][l, h][ok_rows[h]])
            if OUTL(p):
                np.testing.assert_array_equal(hc["outl_idx"][l, h, sl][ok_rows[h]], o["outl_idx"][l, h][ok_rows[h]])
                np.testing.assert_array_equal(hc["outl_val"][l, h, sl][ok_rows[h]], o["outl_val"][l, h][ok_rows[h]])
        # next stage input from the oracle's own residual (bit-exact on ok rows)
        kw = dict(outl_val=o["outl_val"][l:l + 1], outl_idx=o["outl_idx"][l:l + 1]) if OUTL(p) else {}
        dq = oracle.decompress(o["codes"][l:l + 1], o["scales"][l:l + 1], o["ids"][l:l + 1],
                               o["cent"][l:l + 1], p.C, p.bits, p.group, **kw)
        stage_in = stage_in - dq
    if total:
        assert near <= max(1, NEAR_TIE_RATE * total), ("near ties", near, total)
    return o, ok_rows


@pytest.mark.parametrize("name", list(CASES))
def test_compress_matches_oracle(name):
    """Full seeded compression on the GPU, checked chunk by chunk: the final
    assignment and quantisation agree with the oracle run on the GPU's own
    centroids, and the reconstruction error is that of the oracle's own
    k-means (same definition, same seeds)."""
    w, p, n_chunks = CASES[name]
    kc = _new_cache(w, p, n_chunks)
    xs = []
    for k in range(n_chunks):
        x = synth.chunk_kv(w, 11, k, synth.KIND_K if k % 2 == 0 else synth.KIND_V)
        xs.append(x)
        qvg.compress_chunk(p, to_dev(x), kc)
    assert qvg.get_status() == qvg.QVG_OK
    hc = host_cache(kc)
    for k in range(n_chunks):
        assert hc["length"][k] == w.N and hc["start"][k] % 128 == 0
        _check_against_fed_oracle(xs[k], hc, p, k)
    if w.N <= 256:
        # the oracle's own full run reaches the same reconstruction error
        for k in range(n_chunks):
            o = oracle.compress_chunk(xs[k], C=p.C, L=p.L, bits=p.bits, group=p.group, iters=p.iters,
                                      mode=p.scale_mode, seed=p.seed, chunk=k, outlier=OUTL(p), nthreads=NT)
            rg = np.linalg.norm(xs[k] - oracle_rebuild(hc, p, k)) / np.linalg.norm(xs[k])
            ro = np.linalg.norm(xs[k] - o["xhat"]) / np.linalg.norm(xs[k])
            assert abs(rg - ro) <= 0.05 * ro + 1e-6, (rg, ro)


@pytest.mark.parametrize("name", ["longcat", "pro_int2_L3", "pro_outlier_L2"])
def test_compress_is_deterministic(name):
    """The same chunks compressed three times leave byte-identical caches:
    every reduction runs in a fixed order, and no kernel reads what the
    launch before it writes until it has waited for that launch."""
    w, p, n_chunks = CASES[name]
    xs = [synth.chunk_kv(w, 34, k, synth.KIND_K) for k in range(n_chunks)]
    runs = []
    for _ in range(3):
        c = _new_cache(w, p, n_chunks)
        for x in xs:
            qvg.compress_chunk(p, to_dev(x), c)
        runs.append(host_cache(c))
    assert qvg.get_status() == qvg.QVG_OK
    for other in runs[1:]:
        for name_ in runs[0]:
            np.testing.assert_array_equal(other[name_], runs[0][name_], err_msg=name_)


@pytest.mark.parametrize("name", ["tiny", "pro_int2_L3", "longcat"])
def test_kmeans_init_exact(name):
    """Zero Lloyd iterations: the centroids are the seeded picks, bit for bit."""
    w, p0, _ = CASES[name]
    p = qvg.Params(**{**p0.__dict__, "iters": 0})
    kc = _new_cache(w, p, 1)
    x = synth.chunk_kv(w, 12, 0, synth.KIND_K)
    qvg.compress_chunk(p, to_dev(x), kc)
    hc = host_cache(kc)
    o = oracle.compress_chunk(x, C=p.C, L=p.L, bits=p.bits, group=p.group, iters=0, seed=p.seed, chunk=0,
                              nthreads=NT)
    np.testing.assert_array_equal(hc["cent"][0, :, 0], o["cent"][0])
    _check_against_fed_oracle(x, hc, p, 0)


@pytest.mark.parametrize("name", ["tiny", "longcat"])
def test_lloyd_update_step(name):
    """From the same centroids c0: GPU ids after one assignment, then the
    GPU's updated centroids equal the oracle's mean of those members within
    one bf16 ulp (empty clusters keep c0)."""
    w, p0, _ = CASES[name]
    x = synth.chunk_kv(w, 13, 0, synth.KIND_K)
    rng = np.random.default_rng(0)
    N = x.shape[0]
    c0 = np.stack([x[rng.choice(N, p0.C, replace=False), h] for h in range(w.H)])  # [H, C, d]
    c0_bits = torch.from_numpy(c0).to(torch.bfloat16).view(torch.int16)
    res = {}
    for iters in (0, 1):
        p = qvg.Params(C=p0.C, L=1, bits=p0.bits, group=p0.group, iters=iters, flags=qvg.QVG_GIVEN_CENTROIDS)
        kc = _new_cache(w, p, 1)
        kc.view("cent", torch.int16, (1, w.H, 1, p.C, w.d))[0, :, 0] = c0_bits.cuda()
        qvg.compress_chunk(p, to_dev(x), kc)
        res[iters] = host_cache(kc)
    ids0 = res[0]["ids"][0, :, :N].astype(np.int32)
    c1 = res[1]["cent"][0, :, 0]
    exact = 0
    for h in range(w.H):
        m, far = assignment_mismatches(x[:, h], c0_bits.numpy().view(np.uint16)[h], ids0[h])
        assert far == 0
        ref, mean, cnt = oracle.update(x[:, h], ids0[h], c0[h])
        ref_bits = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        ulps = bf16_ulp_diff(c1[h], ref_bits)
        assert ulps.max() <= 1, (h, ulps.max())
        exact += (ulps == 0).sum()
    assert exact >= 0.99 * w.H * p0.C * w.d


@pytest.mark.parametrize("name", ["pro_int2_L3", "pro_outlier_L2", "rtn_outlier_g8", "tiny_outlier_g64_L2",
                                  "d128_g128_L2"])
def test_decompress_exact_and_bf16(name):
    w, p, n_chunks = CASES[name]
    kc = _new_cache(w, p, n_chunks)
    for k in range(n_chunks):
        qvg.compress_chunk(p, to_dev(synth.chunk_kv(w, 14, k, synth.KIND_V)), kc)
    hc = host_cache(kc)
    full = qvg.decompress(p, kc, 0, kc.n_tokens).cpu().numpy()
    half = qvg.decompress(p, kc, 0, kc.n_tokens, out_dtype=qvg.QVG_OUT_BF16).float().cpu().numpy()
    for k in range(n_chunks):
        sl = chunk_slice(hc, k)
        ref = oracle_rebuild(hc, p, k)
        np.testing.assert_array_equal(full[sl], ref)
        np.testing.assert_array_equal(half[sl], synth.bf16_values(ref))


@pytest.mark.parametrize("name", ["tiny", "pro_outlier_L2", "longcat"])
def test_decompress_ragged_range(name):
    """A slot range that starts off a warp boundary and ends in a ragged
    tail (not a multiple of 32) gives the same values as the whole-cache
    rebuild, in fp32 and bf16, and writes nothing past its last row."""
    import torch
    w, p, n_chunks = CASES[name]
    kc = _new_cache(w, p, n_chunks)
    for k in range(n_chunks):
        qvg.compress_chunk(p, to_dev(synth.chunk_kv(w, 15, k, synth.KIND_K)), kc)
    full = qvg.decompress(p, kc, 0, kc.n_tokens)
    for tok0, ntok in ((37, kc.n_tokens - 37 - 19), (5, 1), (kc.n_tokens - 45, 45)):
        for dt, tdt in ((qvg.QVG_OUT_F32, torch.float32), (qvg.QVG_OUT_BF16, torch.bfloat16)):
            guard = 40
            big = torch.full((ntok + guard, w.H, w.d), 7.0, dtype=tdt, device="cuda")
            qvg.decompress(p, kc, tok0, ntok, out_dtype=dt, out=big[:ntok])
            want = full[tok0:tok0 + ntok].to(tdt)
            assert torch.equal(big[:ntok], want), (tok0, ntok, dt)
            assert bool((big[ntok:] == 7.0).all()), (tok0, ntok, dt)
    # an output that is 4-byte but not vector aligned (one fp32 / two bf16
    # elements past a 16-byte boundary) takes the 32-bit store path
    tok0, ntok = 37, kc.n_tokens - 37 - 19
    for dt, tdt, skip in ((qvg.QVG_OUT_F32, torch.float32, 1), (qvg.QVG_OUT_BF16, torch.bfloat16, 2)):
        n = ntok * w.H * w.d
        flat = torch.full((n + skip + 64,), 7.0, dtype=tdt, device="cuda")
        view = flat[skip:skip + n].view(ntok, w.H, w.d)
        assert view.data_ptr() % 16 != 0
        qvg.decompress(p, kc, tok0, ntok, out_dtype=dt, out=view)
        assert torch.equal(view, full[tok0:tok0 + ntok].to(tdt)), dt
        assert bool((flat[:skip] == 7.0).all()) and bool((flat[skip + n:] == 7.0).all()), dt


def _cache_with_chunks(w, p, chunks_kv, seed=0):
    n = len(chunks_kv)
    cap = sum(-(-c[0].shape[0] // 128) * 128 for c in chunks_kv)
    kc = qvg.CompressedKV(p, w.H, w.d, cap, n)
    vc = qvg.CompressedKV(p, w.H, w.d, cap, n)
    for k, v in chunks_kv:
        qvg.compress_chunk(p, to_dev(k), kc)
        qvg.compress_chunk(p, to_dev(v), vc)
    return kc, vc


def _oracle_attention_on(kc, vc, p, q, rows=None):
    hk, hv = host_cache(kc), host_cache(vc)
    kh = np.concatenate([oracle_rebuild(hk, p, k) for k in range(kc.n_chunks)], 0)
    vh = np.concatenate([oracle_rebuild(hv, p, k) for k in range(vc.n_chunks)], 0)
    qq = q if rows is None else q[rows]
    out, lse, am = oracle.attention(qq, kh, vh, nthreads=NT)
    return out, lse, am, kh, hk


def _slot_of_token(hk, n_chunks):
    return np.concatenate([np.arange(hk["start"][k], hk["start"][k] + hk["length"][k]) for k in range(n_chunks)])


def _assert_top1(top1, q, kh, slots, ram, min_agree=0.95):
    """Top-1 slots: equal to the oracle's argmax except at near ties, where
    the GPU's pick must be within the fp16 rounding of the logits of the
    best: q and k_hat enter the tensor core as fp16 (relative rounding
    2^-11 each), so a logit moves by at most ~2^-10 sum_j |q_j k_j|; the
    bound allows 2^-9."""
    Nq, Hq, d = q.shape
    H = kh.shape[1]
    tok_of = {int(s): i for i, s in enumerate(slots)}
    agree = (top1 == slots[ram])
    assert agree.mean() >= min_agree, agree.mean()
    for hq, i in zip(*np.nonzero(~agree)):
        h = hq // (Hq // H)
        t_gpu = tok_of[int(top1[hq, i])]
        t_ref = int(ram[hq, i])
        qq = q[i, hq].astype(np.float64)
        s_gpu = qq @ kh[t_gpu, h].astype(np.float64)
        s_ref = qq @ kh[t_ref, h].astype(np.float64)
        mag = np.abs(qq) @ np.maximum(np.abs(kh[t_gpu, h]), np.abs(kh[t_ref, h])).astype(np.float64)
        assert s_ref - s_gpu <= 2 ** -9 * mag, (hq, i, s_ref - s_gpu, mag)


def _assert_attention(got, ref, Hq):
    for h in range(Hq):
        err = np.abs(got[:, h] - ref[:, h]).max() / np.abs(ref[:, h]).max()
        assert err <= ATTN_TOL, (h, err)


@pytest.mark.parametrize("Hq_mult", [1, 2])
def test_attention_tiny(Hq_mult):
    w, p, n_chunks = CASES["tiny"]
    chunks = [(synth.chunk_kv(w, 15, k, synth.KIND_K), synth.chunk_kv(w, 15, k, synth.KIND_V)) for k in range(n_chunks)]
    kc, vc = _cache_with_chunks(w, p, chunks)
    q = synth.queries(w, 15, n_chunks)
    if Hq_mult > 1:
        q = np.concatenate([q, synth.queries(w, 16, n_chunks)], 1)[:, [0, 2, 1, 3]]
    out, lse, top1 = qvg.attention(p, to_dev(q), kc, vc, want_lse=True, want_top1=True)
    ref, rlse, ram, _, hk = _oracle_attention_on(kc, vc, p, q)
    got = out.cpu().numpy().astype(np.float64)
    _assert_attention(got, ref, q.shape[1])
    np.testing.assert_allclose(lse.cpu().numpy(), rlse, atol=2e-3, rtol=0)
    slots = _slot_of_token(hk, n_chunks)
    agree = (top1.cpu().numpy() == slots[ram]).mean()
    assert agree >= 0.99
    # bf16 output is the rounding of the fp32 one (up to the last bit)
    o16, _, _ = qvg.attention(p, to_dev(q), kc, vc, out_dtype=qvg.QVG_OUT_BF16)
    np.testing.assert_allclose(o16.float().cpu().numpy(), got, rtol=2 ** -7, atol=1e-6 * np.abs(got).max())


def test_attention_longcat_sampled():
    """4680 queries over 2 chunks of 4680 tokens (16 heads, d=128); the fp64
    oracle checks 64 sampled query rows per head."""
    w, p, _ = CASES["longcat"]
    chunks = [(synth.chunk_kv(w, 17, k, synth.KIND_K), synth.chunk_kv(w, 17, k, synth.KIND_V)) for k in range(2)]
    kc, vc = _cache_with_chunks(w, p, chunks)
    q = synth.queries(w, 17, 2)
    out, _, _ = qvg.attention(p, to_dev(q), kc, vc)
    rows = np.random.default_rng(1).choice(q.shape[0], 64, replace=False)
    ref, _, _, _, _ = _oracle_attention_on(kc, vc, p, q, rows)
    _assert_attention(out.cpu().numpy()[rows].astype(np.float64), ref, w.Hq)


@pytest.mark.parametrize("Nq", [16, 300])
def test_attention_split_cache(Nq):
    """Few queries (16: one block, 300: two blocks, x 16 heads) over 2 LongCat
    chunks: qvg_attention splits the cache over extra CTAs and merges the
    splits' partial outputs by their log-sum-exp.  Checked against the fp64
    oracle (output, lse, top-1) and against the same call without a
    workspace, which runs unsplit."""
    w, p, _ = CASES["longcat"]
    chunks = [(synth.chunk_kv(w, 23, k, synth.KIND_K), synth.chunk_kv(w, 23, k, synth.KIND_V)) for k in range(2)]
    kc, vc = _cache_with_chunks(w, p, chunks)
    q = np.ascontiguousarray(synth.queries(w, 23, 2)[:Nq])
    need = qvg.workspace_size(p, qvg.QVG_OP_ATTENTION, Nq, w.H, w.d, w.Hq)
    assert need > 0
    out, lse, top1 = qvg.attention(p, to_dev(q), kc, vc, want_lse=True, want_top1=True)
    ref, rlse, ram, _, hk = _oracle_attention_on(kc, vc, p, q)
    got = out.cpu().numpy().astype(np.float64)
    _assert_attention(got, ref, w.Hq)
    np.testing.assert_allclose(lse.cpu().numpy(), rlse, atol=2e-3, rtol=0)
    # top-1 against fp64: LongCat-like patches hold near-duplicate keys, whose
    # maxima fp16 operand rounding can reorder
    slots = _slot_of_token(hk, 2)
    assert (top1.cpu().numpy() == slots[ram]).mean() >= 0.95
    # the unsplit path (no workspace) on the same inputs: same logits, so the
    # same top-1; the outputs and lse differ only by the rounding of P and of
    # the merge (each split normalises by its own running max)
    import ctypes as ct
    qd = to_dev(q)
    one = torch.empty_like(out)
    lse1 = torch.empty_like(lse)
    top11 = torch.empty_like(top1)
    k, v, pc = kc.c(), vc.c(), p.c()
    st = qvg.lib().qvg_attention(ct.byref(pc), ct.c_void_p(qd.data_ptr()), Nq, w.Hq, ct.byref(k), ct.byref(v),
                                 ct.c_float(0.0), ct.c_void_p(one.data_ptr()), qvg.QVG_OUT_F32,
                                 ct.c_void_p(lse1.data_ptr()), ct.c_void_p(top11.data_ptr()), None, 0, None)
    assert st == qvg.QVG_OK
    one_np = one.cpu().numpy().astype(np.float64)
    assert np.abs(one_np - got).max() <= 1e-4 * np.abs(one_np).max()
    np.testing.assert_allclose(lse1.cpu().numpy(), lse.cpu().numpy(), atol=1e-3, rtol=0)
    assert (top11.cpu().numpy() == top1.cpu().numpy()).mean() >= 0.999


FEW_Q = {
    "tiny": CASES["tiny"][:2],
    "longcat": CASES["longcat"][:2],
    # d = 128 with 8-channel groups: each 64-channel half of a slot carries
    # eight scales
    "d128_int2_g8": (W128, qvg.Params(C=16, L=1, bits=2, group=8, iters=6, seed=31)),
    "d128_int4_g8": (W128, qvg.Params(C=16, L=1, bits=4, group=8, iters=6, seed=32)),
}


@pytest.mark.parametrize("name,n_chunks,Nq,Hq_mult", [("tiny", 5, 5, 1), ("tiny", 5, 40, 2), ("longcat", 2, 16, 1),
                                                      ("longcat", 2, 100, 1), ("d128_int2_g8", 2, 24, 1),
                                                      ("d128_int4_g8", 2, 128, 1)])
def test_attention_few_queries(name, n_chunks, Nq, Hq_mult):
    """At most 128 queries over a one-stage cache without top-1 output.
    Split cache: tiny (d = 64) 10 tiles in two CTAs of 5 per head, the
    LongCat-like layer (d = 128) 74 tiles in nine CTAs of 8 or 9; unsplit:
    d = 128 with 8-channel groups in INT2 and INT4, 6 tiles per head.  With
    GQA and ragged query counts, checked against the fp64 oracle (the
    log-sum-exp within the bound of the fp16 rounding of K_hat) and against
    the call without a workspace."""
    w, p = FEW_Q[name]
    chunks = [(synth.chunk_kv(w, 41, k, synth.KIND_K), synth.chunk_kv(w, 41, k, synth.KIND_V)) for k in range(n_chunks)]
    kc, vc = _cache_with_chunks(w, p, chunks)
    q = synth.queries(w, 41, n_chunks)
    if Hq_mult > 1:  # two query heads per KV head
        q = np.concatenate([q, synth.queries(w, 42, n_chunks)], 1)[:, [0, 2, 1, 3]]
    q = np.ascontiguousarray(q[:Nq])
    Hq = q.shape[1]
    assert qvg.workspace_size(p, qvg.QVG_OP_ATTENTION, Nq, w.H, w.d, Hq) > 0
    out, lse, _ = qvg.attention(p, to_dev(q), kc, vc, want_lse=True)
    ref, rlse, _, _, hk = _oracle_attention_on(kc, vc, p, q)
    got = out.cpu().numpy().astype(np.float64)
    _assert_attention(got, ref, Hq)
    # the log-sum-exp within the bound of the fp16 rounding of K_hat
    k_abs = np.concatenate([stage_abs_rebuild(hk, p, k) for k in range(kc.n_chunks)], 0)
    tol = lse_tolerance(q, k_abs, Hq // w.H)
    assert (np.abs(lse.cpu().numpy() - rlse) <= tol).all(), np.abs(lse.cpu().numpy() - rlse).max()
    one, lse1, _ = qvg.attention(p, to_dev(q), kc, vc, want_lse=True, allow_split=False)
    one_np = one.cpu().numpy().astype(np.float64)
    assert np.abs(one_np - got).max() <= 1e-4 * np.abs(one_np).max()
    np.testing.assert_allclose(lse1.cpu().numpy(), lse.cpu().numpy(), atol=1e-3, rtol=0)


def _oracle_ar(kc, vc, p, q, k_cur, v_cur, rows=None):
    hk, hv = host_cache(kc), host_cache(vc)
    n = kc.n_chunks
    d = kc.d
    kh = np.concatenate([oracle_rebuild(hk, p, k) for k in range(n)] + [np.zeros((0, kc.H, d), np.float32)], 0)
    vh = np.concatenate([oracle_rebuild(hv, p, k) for k in range(n)] + [np.zeros((0, kc.H, d), np.float32)], 0)
    qq = q if rows is None else q[rows]
    return oracle.attention_ar(qq, kh, vh, k_cur, v_cur, _slot_of_token(hk, n) if n else np.zeros(0, np.int64),
                               kc.n_tokens, nthreads=NT)


def _ar_case(w, p, seed, n_cache, raw_len=None):
    chunks = [(synth.chunk_kv(w, seed, k, synth.KIND_K), synth.chunk_kv(w, seed, k, synth.KIND_V))
              for k in range(n_cache)]
    if n_cache:
        kc, vc = _cache_with_chunks(w, p, chunks)
    else:
        kc, vc = _new_cache(w, p, 1), _new_cache(w, p, 1)
    k_cur = synth.chunk_kv(w, seed, n_cache, synth.KIND_K)
    v_cur = synth.chunk_kv(w, seed, n_cache, synth.KIND_V)
    if raw_len is not None:
        k_cur, v_cur = k_cur[:raw_len], v_cur[:raw_len]
    q = synth.queries(w, seed, n_cache)
    return kc, vc, k_cur, v_cur, q


@pytest.mark.parametrize("case,n_cache,raw_len", [("tiny", 3, None), ("tiny", 2, 300), ("pro_int2_L3", 1, 45),
                                                  ("pro_int4_L2", 1, 70), ("tiny", 0, 200), ("tiny", 0, 1)])
def test_attention_ar_step(case, n_cache, raw_len):
    """One AR step: the chunk's queries over the compressed cache plus the
    chunk's own raw bf16 K/V (ragged raw tails, a three-stage cache (stage
    count read at run time), a two-stage INT4 cache (stage count compiled
    in), the first chunk with an empty cache, a one-token chunk), against the
    fp64 oracle on the same concatenated keys."""
    w, p, _ = CASES[case]
    kc, vc, k_cur, v_cur, q = _ar_case(w, p, 31, n_cache, raw_len)
    out, lse, top1 = qvg.attention_ar(p, to_dev(q), kc, vc, to_dev(k_cur), to_dev(v_cur), want_lse=True,
                                      want_top1=True)
    ref, rlse, rtop = _oracle_ar(kc, vc, p, q, k_cur, v_cur)
    got = out.cpu().numpy().astype(np.float64)
    _assert_attention(got, ref, q.shape[1])
    hk = host_cache(kc)
    k_abs = np.concatenate([stage_abs_rebuild(hk, p, k) for k in range(kc.n_chunks)] + [np.abs(k_cur)], 0)
    tol = lse_tolerance(q, k_abs, q.shape[1] // w.H)
    assert (np.abs(lse.cpu().numpy() - rlse) <= tol).all(), np.abs(lse.cpu().numpy() - rlse).max()
    assert (top1.cpu().numpy() == rtop).mean() >= 0.99
    if len(k_cur) == 1 and n_cache == 0:  # a single key returns its value (fp16-rounded)
        np.testing.assert_allclose(got, np.broadcast_to(v_cur[0], got.shape), rtol=2 ** -11, atol=2 ** -24)


def test_attention_ar_without_current_chunk_is_attention():
    """n_cur = 0 is qvg_attention, bit for bit."""
    w, p, _ = CASES["tiny"]
    kc, vc, k_cur, v_cur, q = _ar_case(w, p, 32, 2)
    qd = to_dev(q)
    a, la, ta = qvg.attention(p, qd, kc, vc, want_lse=True, want_top1=True)
    z = to_dev(k_cur[:0])
    b, lb, tb = qvg.attention_ar(p, qd, kc, vc, z, z, want_lse=True, want_top1=True)
    assert torch.equal(a, b) and torch.equal(la, lb) and torch.equal(ta, tb)


@pytest.mark.parametrize("Nq", [4680, 16])
def test_attention_ar_longcat(Nq):
    """LongCat-like AR step (16 heads, d=128): 2 cached chunks of 4680
    tokens plus the current chunk's 4680 raw tokens; 4680 queries (64
    sampled rows per head checked) and 16 queries (split-cache path)."""
    w, p, _ = CASES["longcat"]
    kc, vc, k_cur, v_cur, q = _ar_case(w, p, 33, 2)
    q = np.ascontiguousarray(q[:Nq])
    out, lse, top1 = qvg.attention_ar(p, to_dev(q), kc, vc, to_dev(k_cur), to_dev(v_cur), want_lse=True,
                                      want_top1=True)
    rows = np.random.default_rng(2).choice(Nq, min(Nq, 64), replace=False)
    ref, rlse, rtop = _oracle_ar(kc, vc, p, q, k_cur, v_cur, rows)
    _assert_attention(out.cpu().numpy()[rows].astype(np.float64), ref, w.Hq)
    np.testing.assert_allclose(lse.cpu().numpy()[:, rows], rlse, atol=2e-3, rtol=0)
    # near-duplicate keys in a LongCat-like patch: fp16 operand rounding may reorder maxima
    assert (top1.cpu().numpy()[:, rows] == rtop).mean() >= 0.95
    # current-chunk slots are numbered after the cache
    assert top1.max().item() < kc.n_tokens + len(k_cur)


@pytest.mark.parametrize("name", ["tiny_outlier", "pro_outlier_L2", "rtn_outlier_g8", "tiny_outlier_g16",
                                  "tiny_outlier_g64_L2"])
def test_attention_with_outlier_split(name):
    """Attention and the AR step over caches whose K and V carry the
    outlier side list (one and two stages, RTN with G = 8), against the fp64
    oracle on the rebuild of the same bytes."""
    w, p, n_chunks = CASES[name]
    chunks = [(synth.chunk_kv(w, 27, k, synth.KIND_K), synth.chunk_kv(w, 27, k, synth.KIND_V)) for k in range(n_chunks)]
    kc, vc = _cache_with_chunks(w, p, chunks)
    q = synth.queries(w, 27, n_chunks)
    out, lse, top1 = qvg.attention(p, to_dev(q), kc, vc, want_lse=True, want_top1=True)
    ref, rlse, ram, kh, hk = _oracle_attention_on(kc, vc, p, q)
    _assert_attention(out.cpu().numpy().astype(np.float64), ref, w.Hq)
    np.testing.assert_allclose(lse.cpu().numpy(), rlse, atol=2e-3, rtol=0)
    _assert_top1(top1.cpu().numpy(), q, kh, _slot_of_token(hk, n_chunks), ram)
    kr = synth.chunk_kv(w, 27, n_chunks, synth.KIND_K)[:150]
    vr = synth.chunk_kv(w, 27, n_chunks, synth.KIND_V)[:150]
    out, _, _ = qvg.attention_ar(p, to_dev(q), kc, vc, to_dev(kr), to_dev(vr))
    ref, _, _ = _oracle_ar(kc, vc, p, q, kr, vr)
    _assert_attention(out.cpu().numpy().astype(np.float64), ref, w.Hq)


@pytest.mark.parametrize("bits", [2, 4])
def test_attention_two_stage_longcat(bits):
    """LongCat-like caches of two stages (16 heads, d=128, G=64): the
    multi-stage producer adds each stage into the fp16 tile; attention of
    4680 queries (64 sampled rows per head) and 16 queries (split cache)
    against the fp64 oracle on the rebuild of the same bytes."""
    w, p0, _ = CASES["longcat"]
    p = qvg.Params(**{**p0.__dict__, "L": 2, "bits": bits})
    chunks = [(synth.chunk_kv(w, 36, k, synth.KIND_K), synth.chunk_kv(w, 36, k, synth.KIND_V)) for k in range(2)]
    kc, vc = _cache_with_chunks(w, p, chunks)
    q = synth.queries(w, 36, 2)
    out, _, _ = qvg.attention(p, to_dev(q), kc, vc)
    rows = np.random.default_rng(5).choice(q.shape[0], 64, replace=False)
    ref, _, _, _, _ = _oracle_attention_on(kc, vc, p, q, rows)
    _assert_attention(out.cpu().numpy()[rows].astype(np.float64), ref, w.Hq)
    q16 = np.ascontiguousarray(q[:16])
    out, _, _ = qvg.attention(p, to_dev(q16), kc, vc)
    ref, _, _, _, _ = _oracle_attention_on(kc, vc, p, q16)
    _assert_attention(out.cpu().numpy().astype(np.float64), ref, w.Hq)


def test_outlier_split_zero_residual():
    """C = N: every token is its own centroid, so every residual is zero and
    every group ties at the top: nothing is split off (index 0xFF, value 0),
    the scales are 0, and the rebuild is the input."""
    w = W["tiny"]
    p = qvg.Params(C=16, L=1, bits=2, group=32, iters=3, seed=35, flags=qvg.QVG_OUTLIER)
    x = synth.chunk_kv(w, 35, 0, synth.KIND_V)[:16]
    c = _new_cache(w, p, 1, N=16)
    qvg.compress_chunk(p, to_dev(x), c)
    hc = host_cache(c)
    sl = chunk_slice(hc, 0)
    assert np.all(hc["outl_idx"][:, :, sl] == 0xFF) and not hc["outl_val"][:, :, sl].any()
    assert not hc["scales"][:, :, sl].any()
    np.testing.assert_array_equal(qvg.decompress(p, c, 0, 16).cpu().numpy(), x)


def test_outlier_split_longcat():
    """LongCat-like chunks (16 heads, d=128, C=256, INT2 G=64): the split
    lowers the GPU's reconstruction error of V (x300 outlier channels) and
    of K, and attention over the split cache matches the oracle on 64
    sampled query rows."""
    w, p, _ = CASES["longcat_outlier"]
    p0 = qvg.Params(**{**p.__dict__, "flags": 0})
    errs = {}
    for name, pp in (("split", p), ("plain", p0)):
        for kind in (synth.KIND_K, synth.KIND_V):
            x = synth.chunk_kv(w, 28, 0, kind)
            c = _new_cache(w, pp, 1)
            qvg.compress_chunk(pp, to_dev(x), c)
            xh = qvg.decompress(pp, c, 0, w.N).cpu().numpy()
            errs[name, kind] = np.linalg.norm(x - xh) / np.linalg.norm(x)
    for kind in (synth.KIND_K, synth.KIND_V):
        assert errs["split", kind] < errs["plain", kind], errs
    chunks = [(synth.chunk_kv(w, 28, k, synth.KIND_K), synth.chunk_kv(w, 28, k, synth.KIND_V)) for k in range(2)]
    kc, vc = _cache_with_chunks(w, p, chunks)
    q = synth.queries(w, 28, 2)
    out, _, _ = qvg.attention(p, to_dev(q), kc, vc)
    rows = np.random.default_rng(3).choice(q.shape[0], 64, replace=False)
    ref, _, _, _, _ = _oracle_attention_on(kc, vc, p, q, rows)
    _assert_attention(out.cpu().numpy()[rows].astype(np.float64), ref, w.Hq)


@pytest.mark.parametrize("case,every,n_chunks", [("tiny", 2, 4), ("pro_int2_L3", 2, 3), ("tiny_outlier", 3, 4)])
def test_anchor_chunks(case, every, n_chunks):
    """Temporal anchors: every `every`-th chunk is kept as its bf16 K/V.  Its
    stored rows are the input bit for bit, decompress returns them exactly,
    the compressed chunks still match the fed oracle, and attention and the
    AR step over the mixed cache (bf16 anchor tiles between INT2 tiles, one
    and three stages, with the outlier split) match the fp64 oracle."""
    w, p0, _ = CASES[case]
    p = qvg.Params(**{**p0.__dict__, "anchor_every": every})
    chunks = [(synth.chunk_kv(w, 29, k, synth.KIND_K), synth.chunk_kv(w, 29, k, synth.KIND_V)) for k in range(n_chunks)]
    kc, vc = _cache_with_chunks(w, p, chunks)
    hk = host_cache(kc)
    full = qvg.decompress(p, kc, 0, kc.n_tokens).cpu().numpy()
    for k, (x, _) in enumerate(chunks):
        sl = chunk_slice(hk, k)
        if k % every == 0:
            assert hk["chunk_anchor"][k] >= 0
            np.testing.assert_array_equal(oracle_rebuild(hk, p, k), x)
            np.testing.assert_array_equal(full[sl], x)
        else:
            assert hk["chunk_anchor"][k] == -1
            _check_against_fed_oracle(x, hk, p, k)
            np.testing.assert_array_equal(full[sl], oracle_rebuild(hk, p, k))
    q = synth.queries(w, 29, n_chunks)
    out, lse, top1 = qvg.attention(p, to_dev(q), kc, vc, want_lse=True, want_top1=True)
    ref, rlse, ram, kh, hk = _oracle_attention_on(kc, vc, p, q)
    _assert_attention(out.cpu().numpy().astype(np.float64), ref, w.Hq)
    np.testing.assert_allclose(lse.cpu().numpy(), rlse, atol=2e-3, rtol=0)
    _assert_top1(top1.cpu().numpy(), q, kh, _slot_of_token(hk, n_chunks), ram)
    kr = synth.chunk_kv(w, 29, n_chunks, synth.KIND_K)[:100]
    vr = synth.chunk_kv(w, 29, n_chunks, synth.KIND_V)[:100]
    out, _, _ = qvg.attention_ar(p, to_dev(q), kc, vc, to_dev(kr), to_dev(vr))
    ref, _, _ = _oracle_ar(kc, vc, p, q, kr, vr)
    _assert_attention(out.cpu().numpy().astype(np.float64), ref, w.Hq)


def test_anchor_chunks_longcat():
    """LongCat-like (16 heads, d=128, INT2 G=64): the first of 2 chunks is an
    anchor; attention of 4680 queries (64 sampled rows per head checked)
    and 16 queries (split cache) against the oracle."""
    w, p0, _ = CASES["longcat"]
    p = qvg.Params(**{**p0.__dict__, "anchor_every": 2})
    chunks = [(synth.chunk_kv(w, 30, k, synth.KIND_K), synth.chunk_kv(w, 30, k, synth.KIND_V)) for k in range(2)]
    kc, vc = _cache_with_chunks(w, p, chunks)
    q = synth.queries(w, 30, 2)
    out, _, _ = qvg.attention(p, to_dev(q), kc, vc)
    rows = np.random.default_rng(4).choice(q.shape[0], 64, replace=False)
    ref, _, _, _, _ = _oracle_attention_on(kc, vc, p, q, rows)
    _assert_attention(out.cpu().numpy()[rows].astype(np.float64), ref, w.Hq)
    q16 = np.ascontiguousarray(q[:16])
    out, _, _ = qvg.attention(p, to_dev(q16), kc, vc)
    ref, _, _, _, _ = _oracle_attention_on(kc, vc, p, q16)
    _assert_attention(out.cpu().numpy().astype(np.float64), ref, w.Hq)


def test_ragged_and_degenerate_chunks():
    """Chunks of 300 (two tiles plus a ragged 44), 1 token, 10 tokens with
    C=16 > N, and exactly 128 tokens; attention across all of them."""
    w = W["tiny"]
    p = qvg.Params(C=16, L=2, bits=2, group=32, iters=4, seed=9)
    sizes = [300, 1, 10, 128]
    base_k = np.concatenate([synth.chunk_kv(w, 18, k, synth.KIND_K) for k in range(3)], 0)
    base_v = np.concatenate([synth.chunk_kv(w, 18, k, synth.KIND_V) for k in range(3)], 0)
    chunks, off = [], 0
    for n in sizes:
        chunks.append((base_k[off:off + n], base_v[off:off + n]))
        off += n
    kc, vc = _cache_with_chunks(w, p, chunks)
    hk = host_cache(kc)
    assert list(hk["length"][:4]) == sizes and list(hk["start"][:4]) == [0, 384, 512, 640]
    for k, (x, _) in enumerate(chunks):
        _check_against_fed_oracle(x, hk, p, k)
    full = qvg.decompress(p, kc, 0, kc.n_tokens).cpu().numpy()
    assert not full[300:384].any()  # padding slots read as zero
    q = synth.queries(w, 18, 5)[:77]
    out, _, top1 = qvg.attention(p, to_dev(q), kc, vc, want_top1=True)
    ref, _, ram, _, _ = _oracle_attention_on(kc, vc, p, q)
    _assert_attention(out.cpu().numpy().astype(np.float64), ref, w.Hq)
    assert np.all(np.isin(top1.cpu().numpy(), _slot_of_token(hk, 4)))


def test_single_token_cache_returns_value():
    w = W["tiny"]
    p = qvg.Params(C=16, L=1, bits=2, group=32, iters=2)
    k1 = synth.chunk_kv(w, 19, 0, synth.KIND_K)[:1]
    v1 = synth.chunk_kv(w, 19, 0, synth.KIND_V)[:1]
    kc, vc = _cache_with_chunks(w, p, [(k1, v1)])
    q = synth.queries(w, 19, 1)[:5]
    out, _, _ = qvg.attention(p, to_dev(q), kc, vc)
    vhat = qvg.decompress(p, vc, 0, 1).cpu().numpy()
    np.testing.assert_array_equal(out.cpu().numpy(), np.repeat(vhat, 5, 0))


def test_capacity_is_reported():
    w = W["tiny"]
    p = qvg.Params(C=16, L=1, bits=2, group=32, iters=1)
    kc = qvg.CompressedKV(p, w.H, w.d, 256, 1)
    x = to_dev(synth.chunk_kv(w, 20, 0, synth.KIND_K))
    qvg.compress_chunk(p, x, kc)
    with pytest.raises(qvg.QvgError) as e:
        qvg.compress_chunk(p, x, kc)
    assert e.value.status == qvg.QVG_ERR_CAPACITY
    assert kc.n_chunks == 1 and kc.n_tokens == 256


# ---------------------------------------------------------------- QuantWM

def _quantwm_small():
    # QuantWM shapes with 4 KV heads and one 3-frame chunk (2640 tokens)
    import dataclasses
    return dataclasses.replace(W["quantwm"], H=4, Hq=4)


def test_query_stats_and_basis():
    w = _quantwm_small()
    qh = synth.history_queries(w, 21)
    M, wv, cnt = qvg.query_stats(to_dev(qh), w.H)
    Mo, co = oracle.query_stats(qh, w.H)
    assert int(cnt.item()) == co
    Mg = M.cpu().numpy()
    assert np.abs(Mg - Mo).max() <= 1e-5 * np.abs(Mo).max()
    np.testing.assert_allclose(wv.cpu().numpy(), np.einsum("hjj->hj", Mo) / co, rtol=1e-5)
    M2, _, cnt2 = qvg.query_stats(to_dev(qh), w.H, M=M.clone(), count=cnt.clone(), accumulate=True)
    assert int(cnt2.item()) == 2 * co
    np.testing.assert_allclose(M2.cpu().numpy(), 2 * Mg, rtol=1e-6)
    U, eig, frac = qvg.psac_basis(M, cnt)
    Uo, eo, fo = oracle.psac_basis(Mg.astype(np.float64), co, 8)
    np.testing.assert_allclose(eig.cpu().numpy(), eo, rtol=1e-4)
    np.testing.assert_allclose(frac.cpu().numpy(), fo, atol=1e-5)
    Ug = U.cpu().numpy()
    for h in range(w.H):
        dots = np.einsum("dk,dk->k", Ug[h], Uo[h])
        assert dots.min() > 1 - 1e-4, dots
        # fp32 Jacobi: each of ~10 sweeps applies d-1 rotations to every
        # column pair, so orthonormality drifts by ~sweeps * d * 2^-24 ~ 1e-4
        np.testing.assert_allclose(Ug[h].T @ Ug[h], np.eye(8), atol=2e-4)
    assert 0.69 < frac.cpu().numpy().min() and frac.cpu().numpy().max() < 0.75


@pytest.mark.parametrize("flags,anchor_every,L", [(qvg.QVG_QSAC, 0, 1), (qvg.QVG_PSAC, 0, 1),
                                                  (qvg.QVG_QSAC | qvg.QVG_PSAC, 0, 1),
                                                  (qvg.QVG_QSAC | qvg.QVG_PSAC, 2, 1), (qvg.QVG_PSAC, 0, 2),
                                                  (qvg.QVG_PSAC | qvg.QVG_OUTLIER, 0, 1)])
def test_quantwm_compress_and_attention(flags, anchor_every, L):
    """QuantWM caches (QSAC weights, PSAC on K; with anchor_every = 2 the
    first chunk is a bf16 anchor, which carries no PSAC term; two stages
    with PSAC; PSAC with the outlier split, which K and V then both carry):
    compression against the fed oracle, PSAC codes, the rebuild, and
    attention (plain and AR step) against the fp64 oracle.  The attention
    kernel takes PSAC as a tensor-core product, one buffer fill per stage,
    and with the outlier split the general producer."""
    w = _quantwm_small()
    qh = synth.history_queries(w, 22)
    M, wv, cnt = qvg.query_stats(to_dev(qh), w.H)
    U, _, _ = qvg.psac_basis(M, cnt)
    p = qvg.Params(C=256, L=L, bits=2, group=64, iters=8, seed=23, flags=flags, anchor_every=anchor_every)
    chunks = [(synth.chunk_kv(w, 23, k, synth.KIND_K), synth.chunk_kv(w, 23, k, synth.KIND_V)) for k in range(2)]
    cap = 2 * (-(-w.N // 128) * 128)
    kc = qvg.CompressedKV(p, w.H, w.d, cap, 2)
    pv = qvg.Params(**{**p.__dict__, "flags": flags & qvg.QVG_OUTLIER})
    vc = qvg.CompressedKV(pv, w.H, w.d, cap, 2)
    for k, v in chunks:
        qvg.compress_chunk(p, to_dev(k), kc, qsac_w=wv, psac_basis=U)
        qvg.compress_chunk(pv, to_dev(v), vc)
    hk = host_cache(kc)
    ww = wv.cpu().numpy() if flags & qvg.QVG_QSAC else None
    Uh = U.cpu().numpy() if flags & qvg.QVG_PSAC else None
    for k, (x, _) in enumerate(chunks):
        if anchor_every and k % anchor_every == 0:
            np.testing.assert_array_equal(oracle_rebuild(hk, p, k), x)
            continue
        o, ok = _check_against_fed_oracle(x, hk, p, k, w=ww, psac_U=Uh)
        if Uh is not None:
            sl = chunk_slice(hk, k)
            np.testing.assert_array_equal(hk["psac_basis"][k], Uh)
            for h in range(w.H):
                np.testing.assert_array_equal(hk["psac_p"][h, sl][ok[h]], o["psac_p"][h][ok[h]])
                np.testing.assert_array_equal(hk["psac_s"][h, sl][ok[h]], o["psac_s"][h][ok[h]])
            gpu = qvg.decompress(p, kc, int(hk["start"][k]), int(hk["length"][k])).cpu().numpy()
            ref = oracle_rebuild(hk, p, k)
            assert np.abs(gpu - ref).max() <= 1e-3 * np.abs(ref).max()
    q = synth.history_queries(w, 24, n_tokens=300, stream=1)
    out, _, top1 = qvg.attention(p, to_dev(q), kc, vc, want_top1=True)
    hv = host_cache(vc)
    kh = np.concatenate([oracle_rebuild(hk, p, k) for k in range(2)], 0)
    vh = np.concatenate([oracle_rebuild(hv, pv, k) for k in range(2)], 0)
    ref, _, ram = oracle.attention(q, kh, vh, nthreads=NT)
    _assert_attention(out.cpu().numpy().astype(np.float64), ref, w.Hq)
    # the top-1 slot (the shift rate's GPU side) over the rebuilt keys,
    # PSAC term included
    _assert_top1(top1.cpu().numpy(), q, kh, _slot_of_token(hk, 2), ram)
    # AR step on the same cache: the third chunk's raw K/V join the keys
    # (the PSAC term corrects cached keys only)
    kr, vr = synth.chunk_kv(w, 23, 2, synth.KIND_K)[:700], synth.chunk_kv(w, 23, 2, synth.KIND_V)[:700]
    out, _, _ = qvg.attention_ar(p, to_dev(q), kc, vc, to_dev(kr), to_dev(vr))
    ref, _, _ = oracle.attention_ar(q, kh, vh, kr, vr, _slot_of_token(hk, 2), kc.n_tokens, nthreads=NT)
    _assert_attention(out.cpu().numpy().astype(np.float64), ref, w.Hq)
