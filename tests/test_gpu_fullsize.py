"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (all heads, all query tokens in one call), checked on
sampled outputs the fp64 oracle can compute one by one: compression on
sampled (chunk, head) pairs against the oracle fed the GPU's centroids, and
attention rows sampled from the full query chunk over the whole cache.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import video_diffusion_kv_gb300 as qvg
from video_diffusion_kv_gb300 import synth

from _helpers import ATTN_TOL, assignment_mismatches, host_cache, oracle_rebuild, to_dev

pytestmark = pytest.mark.gpu
NT = 16


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _sub(hc, heads):
    """The host cache restricted to some heads (oracle layout per chunk)."""
    out = dict(hc)
    for k in ("codes", "scales", "ids", "cent"):
        if k in hc:
            out[k] = hc[k][:, heads]
    if "psac_p" in hc:
        out["psac_p"] = hc["psac_p"][heads]
        out["psac_s"] = hc["psac_s"][heads]
        out["psac_basis"] = hc["psac_basis"][:, heads]
    return out


def _check_chunk_heads(x, hc, p, k, heads, w=None, U=None):
    """Fed-oracle check of chunk k on a subset of heads: ids (near ties
    excepted), codes and scales bit for bit, PSAC codes bit for bit."""
    sub = _sub(hc, heads)
    s = int(sub["start"][k])
    n = int(sub["length"][k])
    sl = slice(s, s + n)
    xs = x[:, heads]
    cent = sub["cent"][:, :, k]
    o = oracle.compress_chunk(xs, C=p.C, L=p.L, bits=p.bits, group=p.group, iters=0, seed=p.seed, chunk=k,
                              qsac_w=None if w is None else w[heads], psac_U=None if U is None else U[heads],
                              cent_in=oracle.bf16_bits_to_f32(cent), nthreads=NT)
    near = total = 0
    for i in range(len(heads)):
        ids = sub["ids"][0, i, sl]
        m, far = assignment_mismatches(xs[:, i], cent[0, i, :min(p.C, n)], ids.astype(np.int32),
                                       None if w is None else w[heads][i])
        assert far == 0
        near += m
        total += n
        ok = ids == o["ids"][0, i]
        np.testing.assert_array_equal(sub["codes"][0, i, sl][ok], o["codes"][0, i][ok])
        np.testing.assert_array_equal(sub["scales"][0, i, sl][ok], o["scales"][0, i][ok])
        if U is not None:
            np.testing.assert_array_equal(sub["psac_p"][i, sl][ok], o["psac_p"][i][ok])
    assert near <= max(1, 1e-4 * total), (near, total)


def _oracle_attention_rows(kc, vc, p, pv, q, rows, heads_k):
    hk, hv = host_cache(kc), host_cache(vc)
    kh = np.concatenate([oracle_rebuild(hk, p, k) for k in range(kc.n_chunks)], 0)
    vh = np.concatenate([oracle_rebuild(hv, pv, k) for k in range(vc.n_chunks)], 0)
    out, _, _ = oracle.attention(q[rows], kh, vh, nthreads=NT)
    return out


def _assert_rows(got, ref):
    for h in range(ref.shape[1]):
        err = np.abs(got[:, h] - ref[:, h]).max() / np.abs(ref[:, h]).max()
        assert err <= ATTN_TOL, (h, err)


def _stream(w, p, pv, kinds_seed, chunks, qsac_w=None, U=None, uniq=None):
    per = -(-w.N // 128) * 128
    kc = qvg.CompressedKV(p, w.H, w.d, chunks * per, chunks)
    vc = qvg.CompressedKV(pv, w.H, w.d, chunks * per, chunks)
    xs = {}
    for k in range(chunks):
        src = k if uniq is None else k % uniq
        if src not in xs:
            xs[src] = (synth.chunk_kv(w, kinds_seed, src, synth.KIND_K), synth.chunk_kv(w, kinds_seed, src, synth.KIND_V))
        qvg.compress_chunk(p, to_dev(xs[src][0]), kc, qsac_w=qsac_w, psac_basis=U)
        qvg.compress_chunk(pv, to_dev(xs[src][1]), vc)
    assert qvg.get_status() == qvg.QVG_OK
    return kc, vc, xs


def test_longcat_full():
    """16 heads, d=128, 8 chunks x 4680 (37,440 tokens), C=256, INT2 G=64,
    8 iterations; 4680 queries in one call."""
    w = synth.WORKLOADS["longcat"]
    p = qvg.Params(C=w.C, L=1, bits=w.bits, group=w.group, iters=w.iters, seed=41)
    kc, vc, xs = _stream(w, p, p, 41, w.n_chunks)
    hk = host_cache(kc)
    for k in (0, w.n_chunks - 1):
        _check_chunk_heads(xs[k][0], hk, p, k, [0, 7, 15])
    q = synth.queries(w, 41, w.n_chunks - 1)
    out, _, _ = qvg.attention(p, to_dev(q), kc, vc)
    rows = np.random.default_rng(2).choice(w.Nq, 64, replace=False)
    ref = _oracle_attention_rows(kc, vc, p, p, q, rows, None)
    _assert_rows(out.cpu().numpy()[rows].astype(np.float64), ref)


def test_quantwm_full_qsac_psac():
    """24 heads, d=128, 8 chunks x 2640 (21,120 tokens), C=256, INT2 G=64,
    QSAC weights and the PSAC basis from 3520 history queries per head;
    880 queries in one call."""
    w = synth.WORKLOADS["quantwm"]
    qh = synth.history_queries(w, 42)
    M, wq, cnt = qvg.query_stats(to_dev(qh), w.H)
    U, _, frac = qvg.psac_basis(M, cnt)
    assert 0.69 < float(frac.min()) and float(frac.max()) < 0.75
    p = qvg.Params(C=w.C, L=1, bits=w.bits, group=w.group, iters=w.iters, seed=42,
                   flags=qvg.QVG_QSAC | qvg.QVG_PSAC)
    pv = qvg.Params(C=w.C, L=1, bits=w.bits, group=w.group, iters=w.iters, seed=42)
    kc, vc, xs = _stream(w, p, pv, 42, w.n_chunks, qsac_w=wq, U=U)
    hk = host_cache(kc)
    wn, Un = wq.cpu().numpy(), U.cpu().numpy()
    for k in (0, w.n_chunks - 1):
        _check_chunk_heads(xs[k][0], hk, p, k, [0, 11, 23], w=wn, U=Un)
    q = synth.history_queries(w, 42, n_tokens=w.Nq, stream=1)
    out, _, _ = qvg.attention(p, to_dev(q), kc, vc)
    rows = np.random.default_rng(3).choice(w.Nq, 64, replace=False)
    ref = _oracle_attention_rows(kc, vc, p, pv, q, rows, None)
    _assert_rows(out.cpu().numpy()[rows].astype(np.float64), ref)


def test_rollout_full():
    """8 heads, d=128, 96 chunks x 4680 (449,280 tokens) streamed into one
    cache (12 distinct chunks of the stationary mixture, cycled); the last
    chunk's 4680 queries attend over the whole cache in one call."""
    w = synth.WORKLOADS["rollout"]
    p = qvg.Params(C=w.C, L=1, bits=w.bits, group=w.group, iters=w.iters, seed=43)
    kc, vc, xs = _stream(w, p, p, 43, w.n_chunks, uniq=12)
    hk = host_cache(kc)
    for k in (0, 50, w.n_chunks - 1):
        _check_chunk_heads(xs[k % 12][0], hk, p, k, [0, 5])
    q = synth.queries(w, 43, w.n_chunks - 1)
    out, _, _ = qvg.attention(p, to_dev(q), kc, vc)
    rows = np.random.default_rng(4).choice(w.Nq, 24, replace=False)
    ref = _oracle_attention_rows(kc, vc, p, p, q, rows, None)
    _assert_rows(out.cpu().numpy()[rows].astype(np.float64), ref)
