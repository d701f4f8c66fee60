"""k-means on the GPU against the oracle, step by step through a full run
(Quant VideoGen notes, "Semantic-Aware Smoothing": per chunk and head, the
tokens are clustered by k-means and each token's centroid is subtracted).

The GPU run with `iters = i` leaves the centroids c_i after i Lloyd updates
and the ids of the assignment to c_i; with QVG_KEEP_MEANS it also leaves the
fp32 means of its last update.  Since the GPU is deterministic, the runs
with i = 0 .. I trace one trajectory of the full I-iteration run.  Along it:

  - every update: the fp32 means equal the oracle's update of the GPU's own
    ids and centroids within 1e-4 of the centroid row's largest magnitude
    (the fp32 bar), and the stored bf16 centroids are the round-to-nearest
    of those fp32 means and within 1 bf16 ulp of the oracle's;
  - every assignment: the GPU's ids are the oracle's fp64 argmin over the
    GPU's own centroids except at near ties (the assignment bar);
  - the whole trajectory is compared with the oracle's own run from the same
    seed: the iteration at which the two first assign a token differently
    (through a near tie or a one-ulp centroid rounding) is recorded, and
    where they never do, the final centroids agree within 1 bf16 ulp.
"""
import numpy as np
import pytest
import torch

import oracle
import video_diffusion_kv_gb300 as qvg
from video_diffusion_kv_gb300 import synth

from _helpers import assignment_mismatches, bf16_ulp_diff, host_cache, to_dev

pytestmark = pytest.mark.gpu
MEAN_TOL = 1e-4  # fp32 means: max |dm| / max |m_oracle| per centroid row
W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _gpu_run(w, base, x, chunk_slots, n_prev, iters):
    """Compress x as chunk n_prev of a fresh cache with `iters` Lloyd
    iterations and QVG_KEEP_MEANS; returns (cent bits [H,C,d], ids [H,N],
    fp32 means [H,C,d] or None)."""
    p = qvg.Params(**{**base.__dict__, "iters": iters, "flags": base.flags | qvg.QVG_KEEP_MEANS})
    N = x.shape[0]
    c = qvg.CompressedKV(p, w.H, w.d, (n_prev + 1) * chunk_slots, n_prev + 1)
    c.reset(n_prev, n_prev * chunk_slots)  # earlier slots stay empty: the chunk index seeds the init
    ws = torch.empty(qvg.workspace_size(p, qvg.QVG_OP_COMPRESS, N, w.H, w.d), dtype=torch.uint8, device="cuda")
    qvg.compress_chunk(p, to_dev(x), c, workspace=ws)
    assert qvg.get_status() == qvg.QVG_OK
    hc = host_cache(c)
    s0 = n_prev * chunk_slots
    means = qvg.kept_means(p, ws, w.H, w.d)[0].cpu().numpy().copy() if iters > 0 else None
    return hc["cent"][0, :, n_prev], hc["ids"][0, :, s0:s0 + N].astype(np.int32), means


def _bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("wname,base,chunks,heads", [
    ("tiny", qvg.Params(C=16, L=1, bits=2, group=32, iters=10, seed=61), [0, 1, 2, 3], [0, 1]),
    ("longcat", qvg.Params(C=256, L=1, bits=2, group=64, iters=8, seed=62), [5], [0, 9]),
])
def test_full_lloyd_trajectory(wname, base, chunks, heads):
    w = W[wname]
    slots = -(-w.N // 128) * 128
    I = base.iters
    report, final_or = [], {}
    for k in chunks:
        x = synth.chunk_kv(w, 71, k, synth.KIND_K if k % 2 == 0 else synth.KIND_V)
        runs = [_gpu_run(w, base, x, slots, k, i) for i in range(I + 1)]
        N = x.shape[0]
        Ce = min(base.C, N)
        for h in heads:
            g = x[:, h]
            # the oracle's own run from the same seed: seeded picks, then I x (assign, update)
            picks = oracle.init_picks(N, Ce, base.seed, k, h, 0)
            c_or = g[picks].copy()
            diverged_at, cause = None, None
            for i in range(I + 1):
                cent_g, ids_g, means_g = runs[i]
                cg = oracle.bf16_bits_to_f32(cent_g[h, :Ce])
                if i == 0:
                    np.testing.assert_array_equal(cent_g[h, :Ce], _bits(c_or))  # seeded init, bit for bit
                else:
                    # update i along the GPU trajectory: from the GPU's ids and centroids of step i-1
                    _, ids_prev, _ = runs[i - 1]
                    c_prev = oracle.bf16_bits_to_f32(runs[i - 1][0][h, :Ce])
                    ref_c, ref_m, cnt = oracle.update(g, ids_prev[h], c_prev)
                    m = means_g[h, :Ce]
                    row_max = np.abs(ref_m).max(1)
                    rel = np.abs(m - ref_m).max(1) / np.where(row_max > 0, row_max, 1.0)
                    assert rel.max() <= MEAN_TOL, (wname, k, h, i, float(rel.max()))
                    np.testing.assert_array_equal(cent_g[h, :Ce], _bits(m))  # stored = RNE of the fp32 mean
                    assert bf16_ulp_diff(cent_g[h, :Ce], _bits(ref_c)).max() <= 1, (wname, k, h, i)
                # assignment i: fp64 argmin over the GPU's own centroids, except near ties
                _, far = assignment_mismatches(g, cent_g[h, :Ce], ids_g[h])
                assert far == 0, ("assignment outside near ties", wname, k, h, i)
                # the oracle's own trajectory
                ids_or, _, _, _ = oracle.assign(g, c_or)
                if diverged_at is None:
                    ulps = bf16_ulp_diff(cent_g[h, :Ce], _bits(c_or))
                    assert ulps.max() <= 1, (wname, k, h, i, int(ulps.max()))
                    if (ids_or != ids_g[h]).any():
                        diverged_at = i
                        cause = "near tie" if ulps.max() == 0 else "one-ulp centroid"
                if i < I:
                    c_or, _, _ = oracle.update(g, ids_or, c_or)
            report.append((k, h, diverged_at, cause))
            final_or[(k, h)] = c_or
    print("k-means trajectories (chunk, head, first iteration with a different assignment, cause):", report)
    # the step-by-step oracle loop above is the oracle's own compression (the
    # same definition composed the same way): same final centroids, bit for bit
    k = chunks[0]
    x = synth.chunk_kv(w, 71, k, synth.KIND_K if k % 2 == 0 else synth.KIND_V)
    o = oracle.compress_chunk(x, C=base.C, L=1, bits=base.bits, group=base.group, iters=I, seed=base.seed,
                              chunk=k, nthreads=16)
    for h in heads:
        np.testing.assert_array_equal(o["cent"][0, h, :final_or[(k, h)].shape[0]], _bits(final_or[(k, h)]))


@pytest.mark.parametrize("wname,seed", [("tiny", 63), ("longcat", 64)])
def test_update_fp32_means_from_given_centroids(wname, seed):
    """One Lloyd update from caller-given centroids c0: the fp32 means the
    GPU leaves with QVG_KEEP_MEANS equal the oracle's mean of the same
    members within 1e-4 of the row's largest magnitude; an empty cluster
    keeps c0 exactly."""
    w = W[wname]
    C = 16 if wname == "tiny" else 256
    x = synth.chunk_kv(w, seed, 0, synth.KIND_K)
    N = x.shape[0]
    rng = np.random.default_rng(seed)
    c0 = np.stack([x[rng.choice(N, C, replace=False), h] for h in range(w.H)])
    c0[:, C - 1] = 1e4  # far from every token: stays empty
    c0_bits = torch.from_numpy(c0).to(torch.bfloat16).view(torch.int16)
    out = {}
    for iters in (0, 1):
        p = qvg.Params(C=C, L=1, bits=2, group=w.group, iters=iters,
                       flags=qvg.QVG_GIVEN_CENTROIDS | qvg.QVG_KEEP_MEANS)
        kc = qvg.CompressedKV(p, w.H, w.d, -(-N // 128) * 128, 1)
        kc.view("cent", torch.int16, (1, w.H, 1, C, w.d))[0, :, 0] = c0_bits.cuda()
        ws = torch.empty(qvg.workspace_size(p, qvg.QVG_OP_COMPRESS, N, w.H, w.d), dtype=torch.uint8, device="cuda")
        qvg.compress_chunk(p, to_dev(x), kc, workspace=ws)
        assert qvg.get_status() == qvg.QVG_OK
        out[iters] = (host_cache(kc), qvg.kept_means(p, ws, w.H, w.d)[0].cpu().numpy().copy())
    ids0 = out[0][0]["ids"][0, :, :N].astype(np.int32)
    means = out[1][1]
    c0f = oracle.bf16_bits_to_f32(c0_bits.numpy().view(np.uint16))
    worst = 0.0
    for h in range(w.H):
        _, ref_m, cnt = oracle.update(x[:, h], ids0[h], c0f[h])
        assert cnt[C - 1] == 0
        np.testing.assert_array_equal(means[h, C - 1], c0f[h, C - 1])
        row_max = np.abs(ref_m).max(1)
        rel = np.abs(means[h] - ref_m).max(1) / np.where(row_max > 0, row_max, 1.0)
        worst = max(worst, float(rel.max()))
    assert worst <= MEAN_TOL, worst
    print("%s: worst row-relative fp32 mean difference %.3g" % (wname, worst))
