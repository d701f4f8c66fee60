"""CPU checks of the host-side logic around the kernels: the seeded input
generators keep the properties the input recipe states, and the benchmark's
helpers (source hash of the attention kernel, clock-record parsing, launch
count, config) behave as their docstrings say.  No GPU needed."""
import os
import shutil

import numpy as np
import pytest

import bench
import video_diffusion_kv_gb300 as qvg
from video_diffusion_kv_gb300 import synth

W = synth.WORKLOADS


# ------------------------------------------------------------------ inputs

@pytest.mark.parametrize("name", ["tiny", "qvgpro"])
def test_chunks_are_seeded_bf16_token_major(name):
    w = W[name]
    a = synth.chunk_kv(w, 5, 1, synth.KIND_K)
    assert a.shape == (w.N, w.H, w.d) and a.dtype == np.float32
    np.testing.assert_array_equal(a, synth.bf16_values(a))        # bf16-representable
    np.testing.assert_array_equal(a, synth.chunk_kv(w, 5, 1, synth.KIND_K))  # seeded
    assert not np.array_equal(a, synth.chunk_kv(w, 6, 1, synth.KIND_K))
    assert not np.array_equal(a, synth.chunk_kv(w, 5, 2, synth.KIND_K))
    assert not np.array_equal(a, synth.chunk_kv(w, 5, 1, synth.KIND_V))


def test_outlier_magnitudes_follow_the_recipe():
    """Outlier channels carry x50 (K) and x300 (V) over unit-scale
    prototypes: max|K| of order 1e2, max|V| of order 1e3, while the bulk of
    the values stays of order 1."""
    w = W["tiny"]
    k = np.concatenate([synth.chunk_kv(w, 1, c, synth.KIND_K) for c in range(w.n_chunks)])
    v = np.concatenate([synth.chunk_kv(w, 1, c, synth.KIND_V) for c in range(w.n_chunks)])
    assert 30 < np.abs(k).max() < 600
    assert 200 < np.abs(v).max() < 4000
    assert np.median(np.abs(k)) < 2 and np.median(np.abs(v)) < 2


def test_ar1_neighbouring_frames_are_correlated():
    """The ar1 workload's prototype means follow an AR(1) over frames with
    rho = 0.95: consecutive frames' tokens correlate strongly, chunks far
    apart much less."""
    w = W["longcat"]
    mu = synth._ar1_means(w, 3, synth.KIND_K, 25)
    c1 = np.corrcoef(mu[10].ravel(), mu[11].ravel())[0, 1]
    c24 = np.corrcoef(mu[0].ravel(), mu[24].ravel())[0, 1]
    assert c1 > 0.9
    assert c24 < c1 - 0.3


def test_grouped_queries_repeat_the_kv_head():
    import dataclasses
    w = dataclasses.replace(W["tiny"], Hq=4)
    q = synth.queries(w, 2, 0)
    assert q.shape == (w.Nq, 4, w.d)
    np.testing.assert_array_equal(q[:, 0], q[:, 1])
    np.testing.assert_array_equal(q[:, 2], q[:, 3])


def test_history_queries_hold_the_planted_energy():
    """70 % of the history queries' expected energy lies in the 8 planted
    orthonormal directions, geometric with ratio 0.8."""
    w = W["quantwm"]
    lam, sigma2 = synth.planted_spectrum(w.d)
    assert np.isclose(lam.sum(), 0.70 * w.d) and np.allclose(lam[1:] / lam[:-1], 0.8)
    assert np.isclose(lam.sum() + sigma2 * w.d, w.d)
    U = synth.planted_basis(w, 9)
    for h in range(w.H):
        np.testing.assert_allclose(U[h].T @ U[h], np.eye(8), atol=1e-12)
    q = synth.history_queries(w, 9, n_tokens=4096).astype(np.float64)
    for h in (0, w.H - 1):
        proj = q[:, h] @ U[h]
        frac = (proj ** 2).sum() / (q[:, h] ** 2).sum()
        assert abs(frac - (0.70 + 0.30 * 8 / w.d)) < 0.03, frac


def test_history_queries_channel_activity():
    """The queries' per-channel activity (mean q_j^2, the QSAC weight) is
    3.1 on the quarter of channels that carry the planted directions and
    0.3 on the rest; its mean over channels is 1 (E||q||^2 = d)."""
    w = W["quantwm"]
    act = synth.active_channels(w, 9)
    assert act.shape == (w.H, w.d // 4)
    U = synth.planted_basis(w, 9)
    for h in range(w.H):
        off = np.setdiff1d(np.arange(w.d), act[h])
        assert np.abs(U[h][off]).max() == 0.0
    q = synth.history_queries(w, 9, n_tokens=20000).astype(np.float64)
    for h in (0, w.H - 1):
        m = (q[:, h] ** 2).mean(0)
        on = np.zeros(w.d, bool)
        on[act[h]] = True
        assert abs(m[on].mean() - 3.1) < 0.1 and abs(m[~on].mean() - 0.3) < 0.02
        assert abs(m.mean() - 1.0) < 0.03


# ------------------------------------------------------------------ benchmark helpers

def test_attention_hash_ignores_comments_only(tmp_path, monkeypatch):
    """The recorded DRAM traffic is keyed by the attention sources with
    comments and blank lines removed: a comment edit keeps the key, a code
    edit changes it."""
    src = os.path.join(bench.ROOT, "video_diffusion_kv_gb300", "csrc")
    dst = tmp_path / "video_diffusion_kv_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in bench.ATTN_SOURCES:
        shutil.copy(os.path.join(src, f), dst / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench._attn_source_hash()
    p = dst / "common.cuh"
    text = p.read_text()
    p.write_text("// a new comment\n\n/* and a block\n   comment */\n" + text + "\n// trailing\n")
    assert bench._attn_source_hash() == h0
    p.write_text(text + "\nconstexpr int kUnusedProbe = 1;\n")
    assert bench._attn_source_hash() != h0


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


class _FakeThread:
    def join(self, timeout=None):
        pass


def _sampler(lines, first=0):
    s = bench.ClockSampler(0)
    s.proc, s.thread, s.lines, s.first = _FakeProc(), _FakeThread(), list(lines), first
    return s


def test_clock_record_parsing():
    ok = "2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"
    capped = "1980, 2070, 1400.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active"
    hot = "1500, 2070, 1200.0, 0x0000000000000040, Not Active, Active, Not Active, Not Active"
    r = _sampler([ok, ok, capped]).stop()
    assert r["sm_mhz"] == 2070 and r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"] and r["samples"] == 3
    # only the samples from the start of the timed region count
    r = _sampler([hot, ok, ok], first=1).stop()
    assert r["reasons"] == [] and r["samples"] == 2
    # none inside: the last one read before it
    r = _sampler([ok, hot], first=2).stop()
    assert r["reasons"] == ["hw_thermal_slowdown"] and r["sm_mhz"] == 1500
    # malformed lines are skipped
    r = _sampler(["garbage", ok]).stop()
    assert r["samples"] == 1
    s = bench.ClockSampler(0)
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_launch_count_per_compress():
    """One compress call: per stage, row norms + init + iters x (assign,
    update) + final assign + quantise; then the chunk table."""
    p = qvg.Params(C=256, L=1, bits=2, group=64, iters=8)
    assert bench.launches_per_compress(p) == 1 + 1 + 16 + 1 + 1 + 1
    p3 = qvg.Params(C=16, L=3, bits=2, group=32, iters=10)
    assert bench.launches_per_compress(p3) == 3 * (1 + 1 + 20 + 1 + 1) + 1
    rtn = qvg.Params(C=0, L=1, bits=2, group=32, iters=0)
    assert bench.launches_per_compress(rtn) == 2


def test_config_names_the_workload_only():
    w = bench._workload()
    cfg = bench._config(w, {"parallelism": "single GPU"})
    assert "workload" in cfg and "model" not in cfg
    assert cfg["tokens_per_chunk"] == w.N and cfg["cache_tokens"] == w.N * w.n_chunks
    small = bench._workload(cache_chunks=2)
    assert small.n_chunks == 2 and small.N == w.N
