"""Seeded synthetic video-KV workloads.

This module only draws inputs: bf16 K/V chunks shaped like an
autoregressive video model's cache, query tokens, and history queries with
a planted spectrum.  It holds none of the compression arithmetic and is the
only code that both the CUDA path's tests and the CPU oracle's tests share.

Shapes follow the workloads the pages describe: LongCat-Video-like chunks
of 3 latent frames of 30x52 tokens (~38K tokens over 8 chunks, the
"LongCat-Video needs ~38K latent tokens for 5 s" figure in the QVG notes),
a world-model cache of 22x40 frames (QuantWM write-up), and a one-minute
rollout.  Value structure: token-varying outlier channels with max|K|~1e2 and
max|V|~1e3 (QVG notes, "core tension"), spatio-temporally correlated
prototypes (QVG notes, "entry angle": neighbouring frames and patches hold
similar tokens), and history queries whose energy sits in 8 directions
(QuantWM write-up, PSAC: top-8 directions hold >71% of query energy) on a
quarter of the channels (QSAC: queries are more active on some channels).

Every array is float32 holding bf16-representable values, layout
[tokens, heads, head_dim] (token-major, tokens in raster order
frame, y, x).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

KIND_K, KIND_V, KIND_Q, KIND_QHIST, KIND_QSHIFT = 1, 2, 3, 4, 5


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    H: int                 # KV heads
    d: int                 # head_dim
    frame_hw: tuple        # latent frame (rows, cols)
    frames_per_chunk: int  # T_c
    n_chunks: int          # chunks held in the cache
    dist: str              # "mixture" (16 prototypes) or "ar1" (per-patch AR(1))
    C: int                 # clusters
    L: int                 # progressive stages
    bits: int
    group: int
    iters: int
    Hq: int
    Nq: int                # query tokens per attention call
    patch: tuple = (5, 4)  # prototype patch (rows, cols) for "ar1"
    rho: float = 0.95
    n_proto: int = 16
    sigma: float = 0.1
    p_out: float = 0.02
    k_out: float = 50.0
    v_out: float = 300.0
    hist_frames: int = 0   # history-query frames (QuantWM)

    @property
    def N(self):
        return self.frame_hw[0] * self.frame_hw[1] * self.frames_per_chunk

    @property
    def tokens(self):
        return self.N * self.n_chunks


WORKLOADS = {
    # 2 KV heads, d=64, 4 chunks of one 16x16 frame; 16-prototype mixture.
    "tiny": Workload("tiny", H=2, d=64, frame_hw=(16, 16), frames_per_chunk=1,
                     n_chunks=4, dist="mixture", C=16, L=1, bits=2, group=32,
                     iters=10, Hq=2, Nq=256),
    # LongCat-like layer: 16 heads, d=128, 8 chunks of 3 frames of 30x52.
    "longcat": Workload("longcat", H=16, d=128, frame_hw=(30, 52), frames_per_chunk=3,
                        n_chunks=8, dist="ar1", C=256, L=1, bits=2, group=64,
                        iters=8, Hq=16, Nq=4680),
    # QVG-Pro study on the tiny shapes (stages and bits vary per arm).
    "qvgpro": Workload("qvgpro", H=2, d=64, frame_hw=(16, 16), frames_per_chunk=1,
                       n_chunks=4, dist="mixture", C=16, L=3, bits=2, group=32,
                       iters=10, Hq=2, Nq=256),
    # QuantWM world-model cache: 24 heads, 24 frames of 22x40, chunks of 3 frames.
    "quantwm": Workload("quantwm", H=24, d=128, frame_hw=(22, 40), frames_per_chunk=3,
                        n_chunks=8, dist="ar1", C=256, L=1, bits=2, group=64,
                        iters=8, Hq=24, Nq=880, hist_frames=4),
    # One-minute rollout: 288 frames of 30x52 in 96 chunks, 8 heads.
    "rollout": Workload("rollout", H=8, d=128, frame_hw=(30, 52), frames_per_chunk=3,
                        n_chunks=96, dist="mixture", C=256, L=1, bits=2, group=64,
                        iters=8, Hq=8, Nq=4680),
}


def bf16_values(a: np.ndarray) -> np.ndarray:
    """Round to bf16 (round-to-nearest-even) and return as float32."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def _rng(seed, *tags):
    return np.random.default_rng([int(seed) & 0xFFFFFFFF] + [int(t) for t in tags])


def _patch_index(w: Workload):
    rows, cols = w.frame_hw
    pr, pc = w.patch
    npc = -(-cols // pc)
    y = np.arange(rows)[:, None] // pr
    x = np.arange(cols)[None, :] // pc
    return (y * npc + x).reshape(-1), (-(-rows // pr)) * npc


def _ar1_means(w: Workload, seed, kind, n_frames):
    """Per-patch prototype means evolving as AR(1) over frames:
    mu_f = rho mu_{f-1} + sqrt(1 - rho^2) eta_f,  mu_0 ~ N(0, 1)."""
    _, n_patch = _patch_index(w)
    g = _rng(seed, kind, 7777)
    mu = np.empty((n_frames, n_patch, w.H, w.d), np.float32)
    mu[0] = g.standard_normal((n_patch, w.H, w.d), dtype=np.float32)
    a = math.sqrt(1.0 - w.rho * w.rho)
    for f in range(1, n_frames):
        mu[f] = w.rho * mu[f - 1] + a * g.standard_normal((n_patch, w.H, w.d), dtype=np.float32)
    return mu


def _mixture_protos(w: Workload, seed, kind):
    g = _rng(seed, kind, 8888)
    return g.standard_normal((w.H, w.n_proto, w.d), dtype=np.float32)


def _outlier_scale(w: Workload, seed, kind, n_proto):
    """Per (prototype, head, channel) multiplier: k_out / v_out with
    probability p_out, else 1.  Tokens inherit their prototype's outlier
    channels, so the outlier channels vary from token to token and are
    shared by tokens of similar content."""
    mult = w.k_out if kind == KIND_K else w.v_out
    g = _rng(seed, kind, 6666)
    m = g.random((n_proto, w.H, w.d), dtype=np.float32) < w.p_out
    return np.where(m, np.float32(mult), np.float32(1.0))


def _tokens(w: Workload, seed, kind, proto_kind, first_frame, n_frames, stream, outliers):
    """Prototype (outlier channels scaled when `outliers`) + N(0, sigma^2)
    noise for n_frames frames."""
    hw = w.frame_hw[0] * w.frame_hw[1]
    n = hw * n_frames
    g = _rng(seed, kind, stream, first_frame)
    if w.dist == "ar1":
        mu = _ar1_means(w, seed, proto_kind, first_frame + n_frames)
        pidx, n_patch = _patch_index(w)
        base = mu[first_frame:first_frame + n_frames]                    # [F, P, H, d]
        if outliers:
            base = base * _outlier_scale(w, seed, kind, n_patch)[None]
        base = base[:, pidx].reshape(n, w.H, w.d)
    else:
        protos = _mixture_protos(w, seed, proto_kind)                    # [H, P, d]
        if outliers:
            protos = protos * np.transpose(_outlier_scale(w, seed, kind, w.n_proto), (1, 0, 2))
        pick = _rng(seed, 99, stream, first_frame).integers(0, w.n_proto, size=n)
        base = np.transpose(protos[:, pick], (1, 0, 2))                  # [n, H, d]
    return base + w.sigma * g.standard_normal((n, w.H, w.d), dtype=np.float32)


def chunk_kv(w: Workload, seed: int, chunk: int, kind: int) -> np.ndarray:
    """K (kind=KIND_K) or V (KIND_V) of one chunk: [N, H, d] bf16 values.
    Outlier channels (probability p_out per prototype and channel) carry
    x50 (K) or x300 (V), so max|K| ~ 1e2 and max|V| ~ 1e3."""
    f0 = chunk * w.frames_per_chunk
    x = _tokens(w, seed, kind, kind, f0, w.frames_per_chunk, stream=1, outliers=True)
    return bf16_values(x)


def queries(w: Workload, seed: int, chunk: int) -> np.ndarray:
    """Query tokens of one chunk, drawn like K without outliers
    ([Nq, Hq, d]; Hq == H for these workloads)."""
    f0 = chunk * w.frames_per_chunk
    n_frames = max(1, -(-w.Nq // (w.frame_hw[0] * w.frame_hw[1])))
    x = _tokens(w, seed, KIND_Q, KIND_K, f0, n_frames, stream=3, outliers=False)[: w.Nq]
    if w.Hq != w.H:
        x = np.repeat(x, w.Hq // w.H, axis=1)
    return bf16_values(x)


ACTIVE_FRACTION = 4  # 1 / ACTIVE_FRACTION of the channels carry the planted directions


def active_channels(w: Workload, seed: int) -> np.ndarray:
    """The d / 4 channels of each KV head that the queries are most active on
    ([H, d/4], sorted): the QuantWM write-up's QSAC measures how active the
    history queries are on each channel, i.e. which channels they care about
    more, so the channels are not all alike."""
    g = _rng(seed, KIND_QHIST, 4243)
    n = w.d // ACTIVE_FRACTION
    return np.stack([np.sort(g.permutation(w.d)[:n]) for _ in range(w.H)])


def planted_basis(w: Workload, seed: int) -> np.ndarray:
    """Random orthonormal directions u_1..u_8 per KV head, supported on that
    head's active channels: [H, d, 8]."""
    g = _rng(seed, KIND_QHIST, 4242)
    act = active_channels(w, seed)
    out = np.zeros((w.H, w.d, 8), np.float64)
    for h in range(w.H):
        qm, _ = np.linalg.qr(g.standard_normal((act.shape[1], 8)))
        out[h, act[h]] = qm
    return out


def planted_spectrum(d: int, energy_in_span: float = 0.70, ratio: float = 0.8):
    """Energies lambda_r (geometric, ratio 0.8) of the 8 planted directions,
    summing to energy_in_span * d, and the per-channel variance of the
    isotropic remainder, so that E||q||^2 = d."""
    lam = ratio ** np.arange(8)
    lam = lam / lam.sum() * energy_in_span * d
    sigma2 = (1.0 - energy_in_span) * d / d
    return lam, sigma2


def history_queries(w: Workload, seed: int, n_tokens: int = None, stream: int = 0) -> np.ndarray:
    """Queries q = sum_r a_r u_r + isotropic noise, a_r ~ N(0, lambda_r):
    70% of the expected energy in the 8 planted directions, which live on a
    quarter of the channels, so those channels' mean q_j^2 is
    0.7 * 4 + 0.3 = 3.1 against 0.3 elsewhere.  [n, Hq, d]."""
    if n_tokens is None:
        n_tokens = w.hist_frames * w.frame_hw[0] * w.frame_hw[1]
    U = planted_basis(w, seed)
    lam, sigma2 = planted_spectrum(w.d)
    g = _rng(seed, KIND_QHIST, stream, 1)
    a = g.standard_normal((n_tokens, w.H, 8)) * np.sqrt(lam)[None, None, :]
    q = np.einsum("nhr,hdr->nhd", a, U)
    q += math.sqrt(sigma2) * g.standard_normal((n_tokens, w.H, w.d))
    if w.Hq != w.H:
        q = np.repeat(q, w.Hq // w.H, axis=1)
    return bf16_values(q.astype(np.float32))
