"""Test-side helpers: copy a GPU cache to numpy, run the oracle on the same
bytes, and the near-tie rule for cluster assignments."""
import numpy as np
import torch

import oracle
import video_diffusion_kv_gb300 as qvg

# Tolerances (stated with the checks that use them):
NEAR_TIE = 1e-5        # (s_gpu - s_best) / (||x||_w^2 + ||c_best||_w^2)
NEAR_TIE_RATE = 1e-4   # near-tie mismatches allowed: < 0.01 % of assignments
ATTN_TOL = 2e-3        # max|dO| / max|O_oracle| per head
RECON_TOL = 1e-3       # max|dX| / max|X_oracle| per (chunk, head)


def to_dev(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev, torch.bfloat16)


def host_cache(c: qvg.CompressedKV):
    """numpy copies of a cache's buffers (slot layout) and chunk tables."""
    p = c.params
    L, H, cap, d = p.L, c.H, c.capacity_tokens, c.d
    out = dict(
        codes=c.view("codes", torch.uint8, (L, H, cap, d * p.bits // 8)).cpu().numpy(),
        scales=c.view("scales", torch.int16, (L, H, cap, d // p.group)).cpu().numpy().view(np.uint16),
        start=c.view("chunk_start", torch.int32, (c.max_chunks,)).cpu().numpy(),
        length=c.view("chunk_len", torch.int32, (c.max_chunks,)).cpu().numpy(),
    )
    if p.C > 0:
        out["ids"] = c.view("ids", torch.uint8, (L, H, cap)).cpu().numpy()
        out["cent"] = c.view("cent", torch.int16, (L, H, c.max_chunks, p.C, d)).cpu().numpy().view(np.uint16)
    if p.flags & qvg.QVG_PSAC:
        out["psac_p"] = c.view("psac_p", torch.int8, (H, cap, 8)).cpu().numpy()
        out["psac_s"] = c.view("psac_s", torch.int16, (H, cap)).cpu().numpy().view(np.uint16)
        out["psac_basis"] = c.view("psac_basis", torch.float32, (c.max_chunks, H, d, 8)).cpu().numpy()
    if p.flags & qvg.QVG_OUTLIER:
        ng = d // p.group
        out["outl_val"] = c.view("outl_val", torch.int16, (L, H, cap, ng)).cpu().numpy().view(np.uint16)
        out["outl_idx"] = c.view("outl_idx", torch.uint8, (L, H, cap, ng)).cpu().numpy()
    if p.anchor_every > 0:
        out["anchor"] = c.view("anchor", torch.int16, (-1, H, d)).cpu().numpy().view(np.uint16)
        out["chunk_anchor"] = c.view("chunk_anchor", torch.int32, (c.max_chunks,)).cpu().numpy()
    return out


def chunk_slice(hc, k):
    s = int(hc["start"][k])
    return slice(s, s + int(hc["length"][k]))


def chunk_arrays(hc, p, k):
    """Oracle-layout arrays of chunk k: codes [L,H,N,nb], scales, ids, cent [L,H,C,d]."""
    sl = chunk_slice(hc, k)
    ids = hc["ids"][:, :, sl] if p.C > 0 else np.zeros(hc["codes"][:, :, sl].shape[:3], np.uint8)
    cent = hc["cent"][:, :, k] if p.C > 0 else np.zeros((p.L, hc["codes"].shape[1], 0, 0), np.uint16)
    return hc["codes"][:, :, sl], hc["scales"][:, :, sl], ids, cent


def oracle_rebuild(hc, p, k):
    """Oracle reconstruction [N,H,d] of chunk k from the GPU's stored bytes
    (an anchor chunk: its stored bf16 rows, as they are)."""
    if "chunk_anchor" in hc and hc["chunk_anchor"][k] >= 0:
        r0, n = int(hc["chunk_anchor"][k]), int(hc["length"][k])
        return oracle.bf16_bits_to_f32(hc["anchor"][r0:r0 + n])
    codes, scales, ids, cent = chunk_arrays(hc, p, k)
    kw = {}
    sl = chunk_slice(hc, k)
    if "psac_p" in hc:
        kw = dict(psac_p=hc["psac_p"][:, sl], psac_s=hc["psac_s"][:, sl], psac_U=hc["psac_basis"][k])
    if "outl_val" in hc:
        kw.update(outl_val=hc["outl_val"][:, :, sl], outl_idx=hc["outl_idx"][:, :, sl])
    return oracle.decompress(codes, scales, ids, cent, p.C, p.bits, p.group, **kw)


def stage_abs_rebuild(hc, p, k):
    """sum_l |K_hat_l| [N,H,d] of chunk k, stage by stage (the magnitudes the
    attention kernel rounds to fp16, one stage per buffer fill); an anchor
    chunk's rows, or a one-stage chunk, as |K_hat|."""
    if p.L == 1 or ("chunk_anchor" in hc and hc["chunk_anchor"][k] >= 0):
        return np.abs(oracle_rebuild(hc, p, k))
    codes, scales, ids, cent = chunk_arrays(hc, p, k)
    sl = chunk_slice(hc, k)
    out = 0.0
    for l in range(p.L):
        kw = {}
        if "outl_val" in hc:
            kw = dict(outl_val=hc["outl_val"][l:l + 1, :, sl], outl_idx=hc["outl_idx"][l:l + 1, :, sl])
        out = out + np.abs(oracle.decompress(codes[l:l + 1], scales[l:l + 1], ids[l:l + 1], cent[l:l + 1],
                                             p.C, p.bits, p.group, **kw))
    return out


# Log-sum-exp.  The kernel's operands are fp16 (reading R21: unit roundoff
# 2^-11; Q's bf16 values are exact in fp16, each stage of K_hat is rounded
# once), so logit j of a row moves by at most
#   scale * sum_c |q_c| sum_l |K_hat_l,jc| * 2^-11,
# and the row sum of the fp16-rounded weights by a factor within 1 +- 2^-11;
# the natural-log LSE, 1-Lipschitz in the logits' max norm, then moves by at
# most the largest logit bound + 2^-11.  The checks allow the larger of that
# bound and 2e-3.
LSE_TOL = 2e-3


def lse_tolerance(q, k_abs, grp, scale=None):
    """Per-(query head, query) LSE tolerance [Hq, Nq] for queries q [Nq,Hq,d]
    over keys with stage magnitudes k_abs [Nk,H,d] (query head hq reads key
    head hq // grp)."""
    q = np.abs(np.asarray(q, np.float64))
    Nq, Hq, d = q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    out = np.empty((Hq, Nq))
    for hq in range(Hq):
        kh = np.asarray(k_abs[:, hq // grp], np.float64)
        b = (q[:, hq] @ kh.T).max(axis=1) if len(kh) else np.zeros(Nq)
        out[hq] = scale * b * 2.0 ** -11 + 2.0 ** -11
    return np.maximum(out, LSE_TOL)


def assignment_mismatches(g, cent_bf16_bits, ids_gpu, w=None):
    """Compare GPU ids for one (head, stage) with the oracle's argmin over the
    same centroids.  Returns (number of mismatches, number outside near ties)."""
    cent = oracle.bf16_bits_to_f32(cent_bf16_bits)
    ids_o, best, _, denom = oracle.assign(g, cent, w)
    bad = np.nonzero(ids_o != ids_gpu)[0]
    if len(bad) == 0:
        return 0, 0
    ww = np.ones(g.shape[1]) if w is None else w.astype(np.float64)
    diff = g[bad].astype(np.float64) - cent[ids_gpu[bad]].astype(np.float64)
    s_gpu = (ww * diff * diff).sum(1)
    gap = (s_gpu - best[bad]) / denom[bad]
    return len(bad), int((gap >= NEAR_TIE).sum())


def bf16_ulp_diff(a_bits, b_bits):
    """|a - b| in bf16 ulps (same-sign monotone integer distance)."""
    def key(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, 0x8000 - u, u)
    return np.abs(key(a_bits) - key(b_bits))
