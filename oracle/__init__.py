"""CPU oracle for the QVG / QuantWM KV-cache compression path.

TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg import this module.  It wraps the plain C
implementation in ``qvg_oracle.c`` (built with gcc, no fast-math, no FMA
contraction) through ctypes and shares nothing with the CUDA library.

Every array argument is a numpy array; shapes follow the C functions:
K/V/Q are ``[tokens, heads, head_dim]`` float32 arrays holding bf16 values.
"""
from __future__ import annotations

import ctypes as ct
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qvg_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, -O2, IEEE)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=gnu11", "-O2", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = ct.CDLL(_LIB_PATH)
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ct.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def quant_group(r, bits=2, mode=0):
    """One group: returns (fp16 scale bits, int codes, dequantised fp32)."""
    lib = _load()
    r = _f32(r)
    s = np.zeros(1, np.uint16)
    q = np.zeros(r.size, np.int32)
    rh = np.zeros(r.size, np.float32)
    lib.orc_quant_group(_p(r), ct.c_int(r.size), ct.c_int(bits), ct.c_int(mode),
                        _p(s), _p(q), _p(rh))
    return s[0], q, rh


def quant_group_outlier(r, bits=2, mode=0):
    """One group with the outlier split: returns (fp16 scale bits, int codes,
    dequantised fp32, fp16 outlier bits, outlier index or 0xFF)."""
    lib = _load()
    r = _f32(r)
    s = np.zeros(1, np.uint16)
    q = np.zeros(r.size, np.int32)
    rh = np.zeros(r.size, np.float32)
    ov = np.zeros(1, np.uint16)
    oi = np.zeros(1, np.uint8)
    rc = lib.orc_quant_group_outlier(_p(r), ct.c_int(r.size), ct.c_int(bits), ct.c_int(mode),
                                     _p(s), _p(q), _p(rh), _p(ov), _p(oi))
    if rc != 0:
        raise ValueError("oracle: outlier split needs 2 <= G <= 100")
    return s[0], q, rh, ov[0], int(oi[0])


def pack_row(q, bits):
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.int32)
    out = np.zeros(q.size * bits // 8, np.uint8)
    lib.orc_pack_row(_p(q), ct.c_int(q.size), ct.c_int(bits), _p(out))
    return out


def unpack_row(b, d, bits):
    lib = _load()
    b = np.ascontiguousarray(b, dtype=np.uint8)
    q = np.zeros(d, np.int32)
    lib.orc_unpack_row(_p(b), ct.c_int(d), ct.c_int(bits), _p(q))
    return q


def init_picks(N, C, seed, chunk, head, stage):
    lib = _load()
    idx = np.zeros(C, np.int32)
    lib.orc_init_picks(ct.c_int(N), ct.c_int(C), ct.c_uint64(seed), ct.c_int(chunk),
                       ct.c_int(head), ct.c_int(stage), _p(idx))
    return idx


def assign(g, cent, w=None):
    """g [N,d], cent [C,d] -> ids, best, second, denom (see orc_assign)."""
    lib = _load()
    g, cent = _f32(g), _f32(cent)
    N, d = g.shape
    C = cent.shape[0]
    w = None if w is None else _f32(w)
    ids = np.zeros(N, np.int32)
    b1, b2, den = (np.zeros(N, np.float64) for _ in range(3))
    lib.orc_assign(_p(g), ct.c_int(N), ct.c_int(d), _p(cent), ct.c_int(C), _p(w),
                   _p(ids), _p(b1), _p(b2), _p(den))
    return ids, b1, b2, den


def update(xin, ids, cent):
    """Returns (new bf16-valued centroids, fp32 means, member counts)."""
    lib = _load()
    xin = _f32(xin)
    N, d = xin.shape
    cent = _f32(cent).copy()
    C = cent.shape[0]
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    mean = np.zeros_like(cent)
    cnt = np.zeros(C, np.int32)
    lib.orc_update(_p(xin), ct.c_int(N), ct.c_int(d), _p(ids), ct.c_int(C),
                   _p(cent), _p(mean), _p(cnt))
    return cent, mean, cnt


def inertia(g, cent, ids, w=None):
    lib = _load()
    lib.orc_inertia.restype = ct.c_double
    g, cent = _f32(g), _f32(cent)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = None if w is None else _f32(w)
    return lib.orc_inertia(_p(g), ct.c_int(g.shape[0]), ct.c_int(g.shape[1]),
                           _p(cent), _p(ids), _p(w))


def psac_encode_token(E, U):
    lib = _load()
    E, U = _f32(E), _f32(U)
    d, r = U.shape
    p = np.zeros(r, np.int8)
    s = np.zeros(1, np.uint16)
    lib.orc_psac_encode_token(_p(E), _p(U), ct.c_int(d), ct.c_int(r), _p(p), _p(s))
    return p, s[0]


def compress_chunk(x, C, L, bits, group, iters, mode=0, seed=0, chunk=0,
                   qsac_w=None, psac_U=None, cent_in=None, outlier=False, nthreads=1):
    """Compress one chunk x [N,H,d].  Returns a dict with codes [L,H,N,nb],
    scales (fp16 bits) [L,H,N,d/G], ids [L,H,N], cent (bf16 bits) [L,H,C,d],
    means [L,H,C,d], psac_p [H,N,r], psac_s [H,N], xhat [N,H,d] and
    resid [N,H,d] (the residual after the last stage); with outlier=True
    also outl_val (fp16 bits) and outl_idx [L,H,N,d/G]."""
    lib = _load()
    x = _f32(x)
    N, H, d = x.shape
    r = 0 if psac_U is None else psac_U.shape[-1]
    Cs = max(C, 1)
    out = dict(
        codes=np.zeros((L, H, N, d * bits // 8), np.uint8),
        scales=np.zeros((L, H, N, d // group), np.uint16),
        ids=np.zeros((L, H, N), np.uint8),
        cent=np.zeros((L, H, Cs, d), np.uint16),
        means=np.zeros((L, H, Cs, d), np.float32),
        psac_p=np.zeros((H, N, max(r, 1)), np.int8),
        psac_s=np.zeros((H, N), np.uint16),
        xhat=np.zeros((N, H, d), np.float32),
        resid=np.zeros((N, H, d), np.float32),
    )
    if outlier:
        out["outl_val"] = np.zeros((L, H, N, d // group), np.uint16)
        out["outl_idx"] = np.zeros((L, H, N, d // group), np.uint8)
    qsac_w = None if qsac_w is None else _f32(qsac_w)
    psac_U = None if psac_U is None else _f32(psac_U)
    cent_in = None if cent_in is None else _f32(cent_in)
    rc = lib.orc_compress_chunk(
        _p(x), ct.c_int(N), ct.c_int(H), ct.c_int(d), ct.c_int(C), ct.c_int(L),
        ct.c_int(bits), ct.c_int(group), ct.c_int(iters), ct.c_int(mode),
        ct.c_uint64(seed), ct.c_int(chunk), _p(qsac_w), _p(psac_U), ct.c_int(r),
        _p(cent_in), _p(out["codes"]), _p(out["scales"]), _p(out["ids"]),
        _p(out["cent"]), _p(out["means"]), _p(out["psac_p"]), _p(out["psac_s"]),
        _p(out["xhat"]), _p(out["resid"]), _p(out.get("outl_val")), _p(out.get("outl_idx")),
        ct.c_int(nthreads))
    if rc != 0:
        raise ValueError("oracle: unsupported compression arguments")
    if C == 0:
        out["cent"] = out["cent"][:, :, :0]
        out["means"] = out["means"][:, :, :0]
    if r == 0:
        out["psac_p"] = out["psac_p"][:, :, :0]
    return out


def decompress(codes, scales, ids, cent, C, bits, group, psac_p=None,
               psac_s=None, psac_U=None, outl_val=None, outl_idx=None):
    """Rebuild [N,H,d] fp32 from the stored layout (see orc_decompress)."""
    lib = _load()
    L, H, N, _ = codes.shape
    d = scales.shape[-1] * group
    out = np.zeros((N, H, d), np.float32)
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint16)
    ids = np.ascontiguousarray(ids, np.uint8)
    cent = np.ascontiguousarray(cent, np.uint16) if C > 0 else np.zeros(1, np.uint16)
    r = 0
    if outl_val is not None:
        outl_val = np.ascontiguousarray(outl_val, np.uint16)
        outl_idx = np.ascontiguousarray(outl_idx, np.uint8)
    if psac_p is not None:
        psac_p = np.ascontiguousarray(psac_p, np.int8)
        psac_s = np.ascontiguousarray(psac_s, np.uint16)
        psac_U = _f32(psac_U)
        r = psac_U.shape[-1]
    lib.orc_decompress(_p(codes), _p(scales), _p(ids), _p(cent), ct.c_int(N),
                       ct.c_int(H), ct.c_int(d), ct.c_int(C), ct.c_int(L),
                       ct.c_int(bits), ct.c_int(group), _p(psac_p), _p(psac_s),
                       _p(psac_U), ct.c_int(r), _p(outl_val), _p(outl_idx), _p(out))
    return out


def attention(q, k, v, scale=0.0, nthreads=1):
    """q [Nq,Hq,d], k/v [Nk,H,d] -> out fp64 [Nq,Hq,d], lse [Hq,Nq], argmax [Hq,Nq]."""
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    Nq, Hq, d = q.shape
    Nk, H, _ = k.shape
    out = np.zeros((Nq, Hq, d), np.float64)
    lse = np.zeros((Hq, Nq), np.float64)
    am = np.zeros((Hq, Nq), np.int32)
    rc = lib.orc_attention(_p(q), ct.c_int(Nq), ct.c_int(Hq), _p(k), _p(v),
                           ct.c_int(Nk), ct.c_int(H), ct.c_int(d),
                           ct.c_double(scale), _p(out), _p(lse), _p(am),
                           ct.c_int(nthreads))
    if rc != 0:
        raise ValueError("oracle: bad attention arguments")
    return out, lse, am


def attention_ar(q, k_hat, v_hat, k_cur, v_cur, cache_slots, n_slots, scale=0.0, nthreads=1):
    """Attention of one autoregressive step (Quant VideoGen notes, research
    background: each new chunk attends to the cached K/V of every earlier
    chunk; reading: no mask inside the chunk).  The keys are the cached
    tokens followed by the chunk's own tokens, in one softmax:
        O = softmax(scale q [k_hat; k_cur]^T) [v_hat; v_cur].
    k_hat/v_hat [Nc,H,d] hold the reconstructed cache tokens, whose slot
    numbers are cache_slots [Nc]; current-chunk token j is slot n_slots + j.
    Returns out fp64 [Nq,Hq,d], lse [Hq,Nq] and the top-1 slot [Hq,Nq]."""
    k = np.concatenate([np.asarray(k_hat, np.float32), np.asarray(k_cur, np.float32)], 0)
    v = np.concatenate([np.asarray(v_hat, np.float32), np.asarray(v_cur, np.float32)], 0)
    out, lse, am = attention(q, k, v, scale, nthreads)
    slot_of = np.concatenate([np.asarray(cache_slots, np.int64),
                              n_slots + np.arange(len(k_cur), dtype=np.int64)])
    return out, lse, slot_of[am].astype(np.int32)


def top1(q, k, nthreads=1):
    lib = _load()
    q, k = _f32(q), _f32(k)
    Nq, Hq, d = q.shape
    Nk, H, _ = k.shape
    am = np.zeros((Hq, Nq), np.int32)
    lib.orc_top1(_p(q), ct.c_int(Nq), ct.c_int(Hq), _p(k), ct.c_int(Nk), ct.c_int(H),
                 ct.c_int(d), _p(am), ct.c_int(nthreads))
    return am


def shift_rate(q, k_ref, k_hat, nthreads=1):
    """Top-1 attention-token shift rate (QuantWM write-up, results and the
    ablation: the share of (query, query head) pairs whose highest-logit
    history token differs between the reference cache and the reconstructed
    one).  q [Nq,Hq,d], k_ref and k_hat [Nk,H,d]; ties go to the lowest
    token on both sides."""
    a = top1(q, k_ref, nthreads)
    b = top1(q, k_hat, nthreads)
    return float((a != b).mean())


def query_stats(q, H, M=None, count=0):
    """Accumulate M [H,d,d] (fp64) += sum q q^T; returns (M, count)."""
    lib = _load()
    q = _f32(q)
    n, Hq, d = q.shape
    M = np.zeros((H, d, d), np.float64) if M is None else np.ascontiguousarray(M, np.float64).copy()
    c = np.array([count], np.int64)
    lib.orc_query_stats(_p(q), ct.c_int(n), ct.c_int(Hq), ct.c_int(H), ct.c_int(d),
                        _p(M), _p(c))
    return M, int(c[0])


def jacobi(M, tol=1e-12, max_sweeps=100):
    lib = _load()
    M = np.ascontiguousarray(M, np.float64)
    d = M.shape[0]
    ev = np.zeros(d, np.float64)
    vec = np.zeros((d, d), np.float64)
    sweeps = lib.orc_jacobi(_p(M), ct.c_int(d), ct.c_double(tol), ct.c_int(max_sweeps),
                            _p(ev), _p(vec))
    return ev, vec, sweeps


def psac_basis(M, count, r=8):
    lib = _load()
    M = np.ascontiguousarray(M, np.float64)
    H, d, _ = M.shape
    U = np.zeros((H, d, r), np.float64)
    eig = np.zeros((H, r), np.float64)
    frac = np.zeros(H, np.float64)
    rc = lib.orc_psac_basis(_p(M), ct.c_int64(count), ct.c_int(H), ct.c_int(d),
                            ct.c_int(r), _p(U), _p(eig), _p(frac))
    if rc != 0:
        raise ValueError("oracle: bad psac_basis arguments")
    return U, eig, frac


def f16_bits_to_f32(b):
    return np.asarray(b, np.uint16).view(np.float16).astype(np.float32)


def bf16_bits_to_f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)
