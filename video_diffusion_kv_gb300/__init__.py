"""Python binding of libqvg: compressed video KV cache (QVG / QVG-Pro with
QuantWM QSAC / PSAC) on one GB300.

Argument marshalling only: every step of compression, reconstruction,
attention and the QuantWM statistics runs in the CUDA kernels of
``libqvg.so``; PyTorch provides device memory and streams.  There is no
fallback: if the library is missing or no CUDA device is present, the calls
raise.

Names follow the C ABI in ``include/qvg.h``.
"""
from __future__ import annotations

import ctypes as ct
import dataclasses
import math
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqvg.so")

QVG_OK, QVG_ERR_INVALID_ARG, QVG_ERR_UNSUPPORTED, QVG_ERR_CUDA = 0, 1, 2, 3
QVG_ERR_TIMEOUT, QVG_ERR_WORKSPACE, QVG_ERR_CAPACITY = 4, 5, 6
QVG_QSAC, QVG_PSAC, QVG_GIVEN_CENTROIDS, QVG_OUTLIER, QVG_KEEP_MEANS = 1, 2, 4, 8, 16
QVG_TILE = 128
QVG_PSAC_RANK = 8
QVG_CACHE_NBUF = 14
QVG_OUT_F32, QVG_OUT_BF16 = 0, 1
QVG_OP_COMPRESS, QVG_OP_ATTENTION, QVG_OP_PSAC_BASIS = 0, 1, 2

EXPORTED = (
    "qvg_status_string", "qvg_cache_bytes", "qvg_workspace_size", "qvg_compress_chunk",
    "qvg_decompress", "qvg_attention", "quantwm_query_stats", "quantwm_psac_basis",
    "qvg_get_status", "qvg_last_cuda_error", "qvg_compress_chunk_noalloc", "qvg_attention_ar",
    "qvg_debug_set_wait",
)
NOALLOC_SCRATCH_BYTES = 32 << 20

BUFFER_NAMES = ("codes", "scales", "ids", "cent", "chunk_start", "chunk_len", "tile_chunk",
                "psac_p", "psac_s", "psac_basis", "outl_val", "outl_idx", "anchor", "chunk_anchor")


class QvgError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, status_string(status), status))


class _Params(ct.Structure):
    _fields_ = [("C", ct.c_int32), ("L", ct.c_int32), ("bits", ct.c_int32),
                ("group", ct.c_int32), ("iters", ct.c_int32), ("scale_mode", ct.c_int32),
                ("flags", ct.c_int32), ("anchor_every", ct.c_int32), ("seed", ct.c_uint64)]


class _Cache(ct.Structure):
    _fields_ = [("H", ct.c_int32), ("d", ct.c_int32), ("capacity_tokens", ct.c_int32),
                ("max_chunks", ct.c_int32), ("n_chunks", ct.c_int32), ("n_tokens", ct.c_int32),
                ("codes", ct.c_void_p), ("scales", ct.c_void_p), ("ids", ct.c_void_p),
                ("cent", ct.c_void_p), ("chunk_start", ct.c_void_p), ("chunk_len", ct.c_void_p),
                ("tile_chunk", ct.c_void_p), ("psac_p", ct.c_void_p), ("psac_s", ct.c_void_p),
                ("psac_basis", ct.c_void_p), ("outl_val", ct.c_void_p), ("outl_idx", ct.c_void_p),
                ("anchor", ct.c_void_p), ("chunk_anchor", ct.c_void_p)]


_lib = None


def lib():
    """Load libqvg.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libqvg.so is not built; run __graft_entry__.build() "
                               "or python video_diffusion_kv_gb300/build.py")
        L = ct.CDLL(LIB_PATH)
        L.qvg_status_string.restype = ct.c_char_p
        L.qvg_status_string.argtypes = [ct.c_int]
        vp, i32, sz = ct.c_void_p, ct.c_int32, ct.c_size_t
        L.qvg_cache_bytes.argtypes = [vp, i32, i32, i32, i32, vp]
        L.qvg_workspace_size.argtypes = [vp, i32, i32, i32, i32, i32, vp]
        L.qvg_compress_chunk.argtypes = [vp, vp, i32, vp, vp, vp, vp, sz, vp]
        L.qvg_compress_chunk_noalloc.argtypes = [vp, vp, i32, vp, vp, vp, vp]
        L.qvg_decompress.argtypes = [vp, vp, i32, i32, vp, i32, vp]
        L.qvg_attention.argtypes = [vp, vp, i32, i32, vp, vp, ct.c_float, vp, i32, vp, vp, vp, sz, vp]
        L.qvg_attention_ar.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, i32, ct.c_float, vp, i32, vp, vp, vp,
                                       sz, vp]
        L.quantwm_query_stats.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp]
        L.quantwm_psac_basis.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp]
        L.qvg_get_status.argtypes = [vp]
        L.qvg_debug_set_wait.argtypes = [ct.c_uint64, i32]
        L.qvg_last_cuda_error.restype = ct.c_char_p
        L.qvg_last_cuda_error.argtypes = []
        _lib = L
    return _lib


def status_string(s):
    return lib().qvg_status_string(int(s)).decode()


def _check(s, where):
    if s != QVG_OK:
        if s == QVG_ERR_CUDA:
            where = "%s [%s]" % (where, lib().qvg_last_cuda_error().decode())
        raise QvgError(s, where)


@dataclasses.dataclass
class Params:
    """Method parameters (see qvg_params in include/qvg.h)."""
    C: int = 256
    L: int = 1
    bits: int = 2
    group: int = 64
    iters: int = 8
    scale_mode: int = 0
    flags: int = 0
    seed: int = 0
    anchor_every: int = 0

    def c(self):
        return _Params(self.C, self.L, self.bits, self.group, self.iters, self.scale_mode,
                       self.flags, self.anchor_every, self.seed)


def _ptr(t):
    return None if t is None else ct.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ct.c_void_p(s.cuda_stream)


def kv_bytes_uncompressed(layers, kv_heads, head_dim, tokens, bytes_per_elt=2):
    """KV cache size before compression: 2 (K and V) x layers x KV heads x
    head_dim x tokens x bytes per element ("The 2-bit quantisation trap",
    section 1)."""
    return 2 * layers * kv_heads * head_dim * tokens * bytes_per_elt


def cache_bytes(params: Params, H, d, capacity_tokens, max_chunks):
    """Per-buffer byte sizes of one compressed tensor (dict)."""
    out = (ct.c_size_t * QVG_CACHE_NBUF)()
    p = params.c()
    _check(lib().qvg_cache_bytes(ct.byref(p), H, d, capacity_tokens, max_chunks, out), "qvg_cache_bytes")
    return dict(zip(BUFFER_NAMES, [int(v) for v in out]))


def workspace_size(params: Params, op, n, H, d, Hq=None):
    b = ct.c_size_t(0)
    p = params.c()
    _check(lib().qvg_workspace_size(ct.byref(p), op, n, H, d, Hq or H, ct.byref(b)), "qvg_workspace_size")
    return int(b.value)


class CompressedKV:
    """One compressed tensor (K or V) of one layer: device buffers allocated
    with torch at the sizes libqvg reports, plus the host-side counters."""

    def __init__(self, params: Params, H, d, capacity_tokens, max_chunks, device="cuda"):
        import torch
        capacity_tokens = -(-capacity_tokens // QVG_TILE) * QVG_TILE
        self.params = dataclasses.replace(params)
        self.H, self.d = H, d
        self.capacity_tokens, self.max_chunks = capacity_tokens, max_chunks
        sizes = cache_bytes(params, H, d, capacity_tokens, max_chunks)
        self.sizes = sizes
        self.buffers = {}
        for name in BUFFER_NAMES:
            n = sizes[name]
            self.buffers[name] = torch.zeros(max(n, 0), dtype=torch.uint8, device=device) if n else None
        self.n_chunks = 0
        self.n_tokens = 0

    @property
    def nbytes(self):
        return sum(self.sizes.values())

    def c(self):
        b = self.buffers
        return _Cache(self.H, self.d, self.capacity_tokens, self.max_chunks, self.n_chunks,
                      self.n_tokens, *[_ptr(b[n]) for n in BUFFER_NAMES])

    def reset(self, n_chunks=0, n_tokens=0):
        self.n_chunks, self.n_tokens = n_chunks, n_tokens

    def view(self, name, dtype, shape):
        """Typed view of one buffer (for inspection and checkpointing)."""
        return self.buffers[name].view(dtype).view(*shape)

    def centroid_slot(self, chunk):
        """bf16 [L, H, C, d] view of one chunk's centroids."""
        import torch
        p = self.params
        cent = self.view("cent", torch.bfloat16, (p.L, self.H, self.max_chunks, p.C, self.d))
        return cent[:, :, chunk]


def compress_chunk(params: Params, x, cache: CompressedKV, qsac_w=None, psac_basis=None,
                   workspace=None, stream=None):
    """Append one chunk x (bf16 [N, H, d], contiguous, on the GPU) to cache.
    Returns the first token slot of the chunk.  With QVG_KEEP_MEANS in
    params.flags, pass a workspace and read the fp32 means from it with
    kept_means()."""
    import torch
    assert x.dtype == torch.bfloat16 and x.is_contiguous() and x.dim() == 3
    N = x.shape[0]
    need = workspace_size(params, QVG_OP_COMPRESS, N, cache.H, cache.d)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    c = cache.c()
    p = params.c()
    slot0 = cache.n_tokens
    s = lib().qvg_compress_chunk(ct.byref(p), _ptr(x), N, _ptr(qsac_w), _ptr(psac_basis), ct.byref(c),
                                 _ptr(workspace), workspace.numel(), _stream(stream))
    _check(s, "qvg_compress_chunk")
    cache.n_chunks, cache.n_tokens = c.n_chunks, c.n_tokens
    return slot0


def kept_means(params: Params, workspace, H, d):
    """fp32 [L, H, C, d] view of the centroid means a QVG_KEEP_MEANS
    compression left at the start of its workspace."""
    import torch
    n = params.L * H * params.C * d
    return workspace[:4 * n].view(torch.float32).view(params.L, H, params.C, d)


def compress_chunk_noalloc(params: Params, x, cache: CompressedKV, qsac_w=None, psac_basis=None,
                           stream=None):
    """compress_chunk without a workspace argument: for callers that cannot
    allocate device memory, the library uses its own fixed 32 MiB device
    scratch (see qvg_compress_chunk_noalloc in include/qvg.h; calls that
    overlap on the GPU race on it).  Returns the first token slot."""
    import torch
    assert x.dtype == torch.bfloat16 and x.is_contiguous() and x.dim() == 3
    c = cache.c()
    p = params.c()
    slot0 = cache.n_tokens
    s = lib().qvg_compress_chunk_noalloc(ct.byref(p), _ptr(x), x.shape[0], _ptr(qsac_w), _ptr(psac_basis),
                                         ct.byref(c), _stream(stream))
    _check(s, "qvg_compress_chunk_noalloc")
    cache.n_chunks, cache.n_tokens = c.n_chunks, c.n_tokens
    return slot0


def decompress(params: Params, cache: CompressedKV, tok0, ntok, out_dtype=QVG_OUT_F32, out=None,
               stream=None):
    import torch
    dt = torch.float32 if out_dtype == QVG_OUT_F32 else torch.bfloat16
    if out is None:
        out = torch.empty((ntok, cache.H, cache.d), dtype=dt, device=cache.buffers["codes"].device)
    c = cache.c()
    p = params.c()
    _check(lib().qvg_decompress(ct.byref(p), ct.byref(c), tok0, ntok, _ptr(out), out_dtype, _stream(stream)),
           "qvg_decompress")
    return out


def attention(params: Params, q, kc: CompressedKV, vc: CompressedKV, scale=0.0,
              out_dtype=QVG_OUT_F32, want_lse=False, want_top1=False, out=None, workspace=None,
              stream=None, allow_split=True):
    """O = softmax(scale Q K_hat^T) V_hat over every cached token.
    q: bf16 [Nq, Hq, d].  Returns (out, lse or None, top1 or None).
    allow_split=False passes no workspace, so the cache is never split over
    extra CTAs."""
    import torch
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and q.dim() == 3
    Nq, Hq, d = q.shape
    dt = torch.float32 if out_dtype == QVG_OUT_F32 else torch.bfloat16
    if out is None:
        out = torch.empty((Nq, Hq, d), dtype=dt, device=q.device)
    lse = torch.empty((Hq, Nq), dtype=torch.float32, device=q.device) if want_lse else None
    top1 = torch.empty((Hq, Nq), dtype=torch.int32, device=q.device) if want_top1 else None
    need = workspace_size(params, QVG_OP_ATTENTION, Nq, kc.H, d, Hq) if allow_split else 0
    if not allow_split:
        workspace = None
    elif need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    k, v = kc.c(), vc.c()
    p = params.c()
    s = lib().qvg_attention(ct.byref(p), _ptr(q), Nq, Hq, ct.byref(k), ct.byref(v), float(scale),
                            _ptr(out), out_dtype, _ptr(lse), _ptr(top1), _ptr(workspace),
                            0 if workspace is None else workspace.numel(), _stream(stream))
    _check(s, "qvg_attention")
    return out, lse, top1


def attention_ar(params: Params, q, kc: CompressedKV, vc: CompressedKV, k_cur, v_cur, scale=0.0,
                 out_dtype=QVG_OUT_F32, want_lse=False, want_top1=False, out=None, workspace=None,
                 stream=None):
    """One autoregressive step: softmax(scale Q [K_hat; K_cur]^T) [V_hat; V_cur]
    over the cached tokens and the current chunk's raw bf16 rows.
    q: bf16 [Nq, Hq, d]; k_cur, v_cur: bf16 [n_cur, H, d].  Returns
    (out, lse or None, top1 or None); current-chunk token j is slot
    kc.n_tokens + j in top1."""
    import torch
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and q.dim() == 3
    for x in (k_cur, v_cur):
        assert x.dtype == torch.bfloat16 and x.is_contiguous() and x.dim() == 3
    assert k_cur.shape == v_cur.shape and k_cur.shape[1:] == (kc.H, kc.d)
    Nq, Hq, d = q.shape
    n_cur = k_cur.shape[0]
    dt = torch.float32 if out_dtype == QVG_OUT_F32 else torch.bfloat16
    if out is None:
        out = torch.empty((Nq, Hq, d), dtype=dt, device=q.device)
    lse = torch.empty((Hq, Nq), dtype=torch.float32, device=q.device) if want_lse else None
    top1 = torch.empty((Hq, Nq), dtype=torch.int32, device=q.device) if want_top1 else None
    need = workspace_size(params, QVG_OP_ATTENTION, Nq, kc.H, d, Hq)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    k, v = kc.c(), vc.c()
    p = params.c()
    s = lib().qvg_attention_ar(ct.byref(p), _ptr(q), Nq, Hq, ct.byref(k), ct.byref(v), _ptr(k_cur), _ptr(v_cur),
                               n_cur, float(scale), _ptr(out), out_dtype, _ptr(lse), _ptr(top1), _ptr(workspace),
                               0 if workspace is None else workspace.numel(), _stream(stream))
    _check(s, "qvg_attention_ar")
    return out, lse, top1


def query_stats(q, H, M=None, w=None, count=None, accumulate=False, stream=None):
    """History-query statistics: returns (M fp32 [H,d,d], w fp32 [H,d], count int64 [1])."""
    import torch
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and q.dim() == 3
    n, Hq, d = q.shape
    dev = q.device
    if M is None:
        M = torch.zeros((H, d, d), dtype=torch.float32, device=dev)
    if w is None:
        w = torch.zeros((H, d), dtype=torch.float32, device=dev)
    if count is None:
        count = torch.zeros(1, dtype=torch.int64, device=dev)
    _check(lib().quantwm_query_stats(_ptr(q), n, Hq, H, d, int(accumulate), _ptr(M), _ptr(w), _ptr(count),
                                     _stream(stream)), "quantwm_query_stats")
    return M, w, count


def psac_basis(M, count, rank=QVG_PSAC_RANK, stream=None):
    """Returns (U fp32 [H,d,rank], eigvals fp32 [H,rank], energy_frac fp32 [H])."""
    import torch
    H, d, _ = M.shape
    U = torch.empty((H, d, rank), dtype=torch.float32, device=M.device)
    eig = torch.empty((H, rank), dtype=torch.float32, device=M.device)
    frac = torch.empty((H,), dtype=torch.float32, device=M.device)
    _check(lib().quantwm_psac_basis(_ptr(M), _ptr(count), H, d, rank, _ptr(U), _ptr(eig), _ptr(frac),
                                    _stream(stream)), "quantwm_psac_basis")
    return U, eig, frac


def get_status(stream=None):
    """Synchronise with `stream` (default: the whole device) and return (and
    clear) the device-side error status."""
    return lib().qvg_get_status(None if stream is None else ct.c_void_p(stream.cuda_stream))


def debug_set_wait(limit_ns=0, inject=False):
    """Bound of the device-side waits of the kernels this host thread launches
    next (0: the default 2 s) and the failure-path test hook (see
    qvg_debug_set_wait in include/qvg.h)."""
    _check(lib().qvg_debug_set_wait(int(limit_ns), int(bool(inject))), "qvg_debug_set_wait")


def compression_ratio(params: Params, H, d, tokens_per_chunk, n_chunks, with_psac=False):
    """bf16 bytes / compressed bytes for n_chunks chunks, counting codes,
    fp16 scales, 1-byte ids, bf16 centroids, the outlier side list (fp16
    value + 1-byte channel per group and stage, with QVG_OUTLIER),
    (optionally) the PSAC data, and anchor chunks (anchor_every > 0) at
    their bf16 size, at the stored sizes (padding slots, and the slots an
    anchor chunk reserves in the compressed buffers, excluded)."""
    n_anchor = -(-n_chunks // params.anchor_every) if params.anchor_every > 0 else 0
    n_comp = n_chunks - n_anchor
    N = tokens_per_chunk * n_comp
    side = 3 * d / params.group if params.flags & QVG_OUTLIER else 0
    per_tok = params.L * (d * params.bits / 8 + 2 * d / params.group + (1 if params.C > 0 else 0) + side)
    if with_psac:
        per_tok += QVG_PSAC_RANK + 2
    comp = H * N * per_tok + params.L * H * n_comp * params.C * d * 2
    if with_psac:
        comp += n_comp * H * d * QVG_PSAC_RANK * 4
    comp += n_anchor * tokens_per_chunk * H * d * 2
    return (H * tokens_per_chunk * n_chunks * d * 2) / comp
