"""CPU-side checks of the C ABI: the library loads, exports every function
include/qvg.h declares, sizes buffers by the stated layout, and rejects bad
arguments on the host before anything is launched (no GPU needed)."""
import ctypes as ct
import os
import re
import subprocess

import pytest

import video_diffusion_kv_gb300 as qvg
from video_diffusion_kv_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qvg.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "qvg.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b((?:qvg|quantwm)_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert set(names) == set(qvg.EXPORTED)
    nm = subprocess.run(["nm", "-D", "--defined-only", qvg.LIB_PATH], capture_output=True, text=True).stdout
    for n in names:
        assert re.search(r"\bT %s$" % n, nm, re.M), n
        assert hasattr(lib, n)


def test_status_strings(lib):
    for s in range(7):
        assert qvg.status_string(s)
    assert qvg.status_string(99) == "unknown status"


def test_cache_bytes_layout(lib):
    p = qvg.Params(C=256, L=1, bits=2, group=64)
    s = qvg.cache_bytes(p, H=16, d=128, capacity_tokens=37888, max_chunks=8)
    assert s["codes"] == 16 * 37888 * 32
    assert s["scales"] == 16 * 37888 * 2 * 2
    assert s["ids"] == 16 * 37888
    assert s["cent"] == 16 * 8 * 256 * 128 * 2
    assert s["chunk_start"] == s["chunk_len"] == 32
    assert s["tile_chunk"] == 4 * 37888 // 128
    assert s["psac_p"] == s["psac_s"] == s["psac_basis"] == 0
    p2 = qvg.Params(C=16, L=3, bits=4, group=32, flags=qvg.QVG_PSAC)
    s2 = qvg.cache_bytes(p2, H=2, d=64, capacity_tokens=1024, max_chunks=4)
    assert s2["codes"] == 3 * 2 * 1024 * 32
    assert s2["scales"] == 3 * 2 * 1024 * 2 * 2
    assert s2["psac_p"] == 2 * 1024 * 8 and s2["psac_s"] == 2 * 1024 * 2
    assert s2["psac_basis"] == 4 * 2 * 64 * 8 * 4


def test_compression_ratio_matches_layout(lib):
    """Closed-form ratio == bf16 bytes / bytes of the buffers a full cache
    uses, when chunks fill whole tiles (no padding)."""
    for p, H, d, n, chunks in [(qvg.Params(C=16, L=1, bits=2, group=32), 2, 64, 256, 4),
                               (qvg.Params(C=16, L=3, bits=2, group=32), 2, 64, 256, 4),
                               (qvg.Params(C=16, L=2, bits=4, group=32), 2, 64, 256, 4),
                               (qvg.Params(C=256, L=1, bits=2, group=64), 16, 128, 4608, 8)]:
        s = qvg.cache_bytes(p, H, d, n * chunks, chunks)
        used = s["codes"] + s["scales"] + s["ids"] + s["cent"]
        assert qvg.compression_ratio(p, H, d, n, chunks) == pytest.approx(H * n * chunks * d * 2 / used)
    # INT2, G=64, d=128, C=256, 4680-token chunks: 32 B codes + 4 B scales
    # + 1 B id per token and head, plus 64 KiB of centroids per chunk and head.
    r = qvg.compression_ratio(qvg.Params(C=256, L=1, bits=2, group=64), 16, 128, 4680, 8)
    assert r == pytest.approx(256 / (37 + 256 * 128 * 2 / 4680))


def test_kv_size_formula():
    """The page's worked example: 32 layers x 4096 hidden (K and V, fp16) is
    16 KB per token per layer, ~512 KB per token, ~8 GB for 16,000 tokens."""
    assert qvg.kv_bytes_uncompressed(1, 32, 128, 1) == 16 * 1024
    assert qvg.kv_bytes_uncompressed(32, 32, 128, 1) == 512 * 1024
    assert qvg.kv_bytes_uncompressed(32, 32, 128, 16000) / 2 ** 30 == pytest.approx(7.81, abs=0.01)


def _params(**kw):
    return qvg.Params(**kw).c()


@pytest.mark.parametrize("kw,code", [
    (dict(bits=3), qvg.QVG_ERR_INVALID_ARG),
    (dict(L=0), qvg.QVG_ERR_INVALID_ARG),
    (dict(group=48), qvg.QVG_ERR_INVALID_ARG),
    (dict(group=2), qvg.QVG_ERR_UNSUPPORTED),
    (dict(C=300), qvg.QVG_ERR_UNSUPPORTED),
    (dict(scale_mode=1, bits=4), qvg.QVG_ERR_INVALID_ARG),
    (dict(flags=64), qvg.QVG_ERR_INVALID_ARG),
    (dict(C=0, flags=qvg.QVG_GIVEN_CENTROIDS), qvg.QVG_ERR_INVALID_ARG),
])
def test_param_validation(lib, kw, code):
    out = (ct.c_size_t * qvg.QVG_CACHE_NBUF)()
    p = _params(**kw)
    assert lib.qvg_cache_bytes(ct.byref(p), 2, 128, 1024, 4, out) == code


def test_unsupported_head_dim(lib):
    out = (ct.c_size_t * qvg.QVG_CACHE_NBUF)()
    p = _params(group=32)
    assert lib.qvg_cache_bytes(ct.byref(p), 2, 96, 1024, 4, out) == qvg.QVG_ERR_UNSUPPORTED


def _fake_cache(H=2, d=64, cap=512, max_chunks=2, n_chunks=0, n_tokens=0):
    # Pointers are never dereferenced: every case below fails validation first.
    fake = ct.c_void_p(0x1000)
    return qvg._Cache(H, d, cap, max_chunks, n_chunks, n_tokens, *([fake] * qvg.QVG_CACHE_NBUF))


def test_compress_rejects_on_host(lib):
    p = _params(C=16, group=32)
    x = ct.c_void_p(0x2000)
    ws = ct.c_void_p(0x100000)
    c = _fake_cache()
    assert lib.qvg_compress_chunk(ct.byref(p), x, 0, None, None, ct.byref(c), ws, 1 << 30, None) == qvg.QVG_ERR_INVALID_ARG
    assert lib.qvg_compress_chunk(ct.byref(p), None, 10, None, None, ct.byref(c), ws, 1 << 30, None) == qvg.QVG_ERR_INVALID_ARG
    full = _fake_cache(n_chunks=2, n_tokens=256)
    assert lib.qvg_compress_chunk(ct.byref(p), x, 10, None, None, ct.byref(full), ws, 1 << 30, None) == qvg.QVG_ERR_CAPACITY
    nearly = _fake_cache(n_chunks=1, n_tokens=384)
    assert lib.qvg_compress_chunk(ct.byref(p), x, 200, None, None, ct.byref(nearly), ws, 1 << 30, None) == qvg.QVG_ERR_CAPACITY
    assert lib.qvg_compress_chunk(ct.byref(p), x, 100, None, None, ct.byref(c), ws, 16, None) == qvg.QVG_ERR_WORKSPACE
    assert lib.qvg_compress_chunk(ct.byref(p), x, 100, None, None, ct.byref(c), None, 0, None) == qvg.QVG_ERR_WORKSPACE
    pq = _params(C=16, group=32, flags=qvg.QVG_QSAC)
    assert lib.qvg_compress_chunk(ct.byref(pq), x, 100, None, None, ct.byref(c), ws, 1 << 30, None) == qvg.QVG_ERR_INVALID_ARG
    bad = _fake_cache(cap=500)
    assert lib.qvg_compress_chunk(ct.byref(p), x, 100, None, None, ct.byref(bad), ws, 1 << 30, None) == qvg.QVG_ERR_INVALID_ARG
    # the chunk and the PSAC basis are read in 16-byte vectors
    assert lib.qvg_compress_chunk(ct.byref(p), ct.c_void_p(0x2008), 100, None, None, ct.byref(c), ws, 1 << 30,
                                  None) == qvg.QVG_ERR_INVALID_ARG
    pp = _params(C=16, group=32, flags=qvg.QVG_PSAC)
    basis = ct.cast(ct.c_void_p(0x5004), ct.POINTER(ct.c_float))
    assert lib.qvg_compress_chunk(ct.byref(pp), x, 100, None, basis, ct.byref(c), ws, 1 << 30,
                                  None) == qvg.QVG_ERR_INVALID_ARG
    # the counters are untouched by a rejected call
    assert c.n_chunks == 0 and c.n_tokens == 0


def test_attention_and_decompress_reject_on_host(lib):
    p = _params(C=16, group=32)
    k = _fake_cache(n_chunks=1, n_tokens=128)
    v = _fake_cache(n_chunks=1, n_tokens=256)
    q, o = ct.c_void_p(0x3000), ct.c_void_p(0x4000)
    assert lib.qvg_attention(ct.byref(p), q, 4, 2, ct.byref(k), ct.byref(v), 0.0, o, 0, None, None, None, 0, None) == qvg.QVG_ERR_INVALID_ARG
    assert lib.qvg_attention(ct.byref(p), q, 4, 3, ct.byref(k), ct.byref(k), 0.0, o, 0, None, None, None, 0, None) == qvg.QVG_ERR_INVALID_ARG
    assert lib.qvg_attention(ct.byref(p), q, 4, 2, ct.byref(k), ct.byref(k), 0.0, o, 7, None, None, None, 0, None) == qvg.QVG_ERR_INVALID_ARG
    empty = _fake_cache()
    assert lib.qvg_attention(ct.byref(p), q, 4, 2, ct.byref(empty), ct.byref(empty), 0.0, o, 0, None, None, None, 0, None) == qvg.QVG_ERR_INVALID_ARG
    assert lib.qvg_decompress(ct.byref(p), ct.byref(k), 0, 200, o, 0, None) == qvg.QVG_ERR_INVALID_ARG
    assert lib.qvg_decompress(ct.byref(p), ct.byref(k), -1, 10, o, 0, None) == qvg.QVG_ERR_INVALID_ARG
    # tok0 + ntok past the end even where int32 addition would wrap
    assert lib.qvg_decompress(ct.byref(p), ct.byref(k), 2**31 - 10, 2**31 - 10, o, 0, None) == qvg.QVG_ERR_INVALID_ARG
    assert lib.qvg_decompress(ct.byref(p), ct.byref(k), 0, 64, ct.c_void_p(0x4002), 0, None) == qvg.QVG_ERR_INVALID_ARG
    # queries and outputs move in 16-byte vectors
    kk = _fake_cache(n_chunks=1, n_tokens=128)
    for qq, oo in ((ct.c_void_p(0x3008), o), (q, ct.c_void_p(0x4004))):
        assert lib.qvg_attention(ct.byref(p), qq, 4, 2, ct.byref(kk), ct.byref(kk), 0.0, oo, 0, None, None, None, 0,
                                 None) == qvg.QVG_ERR_INVALID_ARG


def test_outlier_split_arguments(lib):
    """QVG_OUTLIER: groups above 64 channels are refused (above 100 values a
    group can hold more than one value over its P99); the cache must carry
    the two side-list buffers, which qvg_cache_bytes sizes."""
    p = _params(C=16, group=32, flags=qvg.QVG_OUTLIER)
    out = (ct.c_size_t * qvg.QVG_CACHE_NBUF)()
    assert lib.qvg_cache_bytes(ct.byref(p), 2, 64, 512, 2, out) == qvg.QVG_OK
    assert out[10] == 2 * 512 * 2 * 2 and out[11] == 2 * 512 * 2
    p0 = _params(C=16, group=32)
    assert lib.qvg_cache_bytes(ct.byref(p0), 2, 64, 512, 2, out) == qvg.QVG_OK
    assert out[10] == 0 and out[11] == 0
    big = _params(C=16, group=128, flags=qvg.QVG_OUTLIER)
    assert lib.qvg_cache_bytes(ct.byref(big), 2, 128, 512, 2, out) == qvg.QVG_ERR_UNSUPPORTED
    c = _fake_cache()
    c.outl_val = None
    x, ws = ct.c_void_p(0x2000), ct.c_void_p(0x100000)
    assert lib.qvg_compress_chunk(ct.byref(p), x, 100, None, None, ct.byref(c), ws, 1 << 30, None) == qvg.QVG_ERR_INVALID_ARG


def test_anchor_arguments(lib):
    """Temporal anchors: anchor_every >= 0; with anchors the cache carries
    the bf16 anchor arena (ceil(max_chunks / k) chunks of S rows, S the
    capacity per chunk rounded up to a tile) and the per-chunk table; an
    anchor chunk longer than S is refused."""
    p = _params(C=16, group=32, anchor_every=2)
    out = (ct.c_size_t * qvg.QVG_CACHE_NBUF)()
    assert lib.qvg_cache_bytes(ct.byref(p), 2, 64, 512, 4, out) == qvg.QVG_OK
    assert out[12] == 2 * 128 * 2 * 64 * 2 and out[13] == 4 * 4
    p3 = _params(C=16, group=32, anchor_every=3)
    assert lib.qvg_cache_bytes(ct.byref(p3), 2, 64, 512, 4, out) == qvg.QVG_OK
    assert out[12] == 2 * 128 * 2 * 64 * 2
    p0 = _params(C=16, group=32)
    assert lib.qvg_cache_bytes(ct.byref(p0), 2, 64, 512, 4, out) == qvg.QVG_OK
    assert out[12] == 0 and out[13] == 0
    bad = _params(C=16, group=32, anchor_every=-1)
    assert lib.qvg_cache_bytes(ct.byref(bad), 2, 64, 512, 4, out) == qvg.QVG_ERR_INVALID_ARG
    x, ws = ct.c_void_p(0x2000), ct.c_void_p(0x100000)
    c = _fake_cache(cap=512, max_chunks=2)  # S = 256 rows per anchor chunk
    assert lib.qvg_compress_chunk(ct.byref(p), x, 300, None, None, ct.byref(c), ws, 1 << 30, None) == qvg.QVG_ERR_CAPACITY
    c.anchor = None
    assert lib.qvg_compress_chunk(ct.byref(p), x, 100, None, None, ct.byref(c), ws, 1 << 30, None) == qvg.QVG_ERR_INVALID_ARG
    assert c.n_chunks == 0 and c.n_tokens == 0


def test_attention_ar_rejects_on_host(lib):
    """The AR-step call: raw current-chunk buffers must be present and
    16-byte aligned, n_cur >= 0, and there must be at least one key."""
    p = _params(C=16, group=32)
    k = _fake_cache(n_chunks=1, n_tokens=128)
    empty = _fake_cache()
    q, o = ct.c_void_p(0x3000), ct.c_void_p(0x4000)
    kr, vr = ct.c_void_p(0x6000), ct.c_void_p(0x7000)
    f = lib.qvg_attention_ar

    def call(kc, vc, kcur, vcur, n):
        return f(ct.byref(p), q, 4, 2, ct.byref(kc), ct.byref(vc), kcur, vcur, n, 0.0, o, 0, None, None, None, 0, None)

    assert call(k, k, kr, vr, -1) == qvg.QVG_ERR_INVALID_ARG
    assert call(k, k, None, vr, 10) == qvg.QVG_ERR_INVALID_ARG
    assert call(k, k, kr, None, 10) == qvg.QVG_ERR_INVALID_ARG
    assert call(k, k, ct.c_void_p(0x6008), vr, 10) == qvg.QVG_ERR_INVALID_ARG
    assert call(empty, empty, kr, vr, 0) == qvg.QVG_ERR_INVALID_ARG  # no keys
    assert call(empty, empty, None, None, 0) == qvg.QVG_ERR_INVALID_ARG
    assert call(k, k, kr, vr, 2 ** 31 - 100) == qvg.QVG_ERR_INVALID_ARG  # slot numbers overflow int32
    # no query: nothing to launch
    assert f(ct.byref(p), q, 0, 2, ct.byref(empty), ct.byref(empty), kr, vr, 10, 0.0, o, 0, None, None, None, 0,
             None) == qvg.QVG_OK


def test_quantwm_reject_on_host(lib):
    f = ct.c_void_p(0x5000)
    assert lib.quantwm_query_stats(f, 10, 3, 2, 128, 0, f, f, f, None) == qvg.QVG_ERR_INVALID_ARG
    assert lib.quantwm_query_stats(f, 10, 2, 2, 96, 0, f, f, f, None) == qvg.QVG_ERR_UNSUPPORTED
    assert lib.quantwm_psac_basis(f, f, 2, 128, 4, f, f, f, None) == qvg.QVG_ERR_UNSUPPORTED
    assert lib.quantwm_psac_basis(f, f, 2, 256, 8, f, f, f, None) == qvg.QVG_ERR_UNSUPPORTED
    assert lib.quantwm_psac_basis(None, f, 2, 128, 8, f, f, f, None) == qvg.QVG_ERR_INVALID_ARG


def test_attention_workspace_only_for_split_queries(lib):
    """qvg_attention splits the cache over extra CTAs only when the query
    blocks alone cannot fill the GPU: few queries need a workspace (partial
    outputs, log-sum-exp, best logits), a full chunk of queries none."""
    p = qvg.Params(C=256, L=1, bits=2, group=64, iters=8)
    small = qvg.workspace_size(p, qvg.QVG_OP_ATTENTION, 16, 16, 128, 16)
    assert small >= 2 * 16 * 16 * (128 + 3) * 4  # at least two splits
    assert small % 256 == 0
    assert qvg.workspace_size(p, qvg.QVG_OP_ATTENTION, 4680, 16, 128, 16) == 0


def test_debug_set_wait_arguments(lib):
    """The bounded-wait test hook takes inject 0 or 1 and touches no device
    (it only sets the calling host thread's launch settings)."""
    assert lib.qvg_debug_set_wait(ct.c_uint64(1000), 2) == qvg.QVG_ERR_INVALID_ARG
    assert lib.qvg_debug_set_wait(ct.c_uint64(1000), -1) == qvg.QVG_ERR_INVALID_ARG
    assert lib.qvg_debug_set_wait(ct.c_uint64(1000000), 1) == qvg.QVG_OK
    assert lib.qvg_debug_set_wait(ct.c_uint64(0), 0) == qvg.QVG_OK  # back to the default


def test_noalloc_checks_arguments_before_scratch_size(lib):
    """qvg_compress_chunk_noalloc reports argument and capacity errors with
    qvg_compress_chunk's codes, and QVG_ERR_WORKSPACE only for a valid call
    whose workspace would exceed the fixed scratch."""
    p = _params(C=16, group=32)
    x = ct.c_void_p(0x2000)
    c = _fake_cache()
    assert lib.qvg_compress_chunk_noalloc(ct.byref(p), None, 100, None, None, ct.byref(c), None) == qvg.QVG_ERR_INVALID_ARG
    assert lib.qvg_compress_chunk_noalloc(ct.byref(p), x, 70000, None, None, ct.byref(c), None) == qvg.QVG_ERR_INVALID_ARG
    full = _fake_cache(n_chunks=2, n_tokens=256)
    assert lib.qvg_compress_chunk_noalloc(ct.byref(p), x, 10, None, None, ct.byref(full), None) == qvg.QVG_ERR_CAPACITY
    # a valid three-stage chunk of 65,535 tokens x 32 heads needs far more than the scratch
    p3 = _params(C=16, group=32, L=3)
    big = _fake_cache(H=32, cap=65536, max_chunks=1)
    assert qvg.workspace_size(qvg.Params(C=16, L=3, bits=2, group=32), qvg.QVG_OP_COMPRESS, 65535, 32, 64) \
        > qvg.NOALLOC_SCRATCH_BYTES
    assert lib.qvg_compress_chunk_noalloc(ct.byref(p3), x, 65535, None, None, ct.byref(big), None) == qvg.QVG_ERR_WORKSPACE
    assert c.n_chunks == 0 and full.n_chunks == 2 and big.n_chunks == 0


def test_misaligned_cache_buffer_is_refused(lib):
    """Every cache buffer must be 16-byte aligned (the kernels read them with
    vector loads): a cache with any one buffer 8 bytes off is refused by
    compress, decompress and attention before anything is launched.  The
    calls are otherwise valid, so this runs only where no GPU is visible."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-only check: the fake cache pointers must never reach a device")
    fields = [f for f, _ in qvg._Cache._fields_[6:]]
    assert len(fields) == qvg.QVG_CACHE_NBUF
    p = _params(C=16, group=32, flags=qvg.QVG_OUTLIER)
    p.anchor_every = 4
    x, q, o = ct.c_void_p(0x2000), ct.c_void_p(0x3000), ct.c_void_p(0x4000)
    ws = ct.c_void_p(0x100000)
    # control: the same calls on an aligned cache pass the host checks (and
    # then fail for want of a device), so the refusals below are the alignment's
    c = _fake_cache(n_chunks=1, n_tokens=128)
    assert lib.qvg_decompress(ct.byref(p), ct.byref(c), 0, 64, o, 0, None) != qvg.QVG_ERR_INVALID_ARG
    assert lib.qvg_attention(ct.byref(p), q, 4, 2, ct.byref(c), ct.byref(c), 0.0, o, 0, None, None, None, 0,
                             None) != qvg.QVG_ERR_INVALID_ARG
    assert lib.qvg_compress_chunk(ct.byref(p), x, 100, None, None, ct.byref(c), ws, 1 << 30,
                                  None) != qvg.QVG_ERR_INVALID_ARG
    for f in fields:
        c = _fake_cache(n_chunks=1, n_tokens=128)
        setattr(c, f, ct.c_void_p(0x1008))
        assert lib.qvg_decompress(ct.byref(p), ct.byref(c), 0, 64, o, 0, None) == qvg.QVG_ERR_INVALID_ARG, f
        assert lib.qvg_attention(ct.byref(p), q, 4, 2, ct.byref(c), ct.byref(c), 0.0, o, 0, None, None, None, 0,
                                 None) == qvg.QVG_ERR_INVALID_ARG, f
        assert lib.qvg_compress_chunk(ct.byref(p), x, 100, None, None, ct.byref(c), ws, 1 << 30,
                                      None) == qvg.QVG_ERR_INVALID_ARG, f
        assert c.n_chunks == 1 and c.n_tokens == 128


def test_noalloc_scratch_size_matches_header():
    """The binding's scratch size is the header's QVG_NOALLOC_SCRATCH_BYTES."""
    src = open(os.path.join(ROOT, "include", "qvg.h")).read()
    m = re.search(r"#define\s+QVG_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", src)
    assert m, "QVG_NOALLOC_SCRATCH_BYTES not found"
    assert qvg.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))
