"""The entry point for callers that cannot allocate device memory.

qvg_compress_chunk_noalloc takes no workspace: it runs qvg_compress_chunk on
a fixed 32 MiB scratch array that the library holds on the device.  Callers
that cannot provide a workspace -- code inside a framework whose memory pool
owns the device and forbids extra cudaMalloc calls, or code that must not
risk cudaMalloc's device-wide synchronisation -- use it instead.

This file is collected last so that, should it fail, a run that stops at the
first failure has already run every other test.  It must pass on its own in a
fresh process and after the other tests.
"""
import ctypes as ct

import numpy as np
import pytest
import torch

import video_diffusion_kv_gb300 as qvg
from video_diffusion_kv_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _buffers(cache):
    return {n: b.cpu().numpy().copy() for n, b in cache.buffers.items() if b is not None}


@pytest.mark.parametrize("wname,params", [
    ("longcat", qvg.Params(C=256, L=1, bits=2, group=64, iters=8, seed=31)),
    ("qvgpro", qvg.Params(C=16, L=3, bits=2, group=32, iters=10, seed=32)),
])
def test_noalloc_matches_workspace_entry(wname, params):
    """Two chunks in a row through the C ABI: the no-allocation entry point
    leaves exactly the bytes the workspace entry point leaves (the byte and
    index outputs are compared bit for bit, as everywhere in these tests)."""
    w = synth.WORKLOADS[wname]
    lib = qvg.lib()
    cap = 2 * (-(-w.N // 128) * 128)
    ref = qvg.CompressedKV(params, w.H, w.d, cap, 2)
    got = qvg.CompressedKV(params, w.H, w.d, cap, 2)
    need = qvg.workspace_size(params, qvg.QVG_OP_COMPRESS, w.N, w.H, w.d)
    assert need <= qvg.NOALLOC_SCRATCH_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    stream = ct.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = params.c()
    for k in range(2):
        x = torch.from_numpy(synth.chunk_kv(w, 33, k, synth.KIND_K)).to("cuda", torch.bfloat16).contiguous()
        cr = ref.c()
        assert lib.qvg_compress_chunk(ct.byref(p), ct.c_void_p(x.data_ptr()), w.N, None, None, ct.byref(cr),
                                      ct.c_void_p(ws.data_ptr()), need, stream) == qvg.QVG_OK
        ref.n_chunks, ref.n_tokens = cr.n_chunks, cr.n_tokens
        cg = got.c()
        assert lib.qvg_compress_chunk_noalloc(ct.byref(p), ct.c_void_p(x.data_ptr()), w.N, None, None,
                                              ct.byref(cg), stream) == qvg.QVG_OK
        got.n_chunks, got.n_tokens = cg.n_chunks, cg.n_tokens
    assert qvg.get_status() == qvg.QVG_OK
    assert (got.n_chunks, got.n_tokens) == (ref.n_chunks, ref.n_tokens) == (2, cap)
    a, b = _buffers(ref), _buffers(got)
    for name in a:
        np.testing.assert_array_equal(b[name], a[name], err_msg=name)
    # and the reconstruction read back from both caches agrees
    np.testing.assert_array_equal(qvg.decompress(params, got, 0, got.n_tokens).cpu().numpy(),
                                  qvg.decompress(params, ref, 0, ref.n_tokens).cpu().numpy())


def test_noalloc_rejects_oversized_workspace():
    """A configuration whose workspace exceeds the fixed scratch is refused
    before anything runs, and the cache is left untouched."""
    w = synth.WORKLOADS["longcat"]
    params = qvg.Params(C=256, L=3, bits=2, group=64, iters=1, seed=34)
    assert qvg.workspace_size(params, qvg.QVG_OP_COMPRESS, w.N, w.H, w.d) > qvg.NOALLOC_SCRATCH_BYTES
    cache = qvg.CompressedKV(params, w.H, w.d, 4736, 1)
    x = torch.zeros((w.N, w.H, w.d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qvg.QvgError) as e:
        qvg.compress_chunk_noalloc(params, x, cache)
    assert e.value.status == qvg.QVG_ERR_WORKSPACE
    assert cache.n_chunks == 0 and cache.n_tokens == 0
