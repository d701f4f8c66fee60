"""The boundary on the GPU: bounded device waits and calls from several host
threads.

- A kernel whose wait runs out stops, waits (at the default bound) for the
  tensor-core work it has issued, frees its tensor memory and latches
  QVG_ERR_TIMEOUT; qvg_get_status reports it once, and the next normal call
  on the same context is QVG_OK with the usual results.  The wait is made to
  run out with the library's test hook (qvg_debug_set_wait): one extra wait
  on a barrier that nothing completes, bounded at 1 ms.  No fault, trap or
  endless loop is involved.
- First calls racing from two host threads (fresh process) and concurrent
  calls on two streams give the results of the same calls made one after
  the other.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import video_diffusion_kv_gb300 as qvg
from video_diffusion_kv_gb300 import synth

from _helpers import to_dev

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
W = synth.WORKLOADS
TINY = qvg.Params(C=16, L=1, bits=2, group=32, iters=10, seed=41)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    qvg.debug_set_wait(0, False)


def _tiny_caches(n_chunks=4, seed=5):
    w = W["tiny"]
    kc = qvg.CompressedKV(TINY, w.H, w.d, n_chunks * 256, n_chunks)
    vc = qvg.CompressedKV(TINY, w.H, w.d, n_chunks * 256, n_chunks)
    for k in range(n_chunks):
        qvg.compress_chunk(TINY, to_dev(synth.chunk_kv(w, seed, k, synth.KIND_K)), kc)
        qvg.compress_chunk(TINY, to_dev(synth.chunk_kv(w, seed, k, synth.KIND_V)), vc)
    return kc, vc


def _buffers(c):
    return {n: b.cpu().numpy().copy() for n, b in c.buffers.items() if b is not None}


def test_compress_wait_timeout_is_reported_and_recovers():
    """k-means assignment: the injected wait runs out with an MMA in flight;
    the call's status is TIMEOUT, cleared by the read, and the same chunk
    then compresses to the bytes of an undisturbed run."""
    w = W["tiny"]
    x = to_dev(synth.chunk_kv(w, 6, 0, synth.KIND_K))
    ref = qvg.CompressedKV(TINY, w.H, w.d, 256, 1)
    qvg.compress_chunk(TINY, x, ref)
    assert qvg.get_status() == qvg.QVG_OK
    bad = qvg.CompressedKV(TINY, w.H, w.d, 256, 1)
    qvg.debug_set_wait(1_000_000, True)
    try:
        qvg.compress_chunk(TINY, x, bad)  # launches succeed; the device reports
    finally:
        qvg.debug_set_wait(0, False)
    assert qvg.get_status() == qvg.QVG_ERR_TIMEOUT
    assert qvg.get_status() == qvg.QVG_OK  # read once, then cleared
    again = qvg.CompressedKV(TINY, w.H, w.d, 256, 1)
    qvg.compress_chunk(TINY, x, again)
    assert qvg.get_status() == qvg.QVG_OK
    a, b = _buffers(ref), _buffers(again)
    for n in a:
        np.testing.assert_array_equal(a[n], b[n], err_msg=n)


@pytest.mark.parametrize("nq,split", [(256, False), (16, True)])
def test_attention_wait_timeout_is_reported_and_recovers(nq, split):
    """Attention (256 queries with one CTA per head; 16 queries with the
    cache split over several CTAs, then merged): each softmax group's issuer
    waits on a barrier that nothing completes with its first S MMA in
    flight; every role stops, the kernel drains and frees its tensor memory,
    the status is TIMEOUT, and the next call returns the undisturbed
    result."""
    w = W["tiny"]
    kc, vc = _tiny_caches()
    q = to_dev(synth.queries(w, 5, 4)[:nq])
    ref, _, _ = qvg.attention(TINY, q, kc, vc, allow_split=split)
    assert qvg.get_status() == qvg.QVG_OK
    qvg.debug_set_wait(1_000_000, True)
    try:
        qvg.attention(TINY, q, kc, vc, allow_split=split)
    finally:
        qvg.debug_set_wait(0, False)
    assert qvg.get_status() == qvg.QVG_ERR_TIMEOUT
    out, _, _ = qvg.attention(TINY, q, kc, vc, allow_split=split)
    assert qvg.get_status() == qvg.QVG_OK
    torch.testing.assert_close(out, ref, rtol=0, atol=0)


def test_status_on_a_stream():
    """qvg_get_status(stream) synchronises that stream and reads the device
    word: a timeout raised by work on a side stream is reported there."""
    w = W["tiny"]
    x = to_dev(synth.chunk_kv(w, 7, 0, synth.KIND_V))
    s = torch.cuda.Stream()
    c = qvg.CompressedKV(TINY, w.H, w.d, 256, 1)
    torch.cuda.synchronize()
    qvg.debug_set_wait(1_000_000, True)
    try:
        with torch.cuda.stream(s):
            qvg.compress_chunk(TINY, x, c, stream=s)
    finally:
        qvg.debug_set_wait(0, False)
    assert qvg.get_status(s) == qvg.QVG_ERR_TIMEOUT
    assert qvg.get_status(s) == qvg.QVG_OK


_THREADS = textwrap.dedent("""
    import sys, threading
    sys.path.insert(0, %(root)r)
    sys.path.insert(0, %(tests)r)
    import numpy as np, torch
    import video_diffusion_kv_gb300 as qvg
    from video_diffusion_kv_gb300 import synth
    from _helpers import to_dev
    torch.cuda.set_device(0)
    W = synth.WORKLOADS
    jobs = [(W["tiny"], qvg.Params(C=16, L=1, bits=2, group=32, iters=10, seed=51), 2),
            (W["longcat"], qvg.Params(C=256, L=1, bits=2, group=64, iters=8, seed=52), 1)]
    inputs = []
    for w, p, n in jobs:
        ks = [to_dev(synth.chunk_kv(w, 9, k, synth.KIND_K)) for k in range(n)]
        vs = [to_dev(synth.chunk_kv(w, 9, k, synth.KIND_V)) for k in range(n)]
        q = to_dev(synth.queries(w, 9, n)[:512])
        inputs.append((ks, vs, q))
    torch.cuda.synchronize()

    def run(j, stream, out):
        w, p, n = jobs[j]
        ks, vs, q = inputs[j]
        slots = -(-w.N // 128) * 128
        with torch.cuda.stream(stream):
            kc = qvg.CompressedKV(p, w.H, w.d, n * slots, n)
            vc = qvg.CompressedKV(p, w.H, w.d, n * slots, n)
            for k in range(n):
                qvg.compress_chunk(p, ks[k], kc, stream=stream)
                qvg.compress_chunk(p, vs[k], vc, stream=stream)
            o, lse, _ = qvg.attention(p, q, kc, vc, want_lse=True, stream=stream)
            stream.synchronize()
        out[j] = (o.cpu().numpy(), lse.cpu().numpy(),
                  {nm: b.cpu().numpy() for nm, b in kc.buffers.items() if b is not None})

    # first calls of this process, racing from two host threads on two streams
    par = {}
    ts = [threading.Thread(target=run, args=(j, torch.cuda.Stream(), par)) for j in range(2)]
    for t in ts: t.start()
    for t in ts: t.join()
    assert qvg.get_status() == qvg.QVG_OK
    seq = {}
    for j in range(2):
        run(j, torch.cuda.current_stream(), seq)
    for j in range(2):
        np.testing.assert_array_equal(par[j][0], seq[j][0])
        np.testing.assert_array_equal(par[j][1], seq[j][1])
        for nm in seq[j][2]:
            np.testing.assert_array_equal(par[j][2][nm], seq[j][2][nm], err_msg=nm)
    print("THREADS_OK")
""")


def test_first_calls_from_two_threads():
    """A fresh process whose first library calls come from two host threads
    at once, each on its own stream (a tiny and a LongCat-like layer): the
    per-device launch set-up is made once, and every output equals that of
    the same calls made one after the other."""
    code = _THREADS % {"root": ROOT, "tests": os.path.join(ROOT, "tests")}
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "THREADS_OK" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
