"""Multi-layer streaming rollout through the C ABI (tiny shapes): each chunk
step runs, layer by layer, the AR-step attention (queries over the layer's
compressed history plus the chunk's raw K/V), then compresses the chunk
into that layer's cache.  Checked: every step's attention against the fp64
oracle on the same bytes; the layers' caches equal, byte for byte, caches
built by compressing the same chunks alone (layers share nothing); and the
memory accounting (buffer sizes, the bf16 size formula of "The 2-bit
quantisation trap", section 1)."""
import numpy as np
import pytest
import torch

import oracle
import video_diffusion_kv_gb300 as qvg
from video_diffusion_kv_gb300 import synth

from _helpers import ATTN_TOL, host_cache, oracle_rebuild, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def test_layers_by_chunks_rollout():
    w = synth.WORKLOADS["tiny"]
    p = qvg.Params(C=16, L=1, bits=2, group=32, iters=6, seed=41)
    layers, chunks = 3, 3
    cap = chunks * 256
    kcs = [qvg.CompressedKV(p, w.H, w.d, cap, chunks) for _ in range(layers)]
    vcs = [qvg.CompressedKV(p, w.H, w.d, cap, chunks) for _ in range(layers)]
    data = {(li, k): (synth.chunk_kv(w, 50 + li, k, synth.KIND_K), synth.chunk_kv(w, 50 + li, k, synth.KIND_V),
                      synth.queries(w, 50 + li, k)) for li in range(layers) for k in range(chunks)}
    for k in range(chunks):
        for li in range(layers):
            kr, vr, q = data[li, k]
            out, lse, top1 = qvg.attention_ar(p, to_dev(q), kcs[li], vcs[li], to_dev(kr), to_dev(vr),
                                              want_lse=True, want_top1=True)
            hk, hv = host_cache(kcs[li]), host_cache(vcs[li])
            n = kcs[li].n_chunks
            kh = np.concatenate([oracle_rebuild(hk, p, c) for c in range(n)] + [np.zeros((0, w.H, w.d), np.float32)])
            vh = np.concatenate([oracle_rebuild(hv, p, c) for c in range(n)] + [np.zeros((0, w.H, w.d), np.float32)])
            slots = np.concatenate([np.arange(hk["start"][c], hk["start"][c] + hk["length"][c]) for c in range(n)]
                                   + [np.zeros(0, np.int64)])
            ref, rlse, rtop = oracle.attention_ar(q, kh, vh, kr, vr, slots, kcs[li].n_tokens, nthreads=8)
            got = out.cpu().numpy().astype(np.float64)
            for h in range(q.shape[1]):
                assert np.abs(got[:, h] - ref[:, h]).max() <= ATTN_TOL * np.abs(ref[:, h]).max(), (k, li, h)
            np.testing.assert_allclose(lse.cpu().numpy(), rlse, atol=2e-3, rtol=0)
            assert (top1.cpu().numpy() == rtop).mean() >= 0.95
            qvg.compress_chunk(p, to_dev(kr), kcs[li])
            qvg.compress_chunk(p, to_dev(vr), vcs[li])
    assert qvg.get_status() == qvg.QVG_OK
    # each layer's cache equals the same chunks compressed on their own
    for li in range(layers):
        for cs, kind in ((kcs, 0), (vcs, 1)):
            alone = qvg.CompressedKV(p, w.H, w.d, cap, chunks)
            for k in range(chunks):
                qvg.compress_chunk(p, to_dev(data[li, k][kind]), alone)
            a, b = host_cache(cs[li]), host_cache(alone)
            for name in a:
                np.testing.assert_array_equal(a[name], b[name], err_msg=(li, kind, name))
    # memory accounting
    sizes = qvg.cache_bytes(p, w.H, w.d, cap, chunks)
    held = sum(c.nbytes for c in kcs + vcs)
    assert held == 2 * layers * sum(sizes.values())
    assert qvg.kv_bytes_uncompressed(layers, w.H, w.d, chunks * w.N) == 2 * layers * w.H * w.d * chunks * w.N * 2
    ratio = qvg.compression_ratio(p, w.H, w.d, w.N, chunks)
    per_tok = w.d * p.bits / 8 + 2 * w.d / p.group + 1
    assert abs(ratio - (w.H * chunks * w.N * w.d * 2) / (w.H * chunks * w.N * per_tok + w.H * chunks * p.C * w.d * 2)) < 1e-9
