// api.cu -- the extern "C" entry points of libqvg: argument validation,
// workspace carving and the launch sequence of each call.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "common.cuh"

namespace qvg {
__device__ int g_qvg_error = 0;

static thread_local cudaError_t t_last_cuda_error = cudaSuccess;
void note_cuda_error(cudaError_t e) { t_last_cuda_error = e; }

namespace {
// Per-device tables of the launch set-up; each entry is written once, by
// the first call that needs it on that device, and published atomically
// (a racing second writer stores the same value).
std::atomic<int *> g_error_word[kMaxDevices];
std::atomic<int> g_sm_count[kMaxDevices];
std::mutex g_attr_mutex;  // serialises cudaFuncSetAttribute calls of first launches

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    return dev >= 0 && dev < kMaxDevices ? dev : -1;
}

// Bounded-wait settings of the calling host thread (qvg_debug_set_wait).
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s
thread_local uint64_t t_wait_ns = kDefaultWaitNs;
thread_local int t_wait_inject = 0;
}  // namespace

uint64_t wait_limit_ns() { return t_wait_ns; }
int wait_inject() { return t_wait_inject; }

int *device_error_word() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    int *p = g_error_word[dev].load(std::memory_order_acquire);
    if (!p) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_qvg_error) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        p = static_cast<int *>(a);
        g_error_word[dev].store(p, std::memory_order_release);
    }
    return p;
}

int sm_count_current() {
    const int dev = current_device();
    if (dev < 0) return 152;
    int n = g_sm_count[dev].load(std::memory_order_acquire);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            return 152;
        }
        g_sm_count[dev].store(n, std::memory_order_release);
    }
    return n;
}

qvg_status smem_limit_once(std::atomic<uint64_t> &done, const void *func, int bytes) {
    const int dev = current_device();
    if (dev < 0) return QVG_ERR_CUDA;
    const uint64_t bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit) return QVG_OK;
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    if (done.load(std::memory_order_acquire) & bit) return QVG_OK;
    const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        note_cuda_error(e);
        return QVG_ERR_CUDA;
    }
    done.fetch_or(bit, std::memory_order_release);
    return QVG_OK;
}
}  // namespace qvg

using namespace qvg;

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Validation of the method parameters against a head_dim.
qvg_status check_params(const qvg_params *p, int d) {
    if (!p) return QVG_ERR_INVALID_ARG;
    if (p->anchor_every < 0 || p->L < 1 || p->L > 16 || p->C < 0 || p->iters < 0 ||
        p->iters > 10000 || (p->bits != 2 && p->bits != 4) || p->group < 1 ||
        (p->scale_mode != 0 && p->scale_mode != 1) || (p->flags & ~31))
        return QVG_ERR_INVALID_ARG;
    if (p->scale_mode == 1 && p->bits != 2) return QVG_ERR_INVALID_ARG;
    if (p->C > QVG_MAX_CLUSTERS) return QVG_ERR_UNSUPPORTED;
    if (d < 1 || d % p->group != 0) return QVG_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return QVG_ERR_UNSUPPORTED;
    const int e = d / 32;  // channels per lane in the row kernels
    if (p->group < e || !is_pow2(p->group / e) || p->group / e > 32) return QVG_ERR_UNSUPPORTED;
    if (p->group % 8 != 0) return QVG_ERR_UNSUPPORTED;  // the read path rebuilds 8-channel chunks
    if ((p->flags & QVG_GIVEN_CENTROIDS) && p->C == 0) return QVG_ERR_INVALID_ARG;
    // outlier split: at most one value per group lies above its P99 when G <= 100
    if ((p->flags & QVG_OUTLIER) && p->group > 64) return QVG_ERR_UNSUPPORTED;
    return QVG_OK;
}

qvg_status check_cache(const qvg_params *p, const qvg_cache *c) {
    if (!c) return QVG_ERR_INVALID_ARG;
    if (c->H < 1 || c->capacity_tokens <= 0 || c->capacity_tokens % QVG_TILE != 0 ||
        c->max_chunks < 1 || c->n_chunks < 0 || c->n_chunks > c->max_chunks ||
        c->n_tokens < 0 || c->n_tokens % QVG_TILE != 0 || c->n_tokens > c->capacity_tokens)
        return QVG_ERR_INVALID_ARG;
    if (!c->codes || !c->scales || !c->chunk_start || !c->chunk_len || !c->tile_chunk)
        return QVG_ERR_INVALID_ARG;
    if (p->C > 0 && (!c->ids || !c->cent)) return QVG_ERR_INVALID_ARG;
    if ((p->flags & QVG_PSAC) && (!c->psac_p || !c->psac_s || !c->psac_basis))
        return QVG_ERR_INVALID_ARG;
    if ((p->flags & QVG_OUTLIER) && (!c->outl_val || !c->outl_idx)) return QVG_ERR_INVALID_ARG;
    if (p->anchor_every > 0 && (!c->anchor || !c->chunk_anchor)) return QVG_ERR_INVALID_ARG;
    // every buffer is read with vector loads of up to 16 bytes
    const void *bufs[] = {c->codes,  c->scales, c->ids,        c->cent,     c->chunk_start, c->chunk_len, c->tile_chunk,
                          c->psac_p, c->psac_s, c->psac_basis, c->outl_val, c->outl_idx,    c->anchor,    c->chunk_anchor};
    for (const void *b : bufs)
        if (reinterpret_cast<uintptr_t>(b) % 16 != 0) return QVG_ERR_INVALID_ARG;
    return QVG_OK;
}

struct CompressWs {
    float *means;  // QVG_KEEP_MEANS: [L][H][C][d] at offset 0
    int32_t *ids;
    float *cnorm;
    float *xnorm;
    float *delta;
    uint16_t *gbf;
    size_t bytes;
};

CompressWs carve_compress(const qvg_params *p, int N, int H, int d, char *base) {
    CompressWs w{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *ptr = base ? base + off : nullptr;
        off += align_up(bytes);
        return ptr;
    };
    if (p->flags & QVG_KEEP_MEANS)
        w.means = reinterpret_cast<float *>(
            take(sizeof(float) * static_cast<size_t>(p->L) * H * std::max(p->C, 1) * d));
    w.ids = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * static_cast<size_t>(H) * N));
    w.cnorm = reinterpret_cast<float *>(take(sizeof(float) * static_cast<size_t>(H) * std::max(p->C, 1)));
    w.xnorm = reinterpret_cast<float *>(take(sizeof(float) * static_cast<size_t>(H) * N));
    const bool need_delta = p->L > 1 || (p->flags & QVG_PSAC);
    w.delta = need_delta ? reinterpret_cast<float *>(take(sizeof(float) * static_cast<size_t>(N) * H * d)) : nullptr;
    w.gbf = p->L > 1 ? reinterpret_cast<uint16_t *>(take(sizeof(uint16_t) * static_cast<size_t>(N) * H * d)) : nullptr;
    w.bytes = off;
    return w;
}

}  // namespace

namespace qvg {
qvg_status check_compress_args(const qvg_params *p, const void *x_bf16, int N, const float *qsac_w,
                               const float *psac_basis, const qvg_cache *cache, size_t *ws_need) {
    if (!cache || !x_bf16) return QVG_ERR_INVALID_ARG;
    qvg_status s = check_params(p, cache->d);
    if (s != QVG_OK) return s;
    if ((s = check_cache(p, cache)) != QVG_OK) return s;
    if (N < 1 || N > 65535) return QVG_ERR_INVALID_ARG;
    if ((p->flags & QVG_QSAC) && !qsac_w) return QVG_ERR_INVALID_ARG;
    if ((p->flags & QVG_PSAC) && !psac_basis) return QVG_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(x_bf16) % 16 != 0) return QVG_ERR_INVALID_ARG;
    if ((p->flags & QVG_PSAC) && reinterpret_cast<uintptr_t>(psac_basis) % 16 != 0) return QVG_ERR_INVALID_ARG;
    const int Naligned = ceil_div(N, QVG_TILE) * QVG_TILE;
    if (cache->n_chunks >= cache->max_chunks ||
        static_cast<int64_t>(cache->n_tokens) + Naligned > cache->capacity_tokens)
        return QVG_ERR_CAPACITY;
    *ws_need = carve_compress(p, N, cache->H, cache->d, nullptr).bytes;
    return QVG_OK;
}
}  // namespace qvg

extern "C" {

const char *qvg_status_string(qvg_status s) {
    switch (s) {
        case QVG_OK: return "ok";
        case QVG_ERR_INVALID_ARG: return "invalid argument";
        case QVG_ERR_UNSUPPORTED: return "unsupported configuration";
        case QVG_ERR_CUDA: return "CUDA error";
        case QVG_ERR_TIMEOUT: return "device wait exceeded its bound";
        case QVG_ERR_WORKSPACE: return "workspace missing or too small";
        case QVG_ERR_CAPACITY: return "cache capacity exceeded";
    }
    return "unknown status";
}

qvg_status qvg_cache_bytes(const qvg_params *p, int32_t H, int32_t d, int32_t cap,
                           int32_t max_chunks, size_t out[QVG_CACHE_NBUF]) {
    if (!out) return QVG_ERR_INVALID_ARG;
    qvg_status s = check_params(p, d);
    if (s != QVG_OK) return s;
    if (H < 1 || cap <= 0 || cap % QVG_TILE != 0 || max_chunks < 1) return QVG_ERR_INVALID_ARG;
    const size_t L = p->L, rows = static_cast<size_t>(H) * cap;
    out[0] = L * rows * (static_cast<size_t>(d) * p->bits / 8);
    out[1] = L * rows * (d / p->group) * sizeof(uint16_t);
    out[2] = p->C > 0 ? L * rows : 0;
    out[3] = L * H * static_cast<size_t>(max_chunks) * p->C * d * sizeof(uint16_t);
    out[4] = sizeof(int32_t) * static_cast<size_t>(max_chunks);
    out[5] = sizeof(int32_t) * static_cast<size_t>(max_chunks);
    out[6] = sizeof(int32_t) * static_cast<size_t>(cap / QVG_TILE);
    const bool psac = p->flags & QVG_PSAC;
    out[7] = psac ? rows * QVG_PSAC_RANK : 0;
    out[8] = psac ? rows * sizeof(uint16_t) : 0;
    out[9] = psac ? sizeof(float) * static_cast<size_t>(max_chunks) * H * d * QVG_PSAC_RANK : 0;
    const bool outl = p->flags & QVG_OUTLIER;
    out[10] = outl ? L * rows * (d / p->group) * sizeof(uint16_t) : 0;
    out[11] = outl ? L * rows * (d / p->group) : 0;
    const bool anch = p->anchor_every > 0;
    const size_t arows = anch ? static_cast<size_t>((max_chunks + p->anchor_every - 1) / p->anchor_every) *
                                    anchor_stride(cap, max_chunks)
                              : 0;
    out[12] = arows * H * d * sizeof(uint16_t);
    out[13] = anch ? sizeof(int32_t) * static_cast<size_t>(max_chunks) : 0;
    return QVG_OK;
}

qvg_status qvg_workspace_size(const qvg_params *p, int32_t op, int32_t n, int32_t H, int32_t d,
                              int32_t Hq, size_t *bytes) {
    if (!bytes) return QVG_ERR_INVALID_ARG;
    qvg_status s = check_params(p, d);
    if (s != QVG_OK) return s;
    if (n < 0 || H < 1) return QVG_ERR_INVALID_ARG;
    switch (op) {
        case QVG_OP_COMPRESS: *bytes = carve_compress(p, n, H, d, nullptr).bytes; return QVG_OK;
        case QVG_OP_ATTENTION:
            if (Hq < 1) return QVG_ERR_INVALID_ARG;
            *bytes = attention_split_bytes(n, Hq, d, attention_splits(n, Hq, -1));
            return QVG_OK;
        case QVG_OP_PSAC_BASIS: *bytes = 0; return QVG_OK;
    }
    return QVG_ERR_INVALID_ARG;
}


qvg_status qvg_compress_chunk(const qvg_params *p, const void *x_bf16, int32_t N,
                              const float *qsac_w, const float *psac_basis, qvg_cache *cache,
                              void *workspace, size_t ws_bytes, void *stream) {
    size_t need_bytes = 0;
    qvg_status s = check_compress_args(p, x_bf16, N, qsac_w, psac_basis, cache, &need_bytes);
    if (s != QVG_OK) return s;
    const int H = cache->H, d = cache->d;
    const int Naligned = ceil_div(N, QVG_TILE) * QVG_TILE;
    if (need_bytes > 0 && (!workspace || ws_bytes < need_bytes)) return QVG_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0) return QVG_ERR_WORKSPACE;
    const CompressWs ws = carve_compress(p, N, H, d, static_cast<char *>(workspace));
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    const int chunk = cache->n_chunks, slot0 = cache->n_tokens;
    if (p->anchor_every > 0 && chunk % p->anchor_every == 0) {
        // temporal anchor: the chunk's bf16 K/V, kept as given
        const int S = anchor_stride(cache->capacity_tokens, cache->max_chunks);
        if (N > S) return QVG_ERR_CAPACITY;
        const int row0 = (chunk / p->anchor_every) * S;
        if (cudaMemcpyAsync(cache->anchor + static_cast<size_t>(row0) * H * d, x_bf16,
                            static_cast<size_t>(N) * H * d * sizeof(uint16_t), cudaMemcpyDeviceToDevice,
                            st) != cudaSuccess)
            return QVG_ERR_CUDA;
        if ((s = launch_chunk_table(chunk, slot0, N, cache->chunk_start, cache->chunk_len, cache->tile_chunk,
                                    cache->chunk_anchor, row0, st)) != QVG_OK)
            return s;
        cache->n_chunks = chunk + 1;
        cache->n_tokens = slot0 + Naligned;
        return QVG_OK;
    }
    const int C = p->C, Ce = std::min(C, N), L = p->L;
    const float *w = (p->flags & QVG_QSAC) ? qsac_w : nullptr;
    const bool psac = p->flags & QVG_PSAC, outl = p->flags & QVG_OUTLIER;
    const size_t cap = cache->capacity_tokens, nb = static_cast<size_t>(d) * p->bits / 8;
    const size_t ng = d / p->group;
    const size_t cent_hs = static_cast<size_t>(cache->max_chunks) * C * d;
    if (psac) {
        if (cudaMemcpyAsync(cache->psac_basis + static_cast<size_t>(chunk) * H * d * QVG_PSAC_RANK,
                            psac_basis, sizeof(float) * H * d * QVG_PSAC_RANK,
                            cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return QVG_ERR_CUDA;
    }
    for (int l = 0; l < L; ++l) {
        const void *xin = l == 0 ? x_bf16 : static_cast<const void *>(ws.delta);
        const bool f32 = l > 0;
        const uint16_t *g = l == 0 ? static_cast<const uint16_t *>(x_bf16) : ws.gbf;
        uint16_t *cent = C > 0 ? cache->cent + (static_cast<size_t>(l) * H * cache->max_chunks + chunk) * C * d : nullptr;
        if (C > 0) {
            if (!(p->flags & QVG_GIVEN_CENTROIDS)) {
                if ((s = launch_kmeans_init(g, N, H, d, C, Ce, p->seed, chunk, l, cent, cent_hs, w, ws.cnorm, st)) != QVG_OK)
                    return s;
            } else if ((s = launch_centroid_norms(cent, cent_hs, H, C, d, w, ws.cnorm, st)) != QVG_OK) {
                return s;
            }
            if ((s = launch_row_norms(g, N, H, d, w, ws.xnorm, st)) != QVG_OK) return s;
            for (int it = 0; it < p->iters; ++it) {
                if ((s = launch_kmeans_assign(g, N, H, d, cent, cent_hs, Ce, ws.cnorm, C, w, ws.xnorm, ws.ids, st)) !=
                    QVG_OK)
                    return s;
                float *means = ws.means && it == p->iters - 1 ? ws.means + static_cast<size_t>(l) * H * C * d : nullptr;
                if ((s = launch_kmeans_update(xin, f32, N, H, d, ws.ids, cent, cent_hs, Ce, C, w, ws.cnorm, means,
                                              st)) !=
                    QVG_OK)
                    return s;
            }
            if ((s = launch_kmeans_assign(g, N, H, d, cent, cent_hs, Ce, ws.cnorm, C, w, ws.xnorm, ws.ids, st)) !=
                QVG_OK)
                return s;
        }
        const bool last = l == L - 1;
        const size_t lrow = static_cast<size_t>(l) * H * cap + slot0;
        s = launch_residual_quant(
            xin, f32, N, H, d, cent, cent_hs, C, ws.ids, p->bits, p->group, p->scale_mode,
            cache->codes + lrow * nb, cache->scales + lrow * ng, C > 0 ? cache->ids + lrow : nullptr, cap,
            (!last || psac) ? ws.delta : nullptr, !last ? ws.gbf : nullptr,
            (last && psac) ? psac_basis : nullptr, psac ? cache->psac_p + static_cast<size_t>(slot0) * QVG_PSAC_RANK : nullptr,
            psac ? cache->psac_s + slot0 : nullptr, cap, outl ? cache->outl_val + lrow * ng : nullptr,
            outl ? cache->outl_idx + lrow * ng : nullptr, st);
        if (s != QVG_OK) return s;
    }
    if ((s = launch_chunk_table(chunk, slot0, N, cache->chunk_start, cache->chunk_len, cache->tile_chunk,
                                p->anchor_every > 0 ? cache->chunk_anchor : nullptr, -1, st)) != QVG_OK)
        return s;
    cache->n_chunks = chunk + 1;
    cache->n_tokens = slot0 + Naligned;
    return QVG_OK;
}

qvg_status qvg_decompress(const qvg_params *p, const qvg_cache *cache, int32_t tok0, int32_t ntok,
                          void *out, int32_t out_dtype, void *stream) {
    if (!cache || !out) return QVG_ERR_INVALID_ARG;
    qvg_status s = check_params(p, cache->d);
    if (s != QVG_OK) return s;
    if ((s = check_cache(p, cache)) != QVG_OK) return s;
    if (out_dtype != QVG_OUT_F32 && out_dtype != QVG_OUT_BF16) return QVG_ERR_INVALID_ARG;
    if (tok0 < 0 || ntok < 0 || static_cast<int64_t>(tok0) + ntok > cache->n_tokens) return QVG_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(out) % 4 != 0) return QVG_ERR_INVALID_ARG;  // stored in 32-bit words
    if (ntok == 0) return QVG_OK;
    return launch_decompress(p, cache, tok0, ntok, out, out_dtype, static_cast<cudaStream_t>(stream));
}

qvg_status qvg_attention_ar(const qvg_params *p, const void *q_bf16, int32_t Nq, int32_t Hq,
                            const qvg_cache *k, const qvg_cache *v, const void *k_cur_bf16,
                            const void *v_cur_bf16, int32_t n_cur, float scale, void *out,
                            int32_t out_dtype, float *lse, int32_t *top1, void *workspace,
                            size_t ws_bytes, void *stream) {
    if (!k || !v || (!q_bf16 && Nq > 0) || (!out && Nq > 0)) return QVG_ERR_INVALID_ARG;
    if (n_cur < 0 || (n_cur > 0 && (!k_cur_bf16 || !v_cur_bf16))) return QVG_ERR_INVALID_ARG;
    if (n_cur > 0 && ((reinterpret_cast<uintptr_t>(k_cur_bf16) | reinterpret_cast<uintptr_t>(v_cur_bf16)) & 15u))
        return QVG_ERR_INVALID_ARG;
    // queries are read and outputs written in 16-byte vectors
    if (Nq > 0 && ((reinterpret_cast<uintptr_t>(q_bf16) | reinterpret_cast<uintptr_t>(out)) & 15u))
        return QVG_ERR_INVALID_ARG;
    qvg_status s = check_params(p, k->d);
    if (s != QVG_OK) return s;
    if ((s = check_cache(p, k)) != QVG_OK) return s;
    qvg_params pv = *p;
    pv.flags &= ~QVG_PSAC;  // PSAC corrects keys only
    if ((s = check_cache(&pv, v)) != QVG_OK) return s;
    if (k->H != v->H || k->d != v->d || k->n_tokens != v->n_tokens || k->n_chunks != v->n_chunks ||
        k->capacity_tokens != v->capacity_tokens || k->max_chunks != v->max_chunks)
        return QVG_ERR_INVALID_ARG;
    if (Nq < 0 || Hq < 1 || Hq % k->H != 0) return QVG_ERR_INVALID_ARG;
    if (k->n_tokens == 0 && n_cur == 0) return QVG_ERR_INVALID_ARG;
    if (n_cur > INT32_MAX - QVG_TILE - k->n_tokens) return QVG_ERR_INVALID_ARG;  // slot numbers stay int32
    if (out_dtype != QVG_OUT_F32 && out_dtype != QVG_OUT_BF16) return QVG_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return QVG_ERR_INVALID_ARG;
    const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(k->d));
    const float scale_log2 = sc * 1.4426950408889634f;
    if (workspace && reinterpret_cast<uintptr_t>(workspace) % kAlign != 0) return QVG_ERR_WORKSPACE;
    if (Nq == 0) return QVG_OK;
    return launch_attention_ws(p, static_cast<const uint16_t *>(q_bf16), Nq, Hq, k, v, scale_log2,
                               static_cast<const uint16_t *>(k_cur_bf16), static_cast<const uint16_t *>(v_cur_bf16),
                               n_cur, out, out_dtype, lse, top1, workspace, ws_bytes,
                               static_cast<cudaStream_t>(stream));
}

qvg_status qvg_attention(const qvg_params *p, const void *q_bf16, int32_t Nq, int32_t Hq,
                         const qvg_cache *k, const qvg_cache *v, float scale, void *out,
                         int32_t out_dtype, float *lse, int32_t *top1, void *workspace,
                         size_t ws_bytes, void *stream) {
    return qvg_attention_ar(p, q_bf16, Nq, Hq, k, v, nullptr, nullptr, 0, scale, out, out_dtype, lse, top1,
                            workspace, ws_bytes, stream);
}

qvg_status quantwm_query_stats(const void *q_hist_bf16, int32_t n, int32_t Hq, int32_t H, int32_t d,
                               int32_t accumulate, float *M, float *w, int64_t *count,
                               void *stream) {
    if (!M || !w || !count || (n > 0 && !q_hist_bf16)) return QVG_ERR_INVALID_ARG;
    if (n < 0 || H < 1 || Hq < 1 || Hq % H != 0 || (accumulate != 0 && accumulate != 1))
        return QVG_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return QVG_ERR_UNSUPPORTED;
    if (n == 0 && !accumulate) return QVG_ERR_INVALID_ARG;
    return launch_query_stats(static_cast<const uint16_t *>(q_hist_bf16), n, Hq, H, d, accumulate, M, w,
                              count, static_cast<cudaStream_t>(stream));
}

qvg_status quantwm_psac_basis(const float *M, const int64_t *count, int32_t H, int32_t d,
                              int32_t rank, float *U, float *eigvals, float *energy_frac,
                              void *stream) {
    if (!M || !count || !U || !eigvals || !energy_frac || H < 1) return QVG_ERR_INVALID_ARG;
    if (rank != QVG_PSAC_RANK) return QVG_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return QVG_ERR_UNSUPPORTED;
    return launch_psac_basis(M, count, H, d, rank, U, eigvals, energy_frac,
                             static_cast<cudaStream_t>(stream));
}

const char *qvg_last_cuda_error(void) { return cudaGetErrorName(t_last_cuda_error); }

qvg_status qvg_debug_set_wait(uint64_t limit_ns, int32_t inject) {
    if (inject != 0 && inject != 1) return QVG_ERR_INVALID_ARG;
    t_wait_ns = limit_ns == 0 ? kDefaultWaitNs : limit_ns;
    t_wait_inject = inject;
    return QVG_OK;
}

qvg_status qvg_get_status(void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = st ? cudaStreamSynchronize(st) : cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        note_cuda_error(e);
        return QVG_ERR_CUDA;
    }
    int *word = device_error_word();
    if (!word) return QVG_ERR_CUDA;
    int err = 0;
    e = cudaMemcpyAsync(&err, word, sizeof(int), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess && err != 0) {
        e = cudaMemsetAsync(word, 0, sizeof(int), st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        note_cuda_error(e);
        return QVG_ERR_CUDA;
    }
    return static_cast<qvg_status>(err);
}

}  // extern "C"
