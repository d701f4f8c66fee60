// attention_ws.cu -- the host side of the fused attention: launch
// configuration, the cache split for few queries and its log-sum-exp merge
// kernel, and the d = 128 instantiations of the kernel declared in
// attention_ws.cuh (the d = 64 ones compile in attention_ws_d64.cu, in
// parallel).
#include "attention_ws.cuh"

namespace qvg {

extern template qvg_status attn_ws<64, 2>(const AttnWsArgs &, int, cudaStream_t);
extern template qvg_status attn_ws<64, 4>(const AttnWsArgs &, int, cudaStream_t);

// Split-cache merge: split z produced O_z (normalised, fp32) and its
// log-sum-exp lse_z over its share of the cache; the whole-cache result is
// O = sum_z e^{lse_z - m} O_z / sum_z e^{lse_z - m}, lse = m + log sum_z
// e^{lse_z - m} (m = max_z lse_z), and the top-1 slot is that of the largest
// best logit (the first split on ties, i.e. the lowest slot).  One warp per
// (query, query head), lane = D/32 channels.
template <int D>
__global__ void __launch_bounds__(256) k_attn_merge(const float *__restrict__ po, const float *__restrict__ plse,
                                                   const float *__restrict__ pbest, const int32_t *__restrict__ parg,
                                                   int S, int Nq, int Hq, float *__restrict__ out32,
                                                   uint16_t *__restrict__ out16, float *__restrict__ lse,
                                                   int32_t *__restrict__ top1) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (row >= static_cast<long long>(Nq) * Hq) return;
    const int qi = static_cast<int>(row / Hq), hq = static_cast<int>(row % Hq);
    float m = -INFINITY;
    for (int z = 0; z < S; ++z) m = fmaxf(m, plse[(static_cast<size_t>(z) * Hq + hq) * Nq + qi]);
    float acc[E], den = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.0f;
    for (int z = 0; z < S; ++z) {
        const float wz = expf(plse[(static_cast<size_t>(z) * Hq + hq) * Nq + qi] - m);
        const float *oz = po + ((static_cast<size_t>(z) * Nq + qi) * Hq + hq) * D + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(wz, oz[e], acc[e]);
        den += wz;
    }
    const float inv = 1.0f / den;
    const size_t o = (static_cast<size_t>(qi) * Hq + hq) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        if (out32)
            out32[o + e] = acc[e] * inv;
        else
            out16[o + e] = f32_to_bf16(acc[e] * inv);
    }
    if (lane == 0) {
        if (lse) lse[static_cast<size_t>(hq) * Nq + qi] = m + logf(den);
        if (top1) {
            float bb = -INFINITY;
            int arg = 0;
            for (int z = 0; z < S; ++z) {
                const size_t li = (static_cast<size_t>(z) * Hq + hq) * Nq + qi;
                if (pbest[li] > bb) {
                    bb = pbest[li];
                    arg = parg[li];
                }
            }
            top1[static_cast<size_t>(hq) * Nq + qi] = arg;
        }
    }
}

static int attn_sm_count() { return sm_count_current(); }

// Number of cache splits: when (query blocks x query heads) CTAs leave SMs
// idle, each (block, head) pair is split over as many CTAs as fill the SMs
// once (one CTA per SM: the kernel's shared and tensor memory allow no
// more, and a second wave would pay every split's pipeline start again),
// with at least kMinSplitTiles cache tiles per split, at most kMaxSplits.
constexpr int kMaxSplits = 32, kMinSplitTiles = 4;
int attention_splits(int Nq, int Hq, int n_tiles) {
    const int ctas = ceil_div(std::max(Nq, 1), 256) * Hq;
    const int sm = attn_sm_count();
    if (ctas >= sm) return 1;
    int s = std::min(kMaxSplits, sm / ctas);
    if (n_tiles >= 0) s = std::min(s, std::max(1, n_tiles / kMinSplitTiles));
    return std::max(1, s);
}

size_t attention_split_bytes(int Nq, int Hq, int d, int splits) {
    if (splits <= 1) return 0;
    const size_t rows = static_cast<size_t>(splits) * Nq * Hq;
    // O (fp32, d) + lse + best logit + best slot per (split, query, head), 256-byte aligned parts
    auto al = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
    return al(rows * d * 4) + 3 * al(rows * 4);
}

qvg_status launch_attention_ws(const qvg_params *p, const uint16_t *q, int Nq, int Hq, const qvg_cache *k,
                               const qvg_cache *v, float scale_log2, const uint16_t *k_cur, const uint16_t *v_cur,
                               int n_cur, void *out, int out_dtype, float *lse, int32_t *top1, void *workspace,
                               size_t ws_bytes, cudaStream_t st) {
    AttnWsArgs a{};
    a.q = q;
    a.Nq = Nq;
    a.Hq = Hq;
    a.H = k->H;
    a.grp = Hq / k->H;
    a.L = p->L;
    a.C = p->C;
    a.group = p->group;
    a.glog2 = __builtin_ctz(static_cast<unsigned>(p->group));  // a power of two (check_params)
    a.cap = k->capacity_tokens;
    a.max_chunks = k->max_chunks;
    a.n_slots = k->n_tokens;
    a.n_ctiles = k->n_tokens / QVG_TILE;
    a.kraw = k_cur;
    a.vraw = v_cur;
    a.n_raw = n_cur;
    a.kcodes = k->codes;
    a.vcodes = v->codes;
    a.kscales = k->scales;
    a.vscales = v->scales;
    a.kids = k->ids;
    a.vids = v->ids;
    a.kcent = k->cent;
    a.vcent = v->cent;
    a.chunk_start = k->chunk_start;
    a.chunk_len = k->chunk_len;
    a.tile_chunk = k->tile_chunk;
    const bool psac = (p->flags & QVG_PSAC) && k->psac_p;
    a.psac_p = psac ? k->psac_p : nullptr;
    a.psac_s = k->psac_s;
    a.psac_basis = k->psac_basis;
    if (p->anchor_every > 0) {
        a.kanch = k->anchor;
        a.vanch = v->anchor;
        a.chunk_anchor = k->chunk_anchor;
    }
    if (p->flags & QVG_OUTLIER) {
        a.koutv = k->outl_val;
        a.kouti = k->outl_idx;
        a.voutv = v->outl_val;
        a.vouti = v->outl_idx;
    }
    a.scale_log2 = scale_log2;
    a.out32 = out_dtype == QVG_OUT_F32 ? static_cast<float *>(out) : nullptr;
    a.out16 = out_dtype == QVG_OUT_BF16 ? static_cast<uint16_t *>(out) : nullptr;
    a.lse = lse;
    a.top1 = top1;
    a.err = device_error_word();
    a.wait_ns = wait_limit_ns();
    a.inject = wait_inject();
    if (Nq == 0) return QVG_OK;
    const int d = k->d;
    // split the cache over more CTAs when the query blocks alone leave SMs idle
    // (needs the workspace qvg_workspace_size reports for this Nq, Hq, d)
    int splits = attention_splits(Nq, Hq, a.n_ctiles + ceil_div(n_cur, QVG_TILE));
    if (splits > 1 && (!workspace || ws_bytes < attention_split_bytes(Nq, Hq, d, splits))) splits = 1;
    float *po = nullptr, *plse = nullptr, *pbest = nullptr;
    int32_t *parg = nullptr;
    if (splits > 1) {
        const size_t rows = static_cast<size_t>(splits) * Nq * Hq;
        auto al = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
        char *base = static_cast<char *>(workspace);
        po = reinterpret_cast<float *>(base);
        plse = reinterpret_cast<float *>(base + al(rows * d * 4));
        pbest = reinterpret_cast<float *>(base + al(rows * d * 4) + al(rows * 4));
        parg = reinterpret_cast<int32_t *>(base + al(rows * d * 4) + 2 * al(rows * 4));
        a.out32 = po;
        a.out16 = nullptr;
        a.lse = plse;
        a.top1 = top1 ? parg : nullptr;
        a.best = top1 ? pbest : nullptr;
    }
    qvg_status s;
    if (d == 64)
        s = p->bits == 2 ? attn_ws<64, 2>(a, splits, st) : attn_ws<64, 4>(a, splits, st);
    else
        s = p->bits == 2 ? attn_ws<128, 2>(a, splits, st) : attn_ws<128, 4>(a, splits, st);
    if (s != QVG_OK || splits == 1) return s;
    const long long rows = static_cast<long long>(Nq) * Hq;
    const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
    float *o32 = out_dtype == QVG_OUT_F32 ? static_cast<float *>(out) : nullptr;
    uint16_t *o16 = out_dtype == QVG_OUT_BF16 ? static_cast<uint16_t *>(out) : nullptr;
    if (d == 64)
        k_attn_merge<64><<<blocks, 256, 0, st>>>(po, plse, pbest, parg, splits, Nq, Hq, o32, o16, lse, top1);
    else
        k_attn_merge<128><<<blocks, 256, 0, st>>>(po, plse, pbest, parg, splits, Nq, Hq, o32, o16, lse, top1);
    QVG_LAUNCH_CHECK();
    return QVG_OK;
}

}  // namespace qvg
