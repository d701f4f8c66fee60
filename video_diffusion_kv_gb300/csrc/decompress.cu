// decompress.cu -- rebuild K_hat / V_hat from the compressed cache (sm_103a).
//
// Quant VideoGen notes, "overall framework": X_hat = S_X * X_INT + C_i;
// "Progressive Residual Quantization": X_hat = X_hat_1 + Delta_hat_1 + ...
// (stages summed in fp32 in stage order).  QuantWM write-up, PSAC: the
// stored projection of the key error is added back as P_hat U^T.
#include "common.cuh"

namespace qvg {

struct CacheView {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint8_t *ids;
    const uint16_t *cent;
    const int32_t *chunk_start, *chunk_len, *tile_chunk;
    const int8_t *psac_p;
    const uint16_t *psac_s;
    const float *psac_basis;
    int H, cap, max_chunks;
};

// Code of channel j of a packed row.
template <int BITS>
__device__ __forceinline__ int code_at(const uint8_t *row, int j) {
    const uint32_t u = (static_cast<uint32_t>(row[(j * BITS) >> 3]) >> ((j * BITS) & 7)) &
                       ((1u << BITS) - 1u);
    return static_cast<int>(u) - (1 << (BITS - 1));
}

template <int D, int BITS>
__global__ void __launch_bounds__(256) k_decompress(CacheView cv, int L, int C, int group,
                                                   int tok0, int ntok, float *out32,
                                                   uint16_t *out16) {
    constexpr int E = D / 32, NB = D * BITS / 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = cv.H, ng = D / group;
    const int nrows = ntok * H;
    for (int row = blockIdx.x * 8 + warp; row < nrows; row += gridDim.x * 8) {
        const int t = row / H, h = row % H, slot = tok0 + t;
        const int chunk = cv.tile_chunk[slot / QVG_TILE];
        const int start = cv.chunk_start[chunk], len = cv.chunk_len[chunk];
        const bool valid = slot >= start && slot < start + len;
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.0f;
        if (valid) {
            for (int l = 0; l < L; ++l) {
                const size_t srow = (static_cast<size_t>(l) * H + h) * cv.cap + slot;
                const uint8_t *crow = cv.codes + srow * NB;
                const float Sp = f16_to_f32(cv.scales[srow * ng + (lane * E) / group]);
                const uint16_t *cr = nullptr;
                if (C > 0)
                    cr = cv.cent + ((static_cast<size_t>(l) * H + h) * cv.max_chunks + chunk) * C * D +
                         static_cast<size_t>(cv.ids[srow]) * D;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int j = lane * E + e;
                    float v = __fmul_rn(Sp, static_cast<float>(code_at<BITS>(crow, j)));
                    if (C > 0) v = __fadd_rn(v, bf16_to_f32(cr[j]));
                    acc[e] = __fadd_rn(acc[e], v);
                }
            }
            if (cv.psac_p) {
                const size_t prow = static_cast<size_t>(h) * cv.cap + slot;
                const float pSp = f16_to_f32(cv.psac_s[prow]);
                const float *U = cv.psac_basis + (static_cast<size_t>(chunk) * H + h) * D * QVG_PSAC_RANK;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int j = lane * E + e;
                    float corr = 0.0f;
#pragma unroll
                    for (int k = 0; k < QVG_PSAC_RANK; ++k)
                        corr = fmaf(pSp * static_cast<float>(cv.psac_p[prow * QVG_PSAC_RANK + k]),
                                    U[j * QVG_PSAC_RANK + k], corr);
                    acc[e] = acc[e] + corr;
                }
            }
        }
        const size_t o = static_cast<size_t>(row) * D + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if (out32) out32[o + e] = acc[e];
            else out16[o + e] = f32_to_bf16(acc[e]);
        }
    }
}

qvg_status launch_decompress(const qvg_params *p, const qvg_cache *c, int tok0, int ntok,
                             void *out, int out_dtype, cudaStream_t st) {
    CacheView cv{c->codes, c->scales, c->ids, c->cent, c->chunk_start, c->chunk_len,
                 c->tile_chunk, c->psac_p, c->psac_s, c->psac_basis, c->H,
                 c->capacity_tokens, c->max_chunks};
    if (!(p->flags & QVG_PSAC)) cv.psac_p = nullptr;
    float *o32 = out_dtype == QVG_OUT_F32 ? static_cast<float *>(out) : nullptr;
    uint16_t *o16 = out_dtype == QVG_OUT_BF16 ? static_cast<uint16_t *>(out) : nullptr;
    const int rows = ntok * c->H;
    const int blocks = std::max(1, std::min(ceil_div(rows, 8), 152 * 16));
#define QVG_DQ(D_, B_) k_decompress<D_, B_><<<blocks, 256, 0, st>>>(cv, p->L, p->C, p->group, tok0, ntok, o32, o16)
    if (c->d == 64) {
        if (p->bits == 2) QVG_DQ(64, 2); else QVG_DQ(64, 4);
    } else {
        if (p->bits == 2) QVG_DQ(128, 2); else QVG_DQ(128, 4);
    }
#undef QVG_DQ
    QVG_LAUNCH_CHECK();
    return QVG_OK;
}

}  // namespace qvg
