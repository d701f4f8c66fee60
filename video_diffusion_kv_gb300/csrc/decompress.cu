// decompress.cu -- rebuild K_hat / V_hat from the compressed cache (sm_103a).
//
// Quant VideoGen notes, "overall framework": X_hat = S_X * X_INT + C_i;
// "Progressive Residual Quantization": X_hat = X_hat_1 + Delta_hat_1 + ...
// (stages summed in fp32 in stage order).  QuantWM write-up, PSAC: the
// stored projection of the key error is added back as P_hat U^T.
// "Temporally stable 2-bit KV-cache compression for video world models, in practice"
// (hmyw.cn), section 3.4 (outlier separation): a value split off from its
// group is rebuilt from its fp16 copy; section 3.3 (temporal anchors): an
// anchor chunk's values are its stored bf16 K/V.
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
    const uint16_t *outl_val;
    const uint8_t *outl_idx;
    const uint16_t *anchor;
    const int32_t *chunk_anchor;
    int H, cap, max_chunks;
};

// Thread = token slot: a warp rebuilds 32 consecutive slots of one head
// (their codes, scales and ids are contiguous), each thread its own row in
// blocks of 32 channels (the block's codes, scales and centroid piece are
// loaded before its arithmetic); the block's 32 x 32 results are stored
// row by row through shared memory.  Per element, in stage order:
// acc += fl(fl(S q) + c), then the PSAC term as an fp32 FMA chain over the
// rank -- the same operations, in the same order, as any other rebuild.
// OUTL: at the channel a stage split off from its group (code 0), the
// stage's value is fl(o + c), o the stored fp16 outlier.
template <int D, int BITS, bool PSAC, bool OUTL>
__global__ void __launch_bounds__(256, (PSAC || OUTL) ? 2 : 3) k_decompress(CacheView cv, int L, int C, int group,
                                                   int tok0, int ntok, float *out32,
                                                   uint16_t *out16) {
    constexpr int NB = D * BITS / 8, CB = 32 * BITS / 8;  // code bytes per row / per 32-channel block
    const int lane = threadIdx.x & 31;
    const int H = cv.H, ng = D / group;
    const int nblk = ceil_div(ntok, 32);
    const long long wid = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (wid >= static_cast<long long>(H) * nblk) return;
    // t0 < ntok (nblk = ceil(ntok / 32)); a lane past the end decodes nothing
    // and takes part only in the warp's staged stores
    const int h = static_cast<int>(wid / nblk), t0 = static_cast<int>(wid % nblk) * 32, t = t0 + lane;
    const bool live = t < ntok;
    const int nrow = min(32, ntok - t0);
    const int slot = tok0 + (live ? t : t0);
    const int chunk = cv.tile_chunk[slot / QVG_TILE];
    const bool valid = live && slot >= cv.chunk_start[chunk] && slot < cv.chunk_start[chunk] + cv.chunk_len[chunk];
    const int arow = cv.chunk_anchor ? cv.chunk_anchor[chunk] : -1;  // an anchor chunk's first row, or -1
    const uint16_t *arow_p = arow >= 0 && valid ? cv.anchor + (static_cast<size_t>(arow + slot - cv.chunk_start[chunk]) * H + h) * D
                                                : nullptr;
    float pk[QVG_PSAC_RANK];
    const float *U = nullptr;
    if (PSAC && valid && !arow_p) {
        const size_t prow = static_cast<size_t>(h) * cv.cap + slot;
        const float pSp = f16_to_f32(cv.psac_s[prow]);
#pragma unroll
        for (int k = 0; k < QVG_PSAC_RANK; ++k) pk[k] = pSp * static_cast<float>(cv.psac_p[prow * QVG_PSAC_RANK + k]);
        U = cv.psac_basis + (static_cast<size_t>(chunk) * H + h) * D * QVG_PSAC_RANK;
    }
    // the warp's 32 rows x 32 channels pass through shared memory (one row
    // per lane in, one row per store out), so that each store instruction
    // writes whole 128-byte lines instead of 16 bytes of 32 lines
    __shared__ float stage[8][32][33];
    float (*st)[33] = stage[threadIdx.x >> 5];
    uint32_t (*st16)[17] = reinterpret_cast<uint32_t (*)[17]>(&stage[threadIdx.x >> 5][0][0]);
#pragma unroll 1
    for (int cb = 0; cb < D / 32; ++cb) {
        float acc[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] = 0.0f;
        if (arow_p) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 u = *reinterpret_cast<const uint4 *>(arow_p + cb * 32 + 8 * i);
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    acc[8 * i + 2 * k] = __uint_as_float(w4[k] << 16);
                    acc[8 * i + 2 * k + 1] = __uint_as_float(w4[k] & 0xffff0000u);
                }
            }
        } else if (valid) {
            for (int l = 0; l < L; ++l) {
                const size_t srow = (static_cast<size_t>(l) * H + h) * cv.cap + slot;
                uint32_t cw[CB / 4];
                if constexpr (CB == 8) {
                    const uint2 u = *reinterpret_cast<const uint2 *>(cv.codes + srow * NB + cb * CB);
                    cw[0] = u.x;
                    cw[1] = u.y;
                } else {
                    const uint4 u = *reinterpret_cast<const uint4 *>(cv.codes + srow * NB + cb * CB);
                    cw[0] = u.x;
                    cw[1] = u.y;
                    cw[2] = u.z;
                    cw[3] = u.w;
                }
                float S[4], ov[4];
                int oc[4];  // channel split off in each 8-channel block's group, or -1
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    const int gi = (cb * 32 + g8 * 8) / group;
                    S[g8] = f16_to_f32(cv.scales[srow * ng + gi]);
                    oc[g8] = -1;
                    ov[g8] = 0.0f;
                    if constexpr (OUTL) {
                        const int oi = cv.outl_idx[srow * ng + gi];
                        if (oi != 0xFF) {
                            oc[g8] = gi * group + oi;
                            ov[g8] = f16_to_f32(cv.outl_val[srow * ng + gi]);
                        }
                    }
                }
                uint4 cr[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                               make_uint4(0, 0, 0, 0)};
                if (C > 0) {
                    const uint16_t *crow = cv.cent + ((static_cast<size_t>(l) * H + h) * cv.max_chunks + chunk) * C * D +
                                           static_cast<size_t>(cv.ids[srow]) * D + cb * 32;
#pragma unroll
                    for (int i = 0; i < 4; ++i) cr[i] = *reinterpret_cast<const uint4 *>(crow + 8 * i);
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const uint32_t word = cw[(e * BITS) / 32];
                    const int q = static_cast<int>((word >> ((e * BITS) % 32)) & ((1u << BITS) - 1u)) - (1 << (BITS - 1));
                    float v = __fmul_rn(S[e >> 3], static_cast<float>(q));
                    if (OUTL && cb * 32 + e == oc[e >> 3]) v = ov[e >> 3];
                    if (C > 0) {
                        const uint4 c4 = cr[e >> 3];
                        const uint32_t cwd = (e & 7) < 2 ? c4.x : (e & 7) < 4 ? c4.y : (e & 7) < 6 ? c4.z : c4.w;
                        v = __fadd_rn(v, __uint_as_float((e & 1) ? (cwd & 0xffff0000u) : (cwd << 16)));
                    }
                    acc[e] = __fadd_rn(acc[e], v);
                }
            }
            if (U) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float *u = U + (cb * 32 + e) * QVG_PSAC_RANK;
                    float corr = 0.0f;
#pragma unroll
                    for (int k = 0; k < QVG_PSAC_RANK; ++k) corr = fmaf(pk[k], u[k], corr);
                    acc[e] = acc[e] + corr;
                }
            }
        }
        if (out32) {
#pragma unroll
            for (int e = 0; e < 32; ++e) st[lane][e] = acc[e];
            __syncwarp();
            float *o = out32 + (static_cast<size_t>(t0) * H + h) * D + cb * 32 + lane;
            for (int r = 0; r < nrow; ++r) o[static_cast<size_t>(r) * H * D] = st[r][lane];
        } else {
#pragma unroll
            for (int k = 0; k < 16; ++k)
                st16[lane][k] = static_cast<uint32_t>(f32_to_bf16(acc[2 * k])) |
                                (static_cast<uint32_t>(f32_to_bf16(acc[2 * k + 1])) << 16);
            __syncwarp();
            // two rows per store: lanes 0-15 the even row, 16-31 the odd one
            uint32_t *o = reinterpret_cast<uint32_t *>(out16 + (static_cast<size_t>(t0) * H + h) * D + cb * 32) +
                          (lane & 15);
            for (int r = lane >> 4; r < nrow; r += 2) o[static_cast<size_t>(r) * H * D / 2] = st16[r][lane & 15];
        }
        __syncwarp();  // the stage is read before the next block overwrites it
    }
}

qvg_status launch_decompress(const qvg_params *p, const qvg_cache *c, int tok0, int ntok,
                             void *out, int out_dtype, cudaStream_t st) {
    CacheView cv{c->codes, c->scales, c->ids, c->cent, c->chunk_start, c->chunk_len,
                 c->tile_chunk, c->psac_p, c->psac_s, c->psac_basis, c->outl_val, c->outl_idx, c->anchor,
                 c->chunk_anchor, c->H, c->capacity_tokens, c->max_chunks};
    if (p->anchor_every <= 0) cv.chunk_anchor = nullptr;
    if (!(p->flags & QVG_PSAC)) cv.psac_p = nullptr;
    if (!(p->flags & QVG_OUTLIER)) cv.outl_idx = nullptr;
    float *o32 = out_dtype == QVG_OUT_F32 ? static_cast<float *>(out) : nullptr;
    uint16_t *o16 = out_dtype == QVG_OUT_BF16 ? static_cast<uint16_t *>(out) : nullptr;
    const long long warps = static_cast<long long>(c->H) * ceil_div(std::max(ntok, 1), 32);
    const int blocks = static_cast<int>(std::max(1LL, (warps + 7) / 8));
#define QVG_DQ2(D_, B_, O_)                                                                                        \
    (cv.psac_p ? k_decompress<D_, B_, true, O_><<<blocks, 256, 0, st>>>(cv, p->L, p->C, p->group, tok0, ntok, o32, o16) \
               : k_decompress<D_, B_, false, O_><<<blocks, 256, 0, st>>>(cv, p->L, p->C, p->group, tok0, ntok, o32, o16))
#define QVG_DQ(D_, B_) (cv.outl_idx ? QVG_DQ2(D_, B_, true) : QVG_DQ2(D_, B_, false))
    if (c->d == 64) {
        if (p->bits == 2) QVG_DQ(64, 2); else QVG_DQ(64, 4);
    } else {
        if (p->bits == 2) QVG_DQ(128, 2); else QVG_DQ(128, 4);
    }
#undef QVG_DQ
#undef QVG_DQ2
    QVG_LAUNCH_CHECK();
    return QVG_OK;
}

}  // namespace qvg
