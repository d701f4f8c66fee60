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

// Thread = (token slot, 32 channels): D / 32 threads (TPR) rebuild one row
// of one head, and each owns eight 4-channel pieces interleaved with the
// row's other threads (piece i + TPR m, m = 0..7, for thread i), so that the
// m-th store of the row's TPR threads writes 4 TPR contiguous channels --
// whole 32-byte sectors -- and every store instruction of a warp is fully
// used.  The row's packed codes are read whole by each of its threads (one
// to four 16-byte loads) and the pieces' codes picked out of them.  A block
// takes consecutive slots of one head, whose codes, scales and ids are
// contiguous; the heads vary fastest over the blocks.  A row costs two
// dependent memory round trips per stage: first what depends on the slot
// alone (tile table entry, codes, scales,
// id, outlier entries), then what needs the chunk (its start, length and
// anchor row, the centroid pieces).  Per element, in stage order:
// acc += fl(fl(S q) + c), then the PSAC term as an fp32 FMA chain over the
// rank -- the same operations, in the same order, as any other rebuild.
// OUTL: at the channel a stage split off from its group (code 0), the
// stage's value is fl(o + c), o the stored fp16 outlier.  VEC: the output is
// 16-byte (fp32) or 8-byte (bf16) aligned and each piece takes one vector
// store; otherwise 32-bit stores.
template <int D, int BITS>
struct RowStage {
    static constexpr int NW = D * BITS / 32;  // 32-bit words of packed codes per row
    uint32_t w[NW];
    float S[8], ov[8];
    int oc[8];  // channel split off in each piece's group, or -1
    int id;
};

template <int D, int BITS, bool OUTL>
__device__ __forceinline__ void load_row_stage(const CacheView &cv, int l, int h, int slot, int i, int group,
                                               bool want_id, RowStage<D, BITS> &rs) {
    constexpr int TPR = D / 32, NB = D * BITS / 8;
    const int glog = __ffs(group) - 1;  // groups are powers of two: shifts, not divisions
    const int ng = D >> glog;
    const size_t srow = (static_cast<size_t>(l) * cv.H + h) * cv.cap + slot;
    const uint4 *cp = reinterpret_cast<const uint4 *>(cv.codes + srow * NB);
#pragma unroll
    for (int k = 0; k < NB / 16; ++k) {
        const uint4 u = cp[k];
        rs.w[4 * k] = u.x;
        rs.w[4 * k + 1] = u.y;
        rs.w[4 * k + 2] = u.z;
        rs.w[4 * k + 3] = u.w;
    }
    const uint16_t *sp = cv.scales + srow * ng;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const int g = (4 * (i + TPR * m)) >> glog;
        rs.S[m] = f16_to_f32(sp[g]);
        rs.oc[m] = -1;
        rs.ov[m] = 0.0f;
        if constexpr (OUTL) {
            const int oi = cv.outl_idx[srow * ng + g];
            if (oi != 0xFF) {
                rs.oc[m] = g * group + oi;
                rs.ov[m] = f16_to_f32(cv.outl_val[srow * ng + g]);
            }
        }
    }
    rs.id = want_id ? cv.ids[srow] : 0;
}

// The 4 codes of piece m of thread i (channels 4 (i + TPR m) .. + 3), as
// the low 4 BITS bits of the result.
template <int D, int BITS>
__device__ __forceinline__ uint32_t piece_codes(const RowStage<D, BITS> &rs, int i, int m) {
    constexpr int TPR = D / 32;
    if constexpr (BITS == 2) {
        // byte i + TPR m of the row: word TPR m / 4, byte i + (TPR m mod 4)
        return (rs.w[(TPR * m) >> 2] >> (8 * (i + ((TPR * m) & 3)))) & 0xffu;
    } else {
        // 16-bit half i + TPR m: word (i + TPR m) / 2, half (i + TPR m) mod 2
        const int hw = i + TPR * m;
        const uint32_t word = (TPR == 4) ? ((i >> 1) ? rs.w[2 * m + 1] : rs.w[2 * m]) : rs.w[(TPR * m) >> 1];
        return (word >> (16 * (hw & 1))) & 0xffffu;
    }
}

// Centroid pieces of stage l: 4 bf16 channels each.  The id is clamped so
// that a padding slot (whose id is not a cluster) still reads inside the
// chunk's centroids -- its values are then discarded.
template <int D>
__device__ __forceinline__ void load_cent_row(const CacheView &cv, int l, int h, int chunk, int C, int id, int i,
                                              uint2 (&cr)[8]) {
    constexpr int TPR = D / 32;
    const int idc = id < C ? id : C - 1;
    const uint16_t *crow = cv.cent + ((static_cast<size_t>(l) * cv.H + h) * cv.max_chunks + chunk) * C * D +
                           static_cast<size_t>(idc) * D;
#pragma unroll
    for (int m = 0; m < 8; ++m) cr[m] = *reinterpret_cast<const uint2 *>(crow + 4 * (i + TPR * m));
}

// acc += this stage's values of piece m
template <int D, int BITS, bool OUTL>
__device__ __forceinline__ void add_piece(const RowStage<D, BITS> &rs, uint2 cr, bool cent, int i, int m,
                                          float (&acc)[4]) {
    constexpr int TPR = D / 32;
    const uint32_t code = piece_codes<D, BITS>(rs, i, m);
    const uint32_t cw[2] = {cr.x, cr.y};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int q = static_cast<int>((code >> (k * BITS)) & ((1u << BITS) - 1u)) - (1 << (BITS - 1));
        float v = __fmul_rn(rs.S[m], static_cast<float>(q));
        if (OUTL && 4 * (i + TPR * m) + k == rs.oc[m]) v = rs.ov[m];
        if (cent) v = __fadd_rn(v, __uint_as_float((k & 1) ? (cw[k >> 1] & 0xffff0000u) : (cw[k >> 1] << 16)));
        acc[k] = __fadd_rn(acc[k], v);
    }
}

template <int D, int BITS, bool OUTL>
__device__ __forceinline__ void add_row_stage(const RowStage<D, BITS> &rs, const uint2 (&cr)[8], bool cent, int i,
                                              float (&acc)[8][4]) {
#pragma unroll
    for (int m = 0; m < 8; ++m) add_piece<D, BITS, OUTL>(rs, cr[m], cent, i, m, acc[m]);
}

// The 4 bf16 anchor values of piece m (channels 4 (i + TPR m) .. + 3).
template <int D>
__device__ __forceinline__ void anchor_piece(const uint16_t *ap, int i, int m, float (&o)[4]) {
    constexpr int TPR = D / 32;
    const uint2 u = *reinterpret_cast<const uint2 *>(ap + 4 * (i + TPR * m));
    o[0] = __uint_as_float(u.x << 16);
    o[1] = __uint_as_float(u.x & 0xffff0000u);
    o[2] = __uint_as_float(u.y << 16);
    o[3] = __uint_as_float(u.y & 0xffff0000u);
}

template <int D, bool VEC>
__device__ __forceinline__ void store_piece(float *out32, uint16_t *out16, size_t orow, int i, int m,
                                            const float (&o)[4]) {
    constexpr int TPR = D / 32;
    const size_t off = orow + 4 * (i + TPR * m);
    if (out32) {
        if constexpr (VEC) {
            *reinterpret_cast<float4 *>(out32 + off) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) out32[off + k] = o[k];
        }
    } else {
        const uint32_t w0 = static_cast<uint32_t>(f32_to_bf16(o[0])) | (static_cast<uint32_t>(f32_to_bf16(o[1])) << 16);
        const uint32_t w1 = static_cast<uint32_t>(f32_to_bf16(o[2])) | (static_cast<uint32_t>(f32_to_bf16(o[3])) << 16);
        if constexpr (VEC) {
            *reinterpret_cast<uint2 *>(out16 + off) = make_uint2(w0, w1);
        } else {
            uint32_t *o32 = reinterpret_cast<uint32_t *>(out16 + off);
            o32[0] = w0;
            o32[1] = w1;
        }
    }
}

// MULTI: more than one stage, or the PSAC term; otherwise each piece is
// rebuilt and stored at once, so that few values are live and three blocks
// fit on an SM (two for MULTI, one with the PSAC term, without spills).
template <int D, int BITS, bool PSAC, bool OUTL, bool VEC, bool MULTI>
__global__ void __launch_bounds__(256, PSAC ? 1 : MULTI ? 2 : 3) k_decompress(CacheView cv, int L, int C, int group, int tok0, int ntok,
                                                    float *out32, uint16_t *out16) {
    constexpr int TPR = D / 32, RPB = 256 / TPR;  // threads per row, rows per block
    const int H = cv.H, i = threadIdx.x % TPR;
    // block x: head x % H, slots [(x / H) RPB, + RPB) -- the heads vary
    // fastest, so the blocks in flight write whole token rows of the
    // token-major output
    const int h = static_cast<int>(blockIdx.x % static_cast<unsigned>(H));
    const int t = static_cast<int>(blockIdx.x / static_cast<unsigned>(H)) * RPB + threadIdx.x / TPR;
    if (t >= ntok) return;
    const int slot = tok0 + t;
    // slot-only loads: tile table entry and stage 0
    const int chunk = cv.tile_chunk[slot / QVG_TILE];
    RowStage<D, BITS> rs;
    load_row_stage<D, BITS, OUTL>(cv, 0, h, slot, i, group, C > 0, rs);
    // chunk-dependent loads: the chunk's extent and anchor row, the centroid
    // pieces of stage 0
    const int cs = cv.chunk_start[chunk], cl = cv.chunk_len[chunk];
    const bool valid = slot >= cs && slot < cs + cl;
    int arow = cv.chunk_anchor ? cv.chunk_anchor[chunk] : -1;  // the slot's anchor row, or -1
    if (arow >= 0) arow += slot - cs;
    uint2 cr[8];
    if (C > 0) load_cent_row<D>(cv, 0, h, chunk, C, rs.id, i, cr);
    const size_t orow = (static_cast<size_t>(t) * H + h) * D;
    if constexpr (!MULTI) {
        const uint16_t *ap = valid && arow >= 0 ? cv.anchor + (static_cast<size_t>(arow) * H + h) * D : nullptr;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            float o[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (ap)
                anchor_piece<D>(ap, i, m, o);
            else if (valid)
                add_piece<D, BITS, OUTL>(rs, cr[m], C > 0, i, m, o);
            store_piece<D, VEC>(out32, out16, orow, i, m, o);
        }
    } else {
        float acc[8][4];
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[m][k] = 0.0f;
        add_row_stage<D, BITS, OUTL>(rs, cr, C > 0, i, acc);
#pragma unroll 1
        for (int l = 1; l < L; ++l) {
            load_row_stage<D, BITS, OUTL>(cv, l, h, slot, i, group, C > 0, rs);
            if (C > 0) load_cent_row<D>(cv, l, h, chunk, C, rs.id, i, cr);
            add_row_stage<D, BITS, OUTL>(rs, cr, C > 0, i, acc);
        }
        if (!valid) {
#pragma unroll
            for (int m = 0; m < 8; ++m)
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[m][k] = 0.0f;
        } else if (arow >= 0) {
            // an anchor chunk's row is its stored bf16 K/V
            const uint16_t *ap = cv.anchor + (static_cast<size_t>(arow) * H + h) * D;
#pragma unroll
            for (int m = 0; m < 8; ++m) anchor_piece<D>(ap, i, m, acc[m]);
        } else if constexpr (PSAC) {
            const size_t prow = static_cast<size_t>(h) * cv.cap + slot;
            const float pSp = f16_to_f32(cv.psac_s[prow]);
            const uint2 pu = *reinterpret_cast<const uint2 *>(cv.psac_p + prow * QVG_PSAC_RANK);
            float pk[QVG_PSAC_RANK];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                pk[k] = pSp * static_cast<float>(static_cast<int8_t>(pu.x >> (8 * k)));
                pk[4 + k] = pSp * static_cast<float>(static_cast<int8_t>(pu.y >> (8 * k)));
            }
            const float *U = cv.psac_basis + (static_cast<size_t>(chunk) * H + h) * D * QVG_PSAC_RANK;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float *u = U + (4 * (i + TPR * m) + k) * QVG_PSAC_RANK;
                    const float4 u0 = *reinterpret_cast<const float4 *>(u);
                    const float4 u1 = *reinterpret_cast<const float4 *>(u + 4);
                    const float uu[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
                    float corr = 0.0f;
#pragma unroll
                    for (int r = 0; r < QVG_PSAC_RANK; ++r) corr = fmaf(pk[r], uu[r], corr);
                    acc[m][k] = acc[m][k] + corr;
                }
            }
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) store_piece<D, VEC>(out32, out16, orow, i, m, acc[m]);
    }
}

template <int D, int BITS, bool PSAC, bool OUTL>
void launch_dq(const CacheView &cv, const qvg_params *p, int tok0, int ntok, float *o32, uint16_t *o16, bool vec,
               cudaStream_t st) {
    constexpr int RPB = 256 / (D / 32);
    const dim3 grid(static_cast<unsigned>((ntok + RPB - 1) / RPB) * static_cast<unsigned>(cv.H));
    const int L = p->L, C = p->C, G = p->group;
    if (PSAC || L > 1) {
        if (vec) k_decompress<D, BITS, PSAC, OUTL, true, true><<<grid, 256, 0, st>>>(cv, L, C, G, tok0, ntok, o32, o16);
        else k_decompress<D, BITS, PSAC, OUTL, false, true><<<grid, 256, 0, st>>>(cv, L, C, G, tok0, ntok, o32, o16);
    } else if constexpr (!PSAC) {
        if (vec) k_decompress<D, BITS, false, OUTL, true, false><<<grid, 256, 0, st>>>(cv, L, C, G, tok0, ntok, o32, o16);
        else k_decompress<D, BITS, false, OUTL, false, false><<<grid, 256, 0, st>>>(cv, L, C, G, tok0, ntok, o32, o16);
    }
}

template <int D, int BITS>
void launch_dq_flags(const CacheView &cv, const qvg_params *p, int tok0, int ntok, float *o32, uint16_t *o16, bool vec,
                     cudaStream_t st) {
    if (cv.psac_p) {
        if (cv.outl_idx) launch_dq<D, BITS, true, true>(cv, p, tok0, ntok, o32, o16, vec, st);
        else launch_dq<D, BITS, true, false>(cv, p, tok0, ntok, o32, o16, vec, st);
    } else {
        if (cv.outl_idx) launch_dq<D, BITS, false, true>(cv, p, tok0, ntok, o32, o16, vec, st);
        else launch_dq<D, BITS, false, false>(cv, p, tok0, ntok, o32, o16, vec, st);
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
    // vector stores need each thread's 4-channel piece aligned to its size
    const bool vec = reinterpret_cast<uintptr_t>(out) % (o32 ? 16 : 8) == 0;
    if (c->d == 64) {
        if (p->bits == 2) launch_dq_flags<64, 2>(cv, p, tok0, ntok, o32, o16, vec, st);
        else launch_dq_flags<64, 4>(cv, p, tok0, ntok, o32, o16, vec, st);
    } else {
        if (p->bits == 2) launch_dq_flags<128, 2>(cv, p, tok0, ntok, o32, o16, vec, st);
        else launch_dq_flags<128, 4>(cv, p, tok0, ntok, o32, o16, vec, st);
    }
    QVG_LAUNCH_CHECK();
    return QVG_OK;
}

}  // namespace qvg
