// attention.cu -- attention that reads the compressed KV cache (sm_103a).
//
// Quant VideoGen notes, "algorithm-system co-design": dequantisation is fused
// into the attention kernel, so the reconstructed K_hat / V_hat
// (S * q + C_id summed over stages, "overall framework" and "Progressive
// Residual Quantization"; plus the PSAC correction P_hat U^T on K, QuantWM
// write-up) only ever exist in shared memory.
//
// O = softmax(scale * Q K_hat^T) V_hat with an online (streaming) softmax in
// base 2 over tiles of 64 cache slots; fp32 throughout.  One CTA per
// (64 queries, query head).
#include <algorithm>

#include "common.cuh"

namespace qvg {

struct AttnArgs {
    const uint16_t *q;
    int Nq, Hq, H, grp, L, C, group, cap, max_chunks, n_slots;
    const uint8_t *kcodes, *vcodes;
    const uint16_t *kscales, *vscales;
    const uint8_t *kids, *vids;
    const uint16_t *kcent, *vcent;
    const int32_t *chunk_start, *chunk_len, *tile_chunk;
    const int8_t *psac_p;
    const uint16_t *psac_s;
    const float *psac_basis;
    float scale_log2;
    float *out32;
    uint16_t *out16;
    float *lse;
    int32_t *top1;
};

template <int BITS>
__device__ __forceinline__ int acode(const uint8_t *row, int j) {
    const uint32_t u = (static_cast<uint32_t>(row[(j * BITS) >> 3]) >> ((j * BITS) & 7)) &
                       ((1u << BITS) - 1u);
    return static_cast<int>(u) - (1 << (BITS - 1));
}

// Rebuild channels [j0, j0 + NJ) of one cache slot (fp32, stage order).
template <int D, int BITS, int NJ>
__device__ __forceinline__ void rebuild(const AttnArgs &a, const uint8_t *codes,
                                        const uint16_t *scales, const uint8_t *ids,
                                        const uint16_t *cent, int h, int chunk, int slot, int j0,
                                        bool psac, float (&acc)[NJ]) {
    constexpr int NB = D * BITS / 8;
    const int ng = D / a.group;
#pragma unroll
    for (int e = 0; e < NJ; ++e) acc[e] = 0.0f;
    for (int l = 0; l < a.L; ++l) {
        const size_t srow = (static_cast<size_t>(l) * a.H + h) * a.cap + slot;
        const uint8_t *crow = codes + srow * NB;
        const uint16_t *cr = nullptr;
        if (a.C > 0)
            cr = cent + ((static_cast<size_t>(l) * a.H + h) * a.max_chunks + chunk) * a.C * D +
                 static_cast<size_t>(ids[srow]) * D;
#pragma unroll
        for (int e = 0; e < NJ; ++e) {
            const int j = j0 + e;
            const float Sp = f16_to_f32(scales[srow * ng + j / a.group]);
            float v = __fmul_rn(Sp, static_cast<float>(acode<BITS>(crow, j)));
            if (a.C > 0) v = __fadd_rn(v, bf16_to_f32(cr[j]));
            acc[e] = __fadd_rn(acc[e], v);
        }
    }
    if (psac) {
        const size_t prow = static_cast<size_t>(h) * a.cap + slot;
        const float pSp = f16_to_f32(a.psac_s[prow]);
        const float *U = a.psac_basis + (static_cast<size_t>(chunk) * a.H + h) * D * QVG_PSAC_RANK;
        float pk[QVG_PSAC_RANK];
#pragma unroll
        for (int k = 0; k < QVG_PSAC_RANK; ++k)
            pk[k] = pSp * static_cast<float>(a.psac_p[prow * QVG_PSAC_RANK + k]);
#pragma unroll
        for (int e = 0; e < NJ; ++e) {
            float corr = 0.0f;
#pragma unroll
            for (int k = 0; k < QVG_PSAC_RANK; ++k)
                corr = fmaf(pk[k], U[(j0 + e) * QVG_PSAC_RANK + k], corr);
            acc[e] = acc[e] + corr;
        }
    }
}

constexpr int BQ = 64, BK = 64;

template <int D, int BITS>
__global__ void __launch_bounds__(256) k_attention_simt(AttnArgs a) {
    constexpr int NJ = D / 4;     // channels rebuilt per thread
    constexpr int E = D / 32;     // output channels per thread
    constexpr int KTS = BK + 4;   // padded row of the transposed K tile
    extern __shared__ float sm[];
    float *Qs = sm;                       // [BQ][D]
    float *KT = Qs + BQ * D;              // [D][KTS]
    float *Vs = KT + D * KTS;             // [BK][D]
    float *Ps = Vs + BK * D;              // [BQ][BK + 1]
    float *mrow = Ps + BQ * (BK + 1);     // [BQ]
    float *lrow = mrow + BQ;              // [BQ]
    float *crow = lrow + BQ;              // [BQ]
    float *bval = crow + BQ;              // [BQ]
    int *bidx = reinterpret_cast<int *>(bval + BQ);  // [BQ]

    const int tid = threadIdx.x;
    const int hq = blockIdx.y, h = hq / a.grp;
    const int q0 = blockIdx.x * BQ;
    for (int i = tid; i < BQ * D; i += 256) {
        const int r = i / D, j = i % D;
        float v = 0.0f;
        if (q0 + r < a.Nq) v = bf16_to_f32(a.q[(static_cast<size_t>(q0 + r) * a.Hq + hq) * D + j]);
        Qs[i] = v * a.scale_log2;
    }
    if (tid < BQ) {
        mrow[tid] = -INFINITY;
        lrow[tid] = 0.0f;
        bval[tid] = -INFINITY;
        bidx[tid] = 0;
    }
    const int ty = tid >> 4, tx = tid & 15;  // S tile: rows ty*4.., keys tx*4..
    const int py = tid >> 5, px = tid & 31;  // O tile: rows py*8.., channels px*E..
    float O[8][E];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int e = 0; e < E; ++e) O[i][e] = 0.0f;
    const bool psac = a.psac_p != nullptr;
    __syncthreads();

    for (int s0 = 0; s0 < a.n_slots; s0 += BK) {
        const int chunk = a.tile_chunk[s0 / QVG_TILE];
        const int valid = min(BK, max(0, a.chunk_start[chunk] + a.chunk_len[chunk] - s0));
        if (valid == 0) continue;
        {   // rebuild K (transposed) and V tiles
            const int kk = tid >> 2, j0 = (tid & 3) * NJ;
            float kv[NJ];
            if (kk < valid) {
                rebuild<D, BITS, NJ>(a, a.kcodes, a.kscales, a.kids, a.kcent, h, chunk, s0 + kk, j0, psac, kv);
            } else {
#pragma unroll
                for (int e = 0; e < NJ; ++e) kv[e] = 0.0f;
            }
#pragma unroll
            for (int e = 0; e < NJ; ++e) KT[(j0 + e) * KTS + kk] = kv[e];
            if (kk < valid) {
                rebuild<D, BITS, NJ>(a, a.vcodes, a.vscales, a.vids, a.vcent, h, chunk, s0 + kk, j0, false, kv);
            }
#pragma unroll
            for (int e = 0; e < NJ; ++e) Vs[kk * D + j0 + e] = kv[e];
        }
        __syncthreads();
        // S = Q K^T (log2 units)
        float s[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int k = 0; k < 4; ++k) s[i][k] = 0.0f;
        for (int j = 0; j < D; ++j) {
            const float4 kv4 = *reinterpret_cast<const float4 *>(&KT[j * KTS + tx * 4]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float qv = Qs[(ty * 4 + i) * D + j];
                s[i][0] = fmaf(qv, kv4.x, s[i][0]);
                s[i][1] = fmaf(qv, kv4.y, s[i][1]);
                s[i][2] = fmaf(qv, kv4.z, s[i][2]);
                s[i][3] = fmaf(qv, kv4.w, s[i][3]);
            }
        }
        float mnew[4], corr[4], lsum[4], tb[4];
        int ti[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float mx = -INFINITY;
            tb[i] = -INFINITY;
            ti[i] = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (tx * 4 + k >= valid) s[i][k] = -INFINITY;
                mx = fmaxf(mx, s[i][k]);
                if (s[i][k] > tb[i]) { tb[i] = s[i][k]; ti[i] = s0 + tx * 4 + k; }
            }
            for (int o = 8; o > 0; o >>= 1) {
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float ov = __shfl_xor_sync(0xffffffffu, tb[i], o);
                const int oi = __shfl_xor_sync(0xffffffffu, ti[i], o);
                if (ov > tb[i] || (ov == tb[i] && oi < ti[i])) { tb[i] = ov; ti[i] = oi; }
            }
            const float mold = mrow[ty * 4 + i];
            mnew[i] = fmaxf(mold, mx);
            corr[i] = exp2f(mold - mnew[i]);
            float ls = 0.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                s[i][k] = exp2f(s[i][k] - mnew[i]);
                ls += s[i][k];
            }
            for (int o = 8; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
            lsum[i] = ls;
        }
        __syncthreads();  // every thread has read mrow
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty * 4 + i;
#pragma unroll
            for (int k = 0; k < 4; ++k) Ps[r * (BK + 1) + tx * 4 + k] = s[i][k];
            if (tx == 0) {
                lrow[r] = lrow[r] * corr[i] + lsum[i];
                mrow[r] = mnew[i];
                crow[r] = corr[i];
                if (tb[i] > bval[r]) { bval[r] = tb[i]; bidx[r] = ti[i]; }
            }
        }
        __syncthreads();
        // O = O * corr + P V
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float c = crow[py * 8 + i];
#pragma unroll
            for (int e = 0; e < E; ++e) O[i][e] *= c;
        }
        for (int k = 0; k < valid; ++k) {
            float v[E];
#pragma unroll
            for (int e = 0; e < E; ++e) v[e] = Vs[k * D + px * E + e];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float p = Ps[(py * 8 + i) * (BK + 1) + k];
#pragma unroll
                for (int e = 0; e < E; ++e) O[i][e] = fmaf(p, v[e], O[i][e]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = py * 8 + i, qi = q0 + r;
        if (qi >= a.Nq) continue;
        const float inv = 1.0f / lrow[r];
        const size_t o = (static_cast<size_t>(qi) * a.Hq + hq) * D + px * E;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if (a.out32) a.out32[o + e] = O[i][e] * inv;
            else a.out16[o + e] = f32_to_bf16(O[i][e] * inv);
        }
        if (px == 0) {
            if (a.lse) a.lse[static_cast<size_t>(hq) * a.Nq + qi] = (mrow[r] + log2f(lrow[r])) * 0.69314718055994531f;
            if (a.top1) a.top1[static_cast<size_t>(hq) * a.Nq + qi] = bidx[r];
        }
    }
}

template <int D, int BITS>
static qvg_status attn_simt(const AttnArgs &a, cudaStream_t st) {
    const size_t smem = (static_cast<size_t>(BQ) * D + D * (BK + 4) + BK * D + BQ * (BK + 1) + 5 * BQ) * 4;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_attention_simt<D, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        attr = true;
    }
    dim3 grid(ceil_div(a.Nq, BQ), a.Hq);
    k_attention_simt<D, BITS><<<grid, 256, smem, st>>>(a);
    QVG_LAUNCH_CHECK();
    return QVG_OK;
}

qvg_status launch_attention(const qvg_params *p, const uint16_t *q, int Nq, int Hq,
                            const qvg_cache *k, const qvg_cache *v, float scale_log2, void *out,
                            int out_dtype, float *lse, int32_t *top1, cudaStream_t st) {
    AttnArgs a{};
    a.q = q;
    a.Nq = Nq;
    a.Hq = Hq;
    a.H = k->H;
    a.grp = Hq / k->H;
    a.L = p->L;
    a.C = p->C;
    a.group = p->group;
    a.cap = k->capacity_tokens;
    a.max_chunks = k->max_chunks;
    a.n_slots = k->n_tokens;
    a.kcodes = k->codes; a.vcodes = v->codes;
    a.kscales = k->scales; a.vscales = v->scales;
    a.kids = k->ids; a.vids = v->ids;
    a.kcent = k->cent; a.vcent = v->cent;
    a.chunk_start = k->chunk_start;
    a.chunk_len = k->chunk_len;
    a.tile_chunk = k->tile_chunk;
    const bool psac = (p->flags & QVG_PSAC) && k->psac_p;
    a.psac_p = psac ? k->psac_p : nullptr;
    a.psac_s = k->psac_s;
    a.psac_basis = k->psac_basis;
    a.scale_log2 = scale_log2;
    a.out32 = out_dtype == QVG_OUT_F32 ? static_cast<float *>(out) : nullptr;
    a.out16 = out_dtype == QVG_OUT_BF16 ? static_cast<uint16_t *>(out) : nullptr;
    a.lse = lse;
    a.top1 = top1;
    if (Nq == 0) return QVG_OK;
    if (k->d == 64) return p->bits == 2 ? attn_simt<64, 2>(a, st) : attn_simt<64, 4>(a, st);
    return p->bits == 2 ? attn_simt<128, 2>(a, st) : attn_simt<128, 4>(a, st);
}

}  // namespace qvg
