// attention_tc.cu -- tensor-core attention over the compressed KV cache
// (sm_103a, tcgen05 + TMEM).
//
// Quant VideoGen notes, "algorithm-system co-design": dequantisation fused
// with attention, packed INT2 codes.  Per CTA: 128 query rows of one query
// head; the cache is streamed in tiles of 128 slots.  For each tile:
//   1. rebuild K_hat and V_hat in shared memory from codes, fp16 scales,
//      cluster ids and bf16 centroids (fp32 arithmetic in stage order, plus
//      the PSAC correction on K), never writing them to global memory:
//      K_hat as an fp16 pair hi + lo (hi = fp16(K_hat), lo = fp16(K_hat - hi),
//      22 significant bits), V_hat as fp16;
//   2. S = Q K_hi^T + Q K_lo^T on the tensor cores (tcgen05.mma kind::f16,
//      M=128, N=128, fp32 accumulators in TMEM); Q is fp16 (exact for bf16
//      queries in fp16's normal range);
//   3. online softmax in base 2, one thread per query row reading its row of
//      S from TMEM; P = exp2(s - m) rounded to fp16; the running maximum m is
//      raised only when the tile maximum exceeds it by more than 8 (then O is
//      rescaled in TMEM), so P <= 2^8;
//   4. O += P V on the tensor cores (accumulated in TMEM).
// The row sum l adds the fp16-rounded P values the MMA uses.  At the end
// O / l is written, with the log-sum-exp and the top-1 slot.
#include <algorithm>

#include "common.cuh"
#include "umma.cuh"

namespace qvg {

struct AttnTcArgs {
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
    int *err;
};

constexpr uint64_t kAttnWaitNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Code of channel j in a packed row (offset binary).
template <int BITS>
__device__ __forceinline__ int code_of(const uint8_t *row, int j) {
    const uint32_t u = (static_cast<uint32_t>(row[(j * BITS) >> 3]) >> ((j * BITS) & 7)) & ((1u << BITS) - 1u);
    return static_cast<int>(u) - (1 << (BITS - 1));
}

// Reconstruct channels [j0, j0 + NJ) of one slot, fp32, stages in order
// (the same operation order as the standalone reconstruction).
template <int D, int BITS, int NJ>
__device__ __forceinline__ void rebuild_slot(const AttnTcArgs &a, const uint8_t *codes, const uint16_t *scales,
                                             const uint8_t *ids, const uint16_t *cent, int h, int chunk,
                                             int slot, int j0, bool psac, float (&acc)[NJ]) {
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
            float v = __fmul_rn(Sp, static_cast<float>(code_of<BITS>(crow, j)));
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
        for (int k = 0; k < QVG_PSAC_RANK; ++k) pk[k] = pSp * static_cast<float>(a.psac_p[prow * QVG_PSAC_RANK + k]);
#pragma unroll
        for (int e = 0; e < NJ; ++e) {
            float corr = 0.0f;
#pragma unroll
            for (int k = 0; k < QVG_PSAC_RANK; ++k) corr = fmaf(pk[k], U[(j0 + e) * QVG_PSAC_RANK + k], corr);
            acc[e] = acc[e] + corr;
        }
    }
}

template <int D, int BITS>
__global__ void __launch_bounds__(256, 1) k_attention_tc(AttnTcArgs a) {
    constexpr int KB = D / 64;           // 64-channel K blocks of Q / K
    constexpr int QBYTES = KB * 16384;   // 128 rows x D fp16
    constexpr int VBYTES = D * 256;      // D rows x 128 slots fp16
    constexpr int DS = D / 8;            // V channels per producer thread
    extern __shared__ __align__(1024) uint8_t sm_raw[];
    uint8_t *sm = sm_raw + ((1024u - (umma::smem_u32(sm_raw) & 1023u)) & 1023u);
    uint8_t *Qs = sm;
    uint8_t *Khi = Qs + QBYTES;
    uint8_t *Klo = Khi + QBYTES;
    uint8_t *Vt = Klo + QBYTES;  // P (128 x 128 fp16) later reuses Khi (+ Klo when D = 64)
    __shared__ uint64_t bar_s, bar_o;
    __shared__ uint32_t tmem_base;
    __shared__ int fail;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hq = blockIdx.y, h = hq / a.grp, q0 = blockIdx.x * 128;
    const bool psac = a.psac_p != nullptr;

    // Q tile -> fp16, swizzled K-major
    for (int i = tid; i < 128 * (D / 8); i += 256) {
        const int r = i / (D / 8), ci = i % (D / 8), kb = ci >> 3, c = ci & 7;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (q0 + r < a.Nq) {
            const uint4 b = *reinterpret_cast<const uint4 *>(a.q + (static_cast<size_t>(q0 + r) * a.Hq + hq) * D + ci * 8);
            const uint32_t in[4] = {b.x, b.y, b.z, b.w};
            uint32_t o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                o[k] = pack_half2(__uint_as_float(in[k] << 16), __uint_as_float(in[k] & 0xffff0000u));
            v = make_uint4(o[0], o[1], o[2], o[3]);
        }
        *reinterpret_cast<uint4 *>(Qs + kb * 16384 + r * 128 + ((c ^ (r & 7)) << 4)) = v;
    }
    if (warp == 0) {
        umma::tmem_alloc(&tmem_base, 256);
        umma::tmem_relinquish();
    }
    if (tid == 0) {
        umma::mbar_init(&bar_s, 1);
        umma::mbar_init(&bar_o, 1);
        umma::fence_barrier_init();
        fail = 0;
    }
    umma::tc_fence_before();
    __syncthreads();
    umma::tc_fence_after();
    const uint32_t tmem = tmem_base;
    const uint32_t tS = tmem, tO = tmem + 128;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;

    float m_used = -INFINITY, l_sum = 0.0f, best = -INFINITY;
    int best_slot = 0;
    int it = 0;
    const int n_tiles = a.n_slots / QVG_TILE;
    for (int t = 0; t < n_tiles; ++t) {
        const int s0 = t * QVG_TILE;
        const int chunk = a.tile_chunk[t];
        const int nvalid = min(QVG_TILE, max(0, a.chunk_start[chunk] + a.chunk_len[chunk] - s0));
        if (nvalid == 0) continue;
        // (a) the previous PV product must be complete before its operands are overwritten
        if (it > 0) {
            if (tid == 0 && !umma::mbar_wait(&bar_o, (it - 1) & 1, kAttnWaitNs)) fail = 1;
            umma::tc_fence_before();
            __syncthreads();
            umma::tc_fence_after();
            if (fail) break;
        }
        // (b) rebuild the K (hi/lo) and V tiles
        if (warp < 4) {
            const int r = tid;  // slot within the tile
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    float kv[8];
                    if (r < nvalid)
                        rebuild_slot<D, BITS, 8>(a, a.kcodes, a.kscales, a.kids, a.kcent, h, chunk, s0 + r,
                                                 kb * 64 + c8 * 8, psac, kv);
                    else
#pragma unroll
                        for (int e = 0; e < 8; ++e) kv[e] = 0.0f;
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __half h0 = __float2half_rn(kv[2 * e]), h1 = __float2half_rn(kv[2 * e + 1]);
                        hi[e] = static_cast<uint32_t>(__half_as_ushort(h0)) |
                                (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
                        lo[e] = pack_half2(kv[2 * e] - __half2float(h0), kv[2 * e + 1] - __half2float(h1));
                    }
                    const int off = kb * 16384 + r * 128 + ((c8 ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4 *>(Khi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(Klo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
        } else {
            const int u = tid - 128, kg = u >> 3, ds = u & 7;  // slots kg*8.., channels ds*DS..
            uint32_t hv[8][DS / 2];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int r = kg * 8 + k;
                float vv[DS];
                if (r < nvalid)
                    rebuild_slot<D, BITS, DS>(a, a.vcodes, a.vscales, a.vids, a.vcent, h, chunk, s0 + r, ds * DS,
                                              false, vv);
                else
#pragma unroll
                    for (int e = 0; e < DS; ++e) vv[e] = 0.0f;
#pragma unroll
                for (int e = 0; e < DS / 2; ++e) hv[k][e] = pack_half2(vv[2 * e], vv[2 * e + 1]);
            }
            // transpose: channel row j gets the 8 slots kg*8..kg*8+7 (one 16-byte chunk)
#pragma unroll
            for (int e = 0; e < DS; ++e) {
                const int j = ds * DS + e;
                uint32_t w4[4];
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) {
                    const uint32_t a0 = hv[2 * k2][e >> 1], a1 = hv[2 * k2 + 1][e >> 1];
                    const uint32_t lo16 = (e & 1) ? (a0 >> 16) : (a0 & 0xffffu);
                    const uint32_t hi16 = (e & 1) ? (a1 >> 16) : (a1 & 0xffffu);
                    w4[k2] = lo16 | (hi16 << 16);
                }
                const int kb = kg >> 3, c = kg & 7;
                *reinterpret_cast<uint4 *>(Vt + kb * (D * 128) + j * 128 + ((c ^ (j & 7)) << 4)) =
                    make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
        }
        umma::fence_proxy_async_smem();
        umma::tc_fence_before();
        __syncthreads();
        umma::tc_fence_after();
        // (c) S = Q K_hi^T + Q K_lo^T
        if (tid == 0) {
            const uint32_t idesc = umma::idesc_f16(128, 128, 0);
            const uint32_t qa = umma::smem_u32(Qs), kh = umma::smem_u32(Khi), kl = umma::smem_u32(Klo);
#pragma unroll
            for (int s = 0; s < D / 16; ++s) {
                const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                umma::mma_f16(tS, umma::desc_sw128(qa + off), umma::desc_sw128(kh + off), idesc, s != 0);
            }
#pragma unroll
            for (int s = 0; s < D / 16; ++s) {
                const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                umma::mma_f16(tS, umma::desc_sw128(qa + off), umma::desc_sw128(kl + off), idesc, 1);
            }
            umma::mma_commit(&bar_s);
            if (!umma::mbar_wait(&bar_s, it & 1, kAttnWaitNs)) fail = 1;
        }
        umma::tc_fence_before();
        __syncthreads();
        umma::tc_fence_after();
        if (fail) break;
        // (d) softmax rows (warps 0-3); P -> shared memory (reusing K_hi)
        if (warp < 4) {
            const int r = tid;
            float tmax = -INFINITY;
            int targ = 0;
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t v[32];
                umma::tmem_ld32(tS + lane_off + c0, v);
                umma::tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const float s = c0 + k < nvalid ? __uint_as_float(v[k]) * a.scale_log2 : -INFINITY;
                    if (s > tmax) {
                        tmax = s;
                        targ = c0 + k;
                    }
                }
            }
            if (tmax > best) {
                best = tmax;
                best_slot = s0 + targ;
            }
            float corr = 1.0f;
            bool rescale = false;
            if (tmax > m_used + kRescaleThreshold) {
                corr = exp2f(m_used - tmax);  // 0 on the first tile
                rescale = it > 0;
                m_used = tmax;
            }
            float ls = 0.0f;
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t v[32];
                umma::tmem_ld32(tS + lane_off + c0, v);
                umma::tmem_ld_wait();
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int c = c0 + 2 * k;
                    const float p0 = c < nvalid ? exp2f(__uint_as_float(v[2 * k]) * a.scale_log2 - m_used) : 0.0f;
                    const float p1 = c + 1 < nvalid ? exp2f(__uint_as_float(v[2 * k + 1]) * a.scale_log2 - m_used) : 0.0f;
                    pk[k] = pack_half2(p0, p1);
                    const __half2 hp = *reinterpret_cast<const __half2 *>(&pk[k]);
                    ls += __low2float(hp) + __high2float(hp);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int ci = c0 / 8 + i, kb = ci >> 3, c = ci & 7;
                    *reinterpret_cast<uint4 *>(Khi + kb * 16384 + r * 128 + ((c ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
            l_sum = l_sum * corr + ls;
            if (__any_sync(0xffffffffu, rescale)) {
                const float f = rescale ? corr : 1.0f;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t v[32];
                    umma::tmem_ld32(tO + lane_off + c0, v);
                    umma::tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * f);
                    umma::tmem_st32(tO + lane_off + c0, v);
                }
                umma::tmem_st_wait();
            }
        }
        umma::fence_proxy_async_smem();
        umma::tc_fence_before();
        __syncthreads();
        umma::tc_fence_after();
        // (e) O += P V
        if (tid == 0) {
            const uint32_t idesc = umma::idesc_f16(128, D, 0);
            const uint32_t pa = umma::smem_u32(Khi), vb = umma::smem_u32(Vt);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t aoff = (s >> 2) * 16384 + (s & 3) * 32;
                const uint32_t boff = (s >> 2) * (D * 128) + (s & 3) * 32;
                umma::mma_f16(tO, umma::desc_sw128(pa + aoff), umma::desc_sw128(vb + boff), idesc, (it > 0 || s > 0));
            }
            umma::mma_commit(&bar_o);
        }
        ++it;
    }
    // drain the last PV product
    if (it > 0 && !fail) {
        if (tid == 0 && !umma::mbar_wait(&bar_o, (it - 1) & 1, kAttnWaitNs)) fail = 1;
    }
    umma::tc_fence_before();
    __syncthreads();
    umma::tc_fence_after();
    if (fail) {
        if (tid == 0) {
            // record the timeout and let whatever MMA is still in flight drain
            raise_error(a.err, QVG_ERR_TIMEOUT);
            umma::mbar_wait(&bar_s, it & 1, kAttnWaitNs);
            if (it > 0) umma::mbar_wait(&bar_o, (it - 1) & 1, kAttnWaitNs);
        }
    } else if (warp < 4) {
        const int r = tid, qi = q0 + r;
        const float inv = 1.0f / l_sum;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t v[32];
            umma::tmem_ld32(tO + lane_off + c0, v);
            umma::tmem_ld_wait();
            if (qi < a.Nq) {
                const size_t o = (static_cast<size_t>(qi) * a.Hq + hq) * D + c0;
                if (a.out32) {
#pragma unroll
                    for (int k = 0; k < 32; k += 4)
                        *reinterpret_cast<float4 *>(a.out32 + o + k) =
                            make_float4(__uint_as_float(v[k]) * inv, __uint_as_float(v[k + 1]) * inv,
                                        __uint_as_float(v[k + 2]) * inv, __uint_as_float(v[k + 3]) * inv);
                } else {
#pragma unroll
                    for (int k = 0; k < 32; k += 8) {
                        uint32_t w4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w4[e] = static_cast<uint32_t>(f32_to_bf16(__uint_as_float(v[k + 2 * e]) * inv)) |
                                    (static_cast<uint32_t>(f32_to_bf16(__uint_as_float(v[k + 2 * e + 1]) * inv)) << 16);
                        *reinterpret_cast<uint4 *>(a.out16 + o + k) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
            }
        }
        if (qi < a.Nq) {
            if (a.lse) a.lse[static_cast<size_t>(hq) * a.Nq + qi] = (m_used + log2f(l_sum)) * 0.69314718055994531f;
            if (a.top1) a.top1[static_cast<size_t>(hq) * a.Nq + qi] = best_slot;
        }
    }
    umma::tc_fence_before();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, 256);
}

template <int D, int BITS>
static qvg_status attn_tc(const AttnTcArgs &a, cudaStream_t st) {
    constexpr size_t smem = 3 * (D / 64) * 16384 + D * 256 + 1024;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_attention_tc<D, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        attr = true;
    }
    dim3 grid(ceil_div(a.Nq, 128), a.Hq);
    k_attention_tc<D, BITS><<<grid, 256, smem, st>>>(a);
    QVG_LAUNCH_CHECK();
    return QVG_OK;
}

qvg_status launch_attention_tc(const qvg_params *p, const uint16_t *q, int Nq, int Hq, const qvg_cache *k,
                               const qvg_cache *v, float scale_log2, void *out, int out_dtype, float *lse,
                               int32_t *top1, cudaStream_t st) {
    AttnTcArgs a{};
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
    a.scale_log2 = scale_log2;
    a.out32 = out_dtype == QVG_OUT_F32 ? static_cast<float *>(out) : nullptr;
    a.out16 = out_dtype == QVG_OUT_BF16 ? static_cast<uint16_t *>(out) : nullptr;
    a.lse = lse;
    a.top1 = top1;
    a.err = device_error_word();
    if (Nq == 0) return QVG_OK;
    if (k->d == 64) return p->bits == 2 ? attn_tc<64, 2>(a, st) : attn_tc<64, 4>(a, st);
    return p->bits == 2 ? attn_tc<128, 2>(a, st) : attn_tc<128, 4>(a, st);
}

}  // namespace qvg
