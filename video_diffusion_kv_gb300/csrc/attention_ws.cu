// attention_ws.cu -- warp-specialised tensor-core attention over the
// compressed KV cache (sm_103a: tcgen05.mma, TMEM, mbarriers).
//
// Quant VideoGen notes, "algorithm-system co-design": dequantisation is
// fused with attention and the 2-bit codes stay packed in memory.  The
// reconstructed K_hat = sum_l (S_l q_l + C_l) (+ the PSAC term P_hat U^T of
// the QuantWM write-up) and V_hat only ever exist as fp16 tiles in shared
// memory.
//
// One CTA = two 128-row query tiles of one query head (ping-pong, so the
// tensor core computes one tile's S while the other tile's softmax runs).
// Warp roles (16 warps, 128 registers per thread):
//   0-3, 4-7   softmax + epilogue of query tile 0 / 1 (thread = query row)
//   8-11       K producers: rebuild a 128-slot K_hat tile (thread = slot)
//   12-15      V producers: rebuild V_hat^T (thread = slot, double-buffered);
//              warp 12 owns the TMEM allocation and its lane 0 issues every
//              tcgen05.mma (S_0, S_1 before producing the V tile, which must
//              wait for the previous PV products anyway; PV_0, PV_1 after)
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D),
// O1 [384,384+D), fp32.  Per cache tile t:
//   S_i = Q_i K_t^T              (M=128, N=128 slots, K=D; fp16 operands)
//   P_i = exp2(s * scale*log2e - m_i), fp16, m_i raised lazily (by > 8)
//   O_i += P_i V_t               (M=128, N=D, K=128 slots)
// fp16 operands carry K_hat, V_hat, Q and P with a relative rounding of
// 2^-11; on the synthetic LongCat-like and world-model caches this keeps
// max|dO| / max|O| near 6e-5 against the fp64 oracle.
#include <algorithm>

#include "common.cuh"
#include "umma.cuh"

namespace qvg {

struct AttnWsArgs {
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

namespace ws {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kRescale = 8.0f;

__device__ __forceinline__ uint32_t h2(float a, float b) {
    const __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// 2^x with the hardware approximation (MUFU.EX2, relative error ~2^-22);
// -inf gives 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bounded wait that also gives up as soon as another role has failed.
__device__ __forceinline__ bool wait(uint64_t *bar, uint32_t parity, volatile int *fail) {
    if (umma::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = umma::globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (umma::mbar_try_wait(bar, parity)) return true;
        if (*fail) return false;
        if (umma::globaltimer_ns() - t0 > kWaitNs) {
            *fail = 1;
            return false;
        }
    }
}

struct TileInfo {
    int s0, chunk, nvalid;
};

__device__ __forceinline__ TileInfo tile_info(const AttnWsArgs &a, int t) {
    TileInfo ti;
    ti.s0 = t * QVG_TILE;
    ti.chunk = a.tile_chunk[t];
    ti.nvalid = min(QVG_TILE, max(0, a.chunk_start[ti.chunk] + a.chunk_len[ti.chunk] - ti.s0));
    return ti;
}

// K_hat channels [j0, j0 + 8) of one slot (fp32, stage order, then PSAC).
// The general path (several stages, PSAC): kept out of line so the one-stage
// fast path's loop stays small in the instruction cache.
template <int D, int BITS>
__device__ __noinline__ void rebuild8(const AttnWsArgs &a, const uint8_t *codes, const uint16_t *scales,
                                         const uint8_t *ids, const uint16_t *cent, int h, int chunk, int slot,
                                         int j0, const float *pk, float (&acc)[8]) {
    constexpr int NB = D * BITS / 8;
    const int ng = D / a.group;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    for (int l = 0; l < a.L; ++l) {
        const size_t srow = (static_cast<size_t>(l) * a.H + h) * a.cap + slot;
        const float Sp = f16_to_f32(scales[srow * ng + j0 / a.group]);  // 8 | G: one group
        uint32_t bits;
        if constexpr (BITS == 2)
            bits = *reinterpret_cast<const uint16_t *>(codes + srow * NB + j0 / 4);
        else
            bits = *reinterpret_cast<const uint32_t *>(codes + srow * NB + j0 / 2);
        float c[8];
        if (a.C > 0) {
            const uint4 cv = *reinterpret_cast<const uint4 *>(
                cent + ((static_cast<size_t>(l) * a.H + h) * a.max_chunks + chunk) * a.C * D +
                static_cast<size_t>(ids[srow]) * D + j0);
            const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                c[2 * k] = __uint_as_float(cw[k] << 16);
                c[2 * k + 1] = __uint_as_float(cw[k] & 0xffff0000u);
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int q = static_cast<int>((bits >> (e * BITS)) & ((1u << BITS) - 1u)) - (1 << (BITS - 1));
            float v = __fmul_rn(Sp, static_cast<float>(q));
            if (a.C > 0) v = __fadd_rn(v, c[e]);
            acc[e] = __fadd_rn(acc[e], v);
        }
    }
    if (pk) {
        const float *U = a.psac_basis + (static_cast<size_t>(chunk) * a.H + h) * D * QVG_PSAC_RANK;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float4 u0 = *reinterpret_cast<const float4 *>(U + (j0 + e) * QVG_PSAC_RANK);
            const float4 u1 = *reinterpret_cast<const float4 *>(U + (j0 + e) * QVG_PSAC_RANK + 4);
            float corr = 0.0f;
            corr = fmaf(pk[0], u0.x, corr);
            corr = fmaf(pk[1], u0.y, corr);
            corr = fmaf(pk[2], u0.z, corr);
            corr = fmaf(pk[3], u0.w, corr);
            corr = fmaf(pk[4], u1.x, corr);
            corr = fmaf(pk[5], u1.y, corr);
            corr = fmaf(pk[6], u1.z, corr);
            corr = fmaf(pk[7], u1.w, corr);
            acc[e] = acc[e] + corr;
        }
    }
}

// One-stage fast path: the loads of a slot's 64-channel half are issued
// before any arithmetic (code bits, scales, cluster id, then the 128-byte
// bf16 centroid piece), so a producer thread exposes its memory latency once
// per half rather than once per 8 channels.  K_hat = fma(S, q, c) in fp32,
// rounded to fp16; out gets 32 packed half2 words (channels kb*64 ..).
template <int D, int BITS>
__device__ __forceinline__ void rebuild_half_fast(const AttnWsArgs &a, const uint8_t *codes,
                                                  const uint16_t *scales, const uint8_t *ids,
                                                  const uint16_t *cent, int h, int chunk, int slot, int kb,
                                                  uint32_t (&out)[32]) {
    constexpr int NB = D * BITS / 8;
    constexpr int HB = 64 * BITS / 8;      // code bytes of a 64-channel half: 16 (INT2) or 32 (INT4)
    const int ng = D / a.group;
    const size_t srow = static_cast<size_t>(h) * a.cap + slot;
    uint4 cw[HB / 16];
#pragma unroll
    for (int i = 0; i < HB / 16; ++i) cw[i] = *reinterpret_cast<const uint4 *>(codes + srow * NB + kb * HB + 16 * i);
    float S[8];
    if (a.group >= 64) {
        const float s0 = f16_to_f32(scales[srow * ng + (kb * 64) / a.group]);
#pragma unroll
        for (int i = 0; i < 8; ++i) S[i] = s0;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) S[i] = f16_to_f32(scales[srow * ng + (kb * 64 + 8 * i) / a.group]);
    }
    uint4 cr[8];
    if (a.C > 0) {
        const uint16_t *row = cent + (static_cast<size_t>(h) * a.max_chunks + chunk) * a.C * D +
                              static_cast<size_t>(ids[srow]) * D + kb * 64;
#pragma unroll
        for (int i = 0; i < 8; ++i) cr[i] = *reinterpret_cast<const uint4 *>(row + 8 * i);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) cr[i] = make_uint4(0, 0, 0, 0);
    }
    const uint32_t *cb = reinterpret_cast<const uint32_t *>(cw);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t bits = static_cast<uint32_t>((cb[(8 * i * BITS) / 32] >> ((8 * i * BITS) % 32)) &
                                                    ((1ull << (8 * BITS)) - 1ull));
        const uint32_t c4[4] = {cr[i].x, cr[i].y, cr[i].z, cr[i].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int q0 = static_cast<int>((bits >> (2 * e * BITS)) & ((1u << BITS) - 1u)) - (1 << (BITS - 1));
            const int q1 = static_cast<int>((bits >> ((2 * e + 1) * BITS)) & ((1u << BITS) - 1u)) - (1 << (BITS - 1));
            const float v0 = fmaf(S[i], static_cast<float>(q0), __uint_as_float(c4[e] << 16));
            const float v1 = fmaf(S[i], static_cast<float>(q1), __uint_as_float(c4[e] & 0xffff0000u));
            out[4 * i + e] = h2(v0, v1);
        }
    }
}

// One-stage fast path for the V producers: channels [j0, j0 + 8) of 8
// consecutive slots, every load issued before the arithmetic.
template <int D, int BITS>
__device__ __forceinline__ void rebuild_8x8_fast(const AttnWsArgs &a, int h, int chunk, int slot0, int nvalid_rel,
                                                 int j0, uint32_t (&hv)[8][4]) {
    constexpr int NB = D * BITS / 8;
    const int ng = D / a.group;
    const uint16_t *cbase = a.vcent + (static_cast<size_t>(h) * a.max_chunks + chunk) * a.C * D + j0;
    int id[8];
    uint32_t bits[8];
    float S[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const size_t srow = static_cast<size_t>(h) * a.cap + slot0 + k;
        const bool ok = k < nvalid_rel;
        id[k] = (ok && a.C > 0) ? a.vids[srow] : 0;
        if constexpr (BITS == 2)
            bits[k] = ok ? *reinterpret_cast<const uint16_t *>(a.vcodes + srow * NB + j0 / 4) : 0u;
        else
            bits[k] = ok ? *reinterpret_cast<const uint32_t *>(a.vcodes + srow * NB + j0 / 2) : 0u;
        S[k] = ok ? f16_to_f32(a.vscales[srow * ng + j0 / a.group]) : 0.0f;
    }
    uint4 cr[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        cr[k] = (k < nvalid_rel && a.C > 0) ? *reinterpret_cast<const uint4 *>(cbase + static_cast<size_t>(id[k]) * D)
                                            : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t c4[4] = {cr[k].x, cr[k].y, cr[k].z, cr[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int q0 = static_cast<int>((bits[k] >> (2 * e * BITS)) & ((1u << BITS) - 1u)) - (1 << (BITS - 1));
            const int q1 = static_cast<int>((bits[k] >> ((2 * e + 1) * BITS)) & ((1u << BITS) - 1u)) - (1 << (BITS - 1));
            const float v0 = fmaf(S[k], static_cast<float>(q0), __uint_as_float(c4[e] << 16));
            const float v1 = fmaf(S[k], static_cast<float>(q1), __uint_as_float(c4[e] & 0xffff0000u));
            hv[k][e] = k < nvalid_rel ? h2(v0, v1) : 0u;
        }
    }
}

}  // namespace ws

template <int D, int BITS, bool TOP1>
__global__ void __launch_bounds__(ws::kThreads, 1) k_attention_ws(AttnWsArgs a) {
    using namespace ws;
    constexpr int KB = D / 64;
    constexpr int QB = KB * 16384;       // one 128 x D fp16 tile
    constexpr int VB = D * 256;          // D x 128 fp16 (two 64-slot K blocks)
    constexpr int PB = 32768;            // 128 x 128 fp16
    constexpr int DS = D / 8;            // V channels per producer thread
    extern __shared__ __align__(1024) uint8_t sm_raw[];
    uint8_t *sm = sm_raw + ((1024u - (umma::smem_u32(sm_raw) & 1023u)) & 1023u);
    uint8_t *Q0 = sm, *Q1 = Q0 + QB, *Kt = Q1 + QB, *Vt0 = Kt + QB, *P0 = Vt0 + 2 * VB, *P1 = P0 + PB;
    __shared__ uint64_t kfull, vfull[2], kfree, vfree[2], sfull[2], pfull[2], ofull[2];
    __shared__ uint32_t tmem_base;
    __shared__ int fail;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hq = blockIdx.y, h = hq / a.grp, q0 = blockIdx.x * 256;
    const int n_tiles = a.n_slots / QVG_TILE;

    // Q tiles -> fp16 (exact for bf16 values in fp16's normal range), swizzled K-major
    for (int i = tid; i < 256 * (D / 8); i += kThreads) {
        const int rr = i / (D / 8), ci = i % (D / 8), kb = ci >> 3, c = ci & 7;
        const int r = rr & 127;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (q0 + rr < a.Nq) {
            const uint4 b = *reinterpret_cast<const uint4 *>(a.q + (static_cast<size_t>(q0 + rr) * a.Hq + hq) * D + ci * 8);
            v = make_uint4(h2(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xffff0000u)),
                           h2(__uint_as_float(b.y << 16), __uint_as_float(b.y & 0xffff0000u)),
                           h2(__uint_as_float(b.z << 16), __uint_as_float(b.z & 0xffff0000u)),
                           h2(__uint_as_float(b.w << 16), __uint_as_float(b.w & 0xffff0000u)));
        }
        *reinterpret_cast<uint4 *>((rr < 128 ? Q0 : Q1) + kb * 16384 + r * 128 + ((c ^ (r & 7)) << 4)) = v;
    }
    if (warp == 12) {
        umma::tmem_alloc(&tmem_base, 512);
        umma::tmem_relinquish();
    }
    if (tid == 0) {
        umma::mbar_init(&kfull, 128);
        umma::mbar_init(&kfree, 1);
        for (int i = 0; i < 2; ++i) {
            umma::mbar_init(&vfull[i], 128);
            umma::mbar_init(&vfree[i], 1);
            umma::mbar_init(&sfull[i], 1);
            umma::mbar_init(&pfull[i], 128);
            umma::mbar_init(&ofull[i], 1);
        }
        umma::fence_barrier_init();
        fail = 0;
    }
    umma::fence_proxy_async_smem();
    umma::tc_fence_before();
    __syncthreads();
    umma::tc_fence_after();
    const uint32_t tmem = tmem_base;
    volatile int *vfail = &fail;

    if (warp < 8) {
        // ------------------------------------------------ softmax of tile i
        const int i = warp >> 2, r = tid & 127;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + i * 128 + lane_off, tO = tmem + 256 + i * 128 + lane_off;
        uint8_t *Pi = i ? P1 : P0;
        float m_used = -INFINITY, l_sum = 0.0f, best = -INFINITY;
        int best_slot = 0, it = 0;
        for (int t = 0; t < n_tiles; ++t) {
            const TileInfo ti = tile_info(a, t);
            if (ti.nvalid == 0) continue;
            if (!ws::wait(&sfull[i], it & 1, vfail)) break;
            umma::tc_fence_after();
            // row maximum of the raw logits (the scale is positive), then scaled
            // once; four independent chains (the top-1 variant keeps one chain
            // so that ties resolve to the lowest slot)
            float rmax = -INFINITY;
            int targ = 0;
            if constexpr (TOP1) {
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    uint32_t v[32];
                    umma::tmem_ld32(tS + c0, v);
                    umma::tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const float x = c0 + k < ti.nvalid ? __uint_as_float(v[k]) : -INFINITY;
                        if (x > rmax) { rmax = x; targ = c0 + k; }
                    }
                }
            } else {
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    uint32_t v[32];
                    umma::tmem_ld32(tS + c0, v);
                    umma::tmem_ld_wait();
                    if (c0 + 32 <= ti.nvalid) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) m4[k & 3] = fmaxf(m4[k & 3], __uint_as_float(v[k]));
                    } else {
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            if (c0 + k < ti.nvalid) m4[k & 3] = fmaxf(m4[k & 3], __uint_as_float(v[k]));
                    }
                }
                rmax = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            }
            const float tmax = rmax * a.scale_log2;
            if constexpr (TOP1) {
                if (tmax > best) {
                    best = tmax;
                    best_slot = ti.s0 + targ;
                }
            }
            float corr = 1.0f;
            bool rescale = false;
            if (tmax > m_used + kRescale) {
                corr = ex2(m_used - tmax);
                rescale = it > 0;
                m_used = tmax;
            }
            if (it > 0) {  // PV_i of the previous tile done: P_i is free and O_i settled
                if (!ws::wait(&ofull[i], (it - 1) & 1, vfail)) break;
                umma::tc_fence_after();
                if (__any_sync(0xffffffffu, rescale)) {
                    const float f = rescale ? corr : 1.0f;
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t v[32];
                        umma::tmem_ld32(tO + c0, v);
                        umma::tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * f);
                        umma::tmem_st32(tO + c0, v);
                    }
                    umma::tmem_st_wait();
                }
            }
            float ls4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t v[32];
                umma::tmem_ld32(tS + c0, v);
                umma::tmem_ld_wait();
                uint32_t pk[16];
                const float nm = -m_used;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int c = c0 + 2 * k;
                    float p0 = ex2(fmaf(__uint_as_float(v[2 * k]), a.scale_log2, nm));
                    float p1 = ex2(fmaf(__uint_as_float(v[2 * k + 1]), a.scale_log2, nm));
                    if (c0 + 32 > ti.nvalid) {
                        p0 = c < ti.nvalid ? p0 : 0.0f;
                        p1 = c + 1 < ti.nvalid ? p1 : 0.0f;
                    }
                    pk[k] = h2(p0, p1);
                    // the row sum adds the fp16 values the PV product uses
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&pk[k]));
                    ls4[k & 3] += f.x + f.y;
                }
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int ci = c0 / 8 + x, kb = ci >> 3, c = ci & 7;
                    *reinterpret_cast<uint4 *>(Pi + kb * 16384 + r * 128 + ((c ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
                }
            }
            const float ls = (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
            l_sum = l_sum * corr + ls;
            umma::fence_proxy_async_smem();
            umma::tc_fence_before();
            umma::mbar_arrive(&pfull[i]);
            ++it;
        }
        // epilogue: O_i / l
        bool ok = !*vfail && it > 0 && ws::wait(&ofull[i], (it - 1) & 1, vfail);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            umma::tc_fence_after();
            const int qi = q0 + i * 128 + r;
            const float inv = 1.0f / l_sum;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t v[32];
                umma::tmem_ld32(tO + c0, v);
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
                if constexpr (TOP1) a.top1[static_cast<size_t>(hq) * a.Nq + qi] = best_slot;
            }
        }
    } else if (warp < 12) {
        // ------------------------------------------------ K producers (thread = slot)
        const int r = tid - 256;
        const bool psac = a.psac_p != nullptr;
        int it = 0;
        for (int t = 0; t < n_tiles; ++t) {
            const TileInfo ti = tile_info(a, t);
            if (ti.nvalid == 0) continue;
            if (it > 0 && !ws::wait(&kfree, (it - 1) & 1, vfail)) break;
            const bool valid = r < ti.nvalid;
            float pk[QVG_PSAC_RANK];
            if (psac && valid) {
                const size_t prow = static_cast<size_t>(h) * a.cap + ti.s0 + r;
                const float pS = f16_to_f32(a.psac_s[prow]);
                const int2 pv = *reinterpret_cast<const int2 *>(a.psac_p + prow * QVG_PSAC_RANK);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    pk[k] = pS * static_cast<float>(static_cast<int8_t>((pv.x >> (8 * k)) & 0xff));
                    pk[k + 4] = pS * static_cast<float>(static_cast<int8_t>((pv.y >> (8 * k)) & 0xff));
                }
            }
            if (a.L == 1 && !psac) {
#pragma unroll 1
                for (int kb = 0; kb < KB; ++kb) {
                    uint32_t hk[32];
                    if (valid) {
                        rebuild_half_fast<D, BITS>(a, a.kcodes, a.kscales, a.kids, a.kcent, h, ti.chunk, ti.s0 + r, kb, hk);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) hk[e] = 0u;
                    }
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8)
                        *reinterpret_cast<uint4 *>(Kt + kb * 16384 + r * 128 + ((c8 ^ (r & 7)) << 4)) =
                            make_uint4(hk[4 * c8], hk[4 * c8 + 1], hk[4 * c8 + 2], hk[4 * c8 + 3]);
                }
            } else {
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) {
#pragma unroll 2
                    for (int c8 = 0; c8 < 8; ++c8) {
                        uint4 out = make_uint4(0, 0, 0, 0);
                        if (valid) {
                            float kv[8];
                            rebuild8<D, BITS>(a, a.kcodes, a.kscales, a.kids, a.kcent, h, ti.chunk, ti.s0 + r,
                                              kb * 64 + c8 * 8, psac ? pk : nullptr, kv);
                            out = make_uint4(h2(kv[0], kv[1]), h2(kv[2], kv[3]), h2(kv[4], kv[5]), h2(kv[6], kv[7]));
                        }
                        *reinterpret_cast<uint4 *>(Kt + kb * 16384 + r * 128 + ((c8 ^ (r & 7)) << 4)) = out;
                    }
                }
            }
            umma::fence_proxy_async_smem();
            umma::mbar_arrive(&kfull);
            ++it;
        }
    } else {
        // ------------------------------------------------ V producers (8 slots x D/8 channels)
        // and, on warp 12 lane 0, the MMA issuer
        const int u = tid - 384;
        const bool issuer = (warp == 12 && lane == 0);
        const uint32_t idS = umma::idesc_f16(128, 128, 0), idO = umma::idesc_f16(128, D, 0);
        const uint32_t q0a = umma::smem_u32(Q0), q1a = umma::smem_u32(Q1), ka = umma::smem_u32(Kt);
        const uint32_t v0a = umma::smem_u32(Vt0), p0a = umma::smem_u32(P0), p1a = umma::smem_u32(P1);
        uint64_t *last_bar = nullptr;  // barrier of the issuer's latest commit (drained on failure)
        uint32_t last_par = 0;
        int it = 0;
        for (int t = 0; t < n_tiles; ++t) {
            const TileInfo ti = tile_info(a, t);
            if (ti.nvalid == 0) continue;
            if (issuer) {
                // S_i = Q_i K_t^T as soon as the K tile is ready
                if (!ws::wait(&kfull, it & 1, vfail)) break;
                umma::tc_fence_after();
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                    umma::mma_f16(tmem + 0, umma::desc_sw128(q0a + off), umma::desc_sw128(ka + off), idS, s != 0);
                }
                umma::mma_commit(&sfull[0]);
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                    umma::mma_f16(tmem + 128, umma::desc_sw128(q1a + off), umma::desc_sw128(ka + off), idS, s != 0);
                }
                umma::mma_commit(&sfull[1]);
                umma::mma_commit(&kfree);
                last_bar = &kfree;
                last_par = it & 1;
            }
            // V tiles are double-buffered: tile `it` uses buffer it & 1, free
            // once the PV products of tile it - 2 are done
            const int vb = it & 1;
            uint8_t *Vt = Vt0 + vb * VB;
            if (it >= 2 && !ws::wait(&vfree[vb], ((it >> 1) - 1) & 1, vfail)) break;
            // thread = slot: rebuild the slot's V_hat row (64 channels at a time,
            // every load issued first) and store it as column `r` of V_hat^T
            const int r = u;
            const bool valid = r < ti.nvalid;
            const int kbs = r >> 6, cs = (r & 63) >> 3, es = (r & 7) * 2;
#pragma unroll 1
            for (int kb = 0; kb < KB; ++kb) {
                uint32_t hv[32];
                if (valid && a.L == 1) {
                    rebuild_half_fast<D, BITS>(a, a.vcodes, a.vscales, a.vids, a.vcent, h, ti.chunk, ti.s0 + r, kb, hv);
                } else if (valid) {
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        float vv[8];
                        rebuild8<D, BITS>(a, a.vcodes, a.vscales, a.vids, a.vcent, h, ti.chunk, ti.s0 + r,
                                          kb * 64 + c8 * 8, nullptr, vv);
#pragma unroll
                        for (int e = 0; e < 4; ++e) hv[4 * c8 + e] = h2(vv[2 * e], vv[2 * e + 1]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) hv[e] = 0u;
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int j = kb * 64 + 2 * e;
                    uint8_t *col = Vt + kbs * (D * 128) + es;
                    *reinterpret_cast<uint16_t *>(col + j * 128 + ((cs ^ (j & 7)) << 4)) =
                        static_cast<uint16_t>(hv[e] & 0xffffu);
                    *reinterpret_cast<uint16_t *>(col + (j + 1) * 128 + ((cs ^ ((j + 1) & 7)) << 4)) =
                        static_cast<uint16_t>(hv[e] >> 16);
                }
            }
            umma::fence_proxy_async_smem();
            umma::mbar_arrive(&vfull[vb]);
            if (issuer) {
                // O_i += P_i V_t once the V tile and P_i are ready
                if (!ws::wait(&vfull[vb], (it >> 1) & 1, vfail) || !ws::wait(&pfull[0], it & 1, vfail)) break;
                umma::tc_fence_after();
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t aoff = (s >> 2) * 16384 + (s & 3) * 32, boff = (s >> 2) * (D * 128) + (s & 3) * 32;
                    umma::mma_f16(tmem + 256, umma::desc_sw128(p0a + aoff), umma::desc_sw128(v0a + vb * VB + boff), idO, (it | s) != 0);
                }
                umma::mma_commit(&ofull[0]);
                last_bar = &ofull[0];
                if (!ws::wait(&pfull[1], it & 1, vfail)) break;
                umma::tc_fence_after();
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t aoff = (s >> 2) * 16384 + (s & 3) * 32, boff = (s >> 2) * (D * 128) + (s & 3) * 32;
                    umma::mma_f16(tmem + 384, umma::desc_sw128(p1a + aoff), umma::desc_sw128(v0a + vb * VB + boff), idO, (it | s) != 0);
                }
                umma::mma_commit(&ofull[1]);
                umma::mma_commit(&vfree[vb]);
                last_bar = &vfree[vb];
                last_par = (it >> 1) & 1;
            }
            ++it;
        }
        // on failure, let the MMAs already issued drain before TMEM is released
        if (issuer && *vfail && last_bar) umma::mbar_wait(last_bar, last_par, kWaitNs);
    }
    umma::tc_fence_before();
    __syncthreads();
    if (tid == 0 && *vfail) raise_error(a.err, QVG_ERR_TIMEOUT);
    if (warp == 12) {
        umma::tc_fence_after();
        umma::tmem_dealloc(tmem, 512);
    }
}

template <int D, int BITS, bool TOP1>
static qvg_status attn_ws_t(const AttnWsArgs &a, cudaStream_t st) {
    constexpr size_t smem = 3 * (D / 64) * 16384 + 2 * D * 256 + 2 * 32768 + 1024;
    static bool attr = false;
    if (!attr) {
        const cudaError_t e = cudaFuncSetAttribute(k_attention_ws<D, BITS, TOP1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            note_cuda_error(e);
            return QVG_ERR_CUDA;
        }
        attr = true;
    }
    dim3 grid(ceil_div(a.Nq, 256), a.Hq);
    k_attention_ws<D, BITS, TOP1><<<grid, ws::kThreads, smem, st>>>(a);
    QVG_LAUNCH_CHECK();
    return QVG_OK;
}

template <int D, int BITS>
static qvg_status attn_ws(const AttnWsArgs &a, cudaStream_t st) {
    return a.top1 ? attn_ws_t<D, BITS, true>(a, st) : attn_ws_t<D, BITS, false>(a, st);
}

qvg_status launch_attention_ws(const qvg_params *p, const uint16_t *q, int Nq, int Hq, const qvg_cache *k,
                               const qvg_cache *v, float scale_log2, void *out, int out_dtype, float *lse,
                               int32_t *top1, cudaStream_t st) {
    AttnWsArgs a{};
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
    if (k->d == 64) return p->bits == 2 ? attn_ws<64, 2>(a, st) : attn_ws<64, 4>(a, st);
    return p->bits == 2 ? attn_ws<128, 2>(a, st) : attn_ws<128, 4>(a, st);
}

}  // namespace qvg
