// attention_ws.cuh -- warp-specialised tensor-core attention over the
// compressed KV cache (sm_103a: tcgen05.mma, TMEM, mbarriers).
//
// Quant VideoGen notes, "algorithm-system co-design": dequantisation is
// fused with attention and the 2-bit codes stay packed in memory.  The
// reconstructed K_hat = sum_l (S_l q_l + C_l) (+ the PSAC term P_hat U^T of
// the QuantWM write-up) and V_hat only ever exist in shared memory (as fp16
// tiles, one per stage) and as products in tensor memory.
//
// One CTA = two 128-row query tiles of one query head, which share every
// rebuilt K_hat / V_hat tile; the warp roles and barriers are listed above
// the kernel.
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D),
// O1 [384,384+D), fp32; P_i (fp16 pairs) over S_i's first 64 columns.  Per
// cache tile t:
//   S_i = Q_i K_t^T              (M=128, N=128 slots, K=D; Q, K_hat from shared memory)
//   P_i = exp2(s * scale*log2e - m_i), fp16, m_i raised lazily (by > 8)
//   O_i += P_i V_t               (M=128, N=D, K=128 slots; P_i from TMEM)
// fp16 operands carry K_hat, V_hat, Q and P with a relative rounding of
// 2^-11; on the synthetic LongCat-like and world-model caches this keeps
// max|dO| / max|O| near 6e-5 against the fp64 oracle.
#pragma once

#include <algorithm>
#include <climits>

#include "common.cuh"
#include "umma.cuh"

namespace qvg {

struct AttnWsArgs {
    const uint16_t *q;
    int Nq, Hq, H, grp, L, C, group, cap, max_chunks, n_slots;
    int glog2;  // log2(group): groups are powers of two, so the producers shift instead of divide
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
    float *best;  // split mode with top-1: each split's best scaled logit
    int *err;
    // the current chunk's own K/V (bf16 [n_raw][H][D]), attended after the
    // n_ctiles = n_slots / QVG_TILE cache tiles; raw row j is slot n_slots + j
    const uint16_t *kraw, *vraw;
    int n_raw, n_ctiles;
    // outlier split ("Temporally stable 2-bit KV-cache compression for video
    // world models, in practice", section 3.4): per stage and group, the fp16
    // value split off and its channel in the group (0xFF: none), or NULL
    const uint16_t *koutv, *voutv;
    const uint8_t *kouti, *vouti;
    // temporal anchors (the same page, section 3.3): anchor chunks are
    // read as bf16 rows of these arenas; chunk_anchor[c] = first row, or -1
    const uint16_t *kanch, *vanch;
    const int32_t *chunk_anchor;
    // bound of the pipeline's waits (ns); inject: the test hook that makes
    // each softmax group's MMA issuer wait once on a barrier nothing completes
    uint64_t wait_ns;
    int inject;
};

namespace ws {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kNbuf = 2;  // K_hat and V_hat tiles in flight, each
// Per-CTA tile table in shared memory (chunk; valid slots and first row),
// filled once at launch: the tile lookup otherwise chains three dependent
// global loads (tile -> chunk -> start / length) in every producer's and
// softmax warp's tile loop.  Tiles past kTabMax, or whose first row does not
// fit the packed field, are looked up directly.
constexpr int kTabMax = 4096;
constexpr int kTabDirect = INT_MIN;
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

// Bounded wait that also gives up as soon as another role has failed.  The
// global timer (slow to read) is consulted only after 32 unsuccessful
// try_waits, so a short wait never reads it.
__device__ __forceinline__ bool wait(uint64_t *bar, uint32_t parity, volatile int *fail, uint64_t limit_ns) {
    for (int i = 0; i < 32; ++i)
        if (umma::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = umma::globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (umma::mbar_try_wait(bar, parity)) return true;
        if (*fail) return false;
        if (umma::globaltimer_ns() - t0 > limit_ns) {
            *fail = 1;
            return false;
        }
    }
}

// Tile t covers slots [t QVG_TILE, (t + 1) QVG_TILE), of which the first
// nvalid hold tokens.  Tiles below n_ctiles are cache tiles (chunk = the
// chunk that owns them, base = the first slot); the rest hold the current
// chunk's raw rows (chunk = -1).  A tile of an anchor chunk is read raw as
// well, from the anchor arena (chunk = -2).  A raw tile's base is the row of
// its first slot in its source.  RAW = false: no raw tile can occur (no
// current-chunk rows, no anchors), and the lookup is the cache's alone.
struct TileInfo {
    int base, chunk, nvalid;
};

template <bool RAW>
__device__ __forceinline__ TileInfo tile_info(const AttnWsArgs &a, int t) {
    TileInfo ti;
    const int s0 = t * QVG_TILE;
    ti.base = s0;
    if constexpr (!RAW) {
        ti.chunk = a.tile_chunk[t];
        ti.nvalid = min(QVG_TILE, max(0, a.chunk_start[ti.chunk] + a.chunk_len[ti.chunk] - s0));
        return ti;
    }
    if (t < a.n_ctiles) {
        const int c = a.tile_chunk[t], start = a.chunk_start[c];
        ti.chunk = c;
        ti.nvalid = min(QVG_TILE, max(0, start + a.chunk_len[c] - s0));
        if (a.chunk_anchor) {
            const int arow = a.chunk_anchor[c];
            if (arow >= 0) {
                ti.chunk = -2;
                ti.base = arow + s0 - start;
            }
        }
    } else {
        ti.chunk = -1;
        ti.nvalid = min(QVG_TILE, a.n_raw - (t - a.n_ctiles) * QVG_TILE);
        ti.base = s0 - a.n_slots;
    }
    return ti;
}

template <bool RAW>
__device__ __forceinline__ int2 tile_entry(const AttnWsArgs &a, int t) {
    const TileInfo ti = tile_info<RAW>(a, t);
    if (ti.base >= (1 << 23)) return make_int2(kTabDirect, 0);
    return make_int2(ti.chunk, ti.nvalid | (ti.base << 8));
}

// Tile tb + t from the CTA's table (t counts from tb).
template <bool RAW>
__device__ __forceinline__ TileInfo tile_at(const AttnWsArgs &a, const int2 *tab, int tab_n, int tb, int t) {
    if (t < tab_n) {
        const int2 e = tab[t];
        if (e.x != kTabDirect) return TileInfo{e.y >> 8, e.x, e.y & 0xFF};
    }
    return tile_info<RAW>(a, tb + t);
}

// Eight bf16 values -> eight fp16 values (exact inside fp16's normal range).
__device__ __forceinline__ uint4 bf16x8_to_f16(uint4 b) {
    return make_uint4(h2(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xffff0000u)),
                      h2(__uint_as_float(b.y << 16), __uint_as_float(b.y & 0xffff0000u)),
                      h2(__uint_as_float(b.z << 16), __uint_as_float(b.z & 0xffff0000u)),
                      h2(__uint_as_float(b.w << 16), __uint_as_float(b.w & 0xffff0000u)));
}

// One-stage fast path, split into its loads and its arithmetic so that a
// producer can put the loads of a 64-channel half in flight before it waits
// for its buffer.  K_hat (or V_hat) = fma(S, q, c) in fp32, rounded to fp16.
template <int BITS>
struct HalfData {
    uint4 cw[BITS == 2 ? 1 : 2];  // 64 codes
    uint32_t s2[4];               // fp16 scales of the 8-channel blocks, two per word
    uint4 cr[8];                  // 64 bf16 centroid channels
    uint32_t oi[2], ov[4];        // outlier split: per group of the half (1, 2, 4 or 8 groups of
                                  // 64, 32, 16 or 8 channels), the channel split off (byte g of
                                  // oi; 0xFF none) and its fp16 value (half g of ov)
};

// OUTL: 0 without the outlier split, else the groups per 64-channel half
// (1, 2, 4 or 8 for groups of 64, 32, 16 or 8 channels).
template <int D, int BITS, int OUTL>
__device__ __forceinline__ void load_half(const AttnWsArgs &a, const uint8_t *codes, const uint16_t *scales,
                                          const uint16_t *cent, const uint16_t *outv, const uint8_t *outi, int h,
                                          int chunk, int slot, int id, int kb, HalfData<BITS> &hd) {
    constexpr int NB = D * BITS / 8;
    constexpr int HB = 64 * BITS / 8;
    const int ng = D >> a.glog2;
    const size_t srow = static_cast<size_t>(h) * a.cap + slot;
    hd.oi[0] = hd.oi[1] = 0xFFFFFFFFu;
    hd.ov[0] = hd.ov[1] = hd.ov[2] = hd.ov[3] = 0u;
    if (OUTL) {
        // the half's NG groups are entries [srow * ng + kb * NG, + NG) of the
        // side list: a multiple of NG, so one aligned vector (the cache's
        // buffers are 16-byte aligned)
        constexpr int NG = OUTL;
        const size_t e0 = srow * ng + static_cast<size_t>(kb) * NG;
        if constexpr (NG == 1) {
            hd.oi[0] = 0xFFFFFF00u | outi[e0];
            hd.ov[0] = outv[e0];
        } else if constexpr (NG == 2) {
            hd.oi[0] = 0xFFFF0000u | *reinterpret_cast<const uint16_t *>(outi + e0);
            hd.ov[0] = *reinterpret_cast<const uint32_t *>(outv + e0);
        } else if constexpr (NG == 4) {
            hd.oi[0] = *reinterpret_cast<const uint32_t *>(outi + e0);
            const uint2 v = *reinterpret_cast<const uint2 *>(outv + e0);
            hd.ov[0] = v.x;
            hd.ov[1] = v.y;
        } else {
            const uint2 i2 = *reinterpret_cast<const uint2 *>(outi + e0);
            hd.oi[0] = i2.x;
            hd.oi[1] = i2.y;
            const uint4 v = *reinterpret_cast<const uint4 *>(outv + e0);
            hd.ov[0] = v.x;
            hd.ov[1] = v.y;
            hd.ov[2] = v.z;
            hd.ov[3] = v.w;
        }
    }
#pragma unroll
    for (int i = 0; i < HB / 16; ++i) hd.cw[i] = *reinterpret_cast<const uint4 *>(codes + srow * NB + kb * HB + 16 * i);
    if (a.group >= 64) {
        const uint32_t s0 = scales[srow * ng + ((kb * 64) >> a.glog2)];
#pragma unroll
        for (int i = 0; i < 4; ++i) hd.s2[i] = s0 | (s0 << 16);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            hd.s2[i] = static_cast<uint32_t>(scales[srow * ng + ((kb * 64 + 16 * i) >> a.glog2)]) |
                       (static_cast<uint32_t>(scales[srow * ng + ((kb * 64 + 16 * i + 8) >> a.glog2)]) << 16);
    }
    if (a.C > 0) {
        const uint16_t *row = cent + ((static_cast<size_t>(h) * a.max_chunks + chunk) * a.C + id) * D + kb * 64;
#pragma unroll
        for (int i = 0; i < 8; ++i) hd.cr[i] = *reinterpret_cast<const uint4 *>(row + 8 * i);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) hd.cr[i] = make_uint4(0, 0, 0, 0);
    }
}

// A raw bf16 row of the current chunk in the same form: scale 0 and the row
// in place of the centroid, so the decode's fma(0, q, x) = x rounds the bf16
// value straight to fp16.
template <int D, int BITS>
__device__ __forceinline__ void load_half_raw(const uint16_t *raw, int H, int h, int j, int kb, HalfData<BITS> &hd) {
#pragma unroll
    for (int i = 0; i < (BITS == 2 ? 1 : 2); ++i) hd.cw[i] = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < 4; ++i) hd.s2[i] = 0u;
    hd.oi[0] = hd.oi[1] = 0xFFFFFFFFu;
    hd.ov[0] = hd.ov[1] = hd.ov[2] = hd.ov[3] = 0u;
    const uint16_t *row = raw + (static_cast<size_t>(j) * H + h) * D + kb * 64;
#pragma unroll
    for (int i = 0; i < 8; ++i) hd.cr[i] = *reinterpret_cast<const uint4 *>(row + 8 * i);
}

// A 16-byte store into a tile line.  SH: by 32-bit shared address, for the
// out-of-line producers, where the compiler cannot see that the line is in
// shared memory (a generic store there took the G = 16 outlier read path
// from 3.75 to 3.98 ms); inlined, the plain store is left to the compiler
// (the explicit form took the inlined PSAC producer from 2.38 to 3.37 ms).
template <bool SH>
__device__ __forceinline__ void st_line16(uint8_t *dst, uint4 v) {
    if constexpr (SH)
        umma::st_shared_v4(umma::smem_u32(dst), v);
    else
        *reinterpret_cast<uint4 *>(dst) = v;
}

// Zeroes one slot's 128-byte line of a 64-channel block (padding slots).
template <bool SH>
__device__ __forceinline__ void zero_line(uint8_t *dst) {
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) st_line16<SH>(dst + (c8 << 4), make_uint4(0, 0, 0, 0));
}

// Packed fp32 pairs (Blackwell f32x2 arithmetic).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void up2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Decodes the half and stores it as the eight swizzled 16-byte chunks of the
// slot's 128-byte line `dst` (chunk c at position c ^ (r % 8)), one chunk as
// soon as its four words are ready.  Codes become floats without a
// conversion instruction: OR-ing a B-bit code c, at bit k of a word, into the
// mantissa of 2^23 (0x4B000000) gives the float 2^23 + c 2^k exactly
// (k + B <= 23); one packed FMA with (2^-k0, 2^-k1) and the matching offsets
// gives q = c - 2^(B-1) exactly for both codes of a pair (every
// intermediate is an integer below 2^24), and K_hat = fma(S, q, c_bf16) has
// the single rounding of the plain fp32 expression.
// NOSHIFT: each pair's codes are taken where they sit in the block's word
// (a block's upper half is shifted down once where k + B <= 23 would not
// hold, for B = 4), with four (scale, offset) constant pairs; otherwise the
// pair is shifted down to bit 0 first, with one constant pair.  Without the
// shifts the outlier-split and PSAC kernels run 1-3.5 % faster; the
// raw-tile kernel (mode 1) loses up to 20 % to the constants' registers, and
// the plain one (mode 0) gains 0.8 % on 16 heads but loses 7 % on a one-wave
// 8-head grid and 3.5 % at 16 queries, so both keep the shifts.
template <int BITS, bool SH = false, bool NOSHIFT = false>
__device__ __forceinline__ void decode_store_half(const HalfData<BITS> &hd, uint8_t *dst, int r) {
    constexpr uint32_t M = (1u << BITS) - 1u, MAGIC = 0x4B000000u;
    constexpr float E23 = 8388608.0f, HALF = static_cast<float>(1 << (BITS - 1));
    const uint32_t *cb = reinterpret_cast<const uint32_t *>(hd.cw);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t blk = cb[(8 * i * BITS) / 32] >> ((8 * i * BITS) % 32);
        const uint32_t blk_hi = blk >> 16;  // used only where a code would sit above bit 23 - B
        const float S = f16_to_f32(static_cast<uint16_t>(hd.s2[i >> 1] >> (16 * (i & 1))));
        const uint64_t S2 = pk2(S, S);
        const uint32_t c4[4] = {hd.cr[i].x, hd.cr[i].y, hd.cr[i].z, hd.cr[i].w};
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            // the pair's codes at bits k0 and k0 + B of x
            constexpr int kMax = 23 - 2 * BITS;  // highest k0 whose pair fits the mantissa
            const int kp = 2 * e * BITS;
            const bool hi = NOSHIFT && kp > kMax;
            const uint32_t x = !NOSHIFT ? blk >> kp : hi ? blk_hi : blk;
            const int k0 = !NOSHIFT ? 0 : hi ? kp - 16 : kp, k1 = k0 + BITS;
            const uint64_t mag = pk2(__uint_as_float((x & (M << k0)) | MAGIC), __uint_as_float((x & (M << k1)) | MAGIC));
            const float s0 = 1.0f / static_cast<float>(1 << k0), s1 = 1.0f / static_cast<float>(1 << k1);
            const uint64_t q2 = fma2(mag, pk2(s0, s1), pk2(-(E23 * s0 + HALF), -(E23 * s1 + HALF)));
            const uint64_t v2 = fma2(S2, q2, pk2(__uint_as_float(c4[e] << 16), __uint_as_float(c4[e] & 0xffff0000u)));
            float v0, v1;
            up2(v2, v0, v1);
            w[e] = h2(v0, v1);
        }
        st_line16<SH>(dst + ((i ^ (r & 7)) << 4), make_uint4(w[0], w[1], w[2], w[3]));
    }
}

// Outlier split, one stage: the channel a group split off holds code 0, so
// the decode above wrote fp16(c) there; it becomes fp16(fl(o + c)), the
// rebuild of an outlier, o its stored fp16 value.  c is read back from that
// slot: bf16 -> fp16 is exact for |c| >= 2^-14 (and for 0), and only a
// centroid channel in fp16's subnormal range is re-read from the row.
template <int D, int BITS, int NG>
__device__ __forceinline__ void patch_outliers(const AttnWsArgs &a, const uint16_t *cent, const HalfData<BITS> &hd,
                                               int h, int chunk, int id, int kb, uint8_t *dst, int r) {
    constexpr int G = 64 / NG;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        const uint32_t oi = (hd.oi[g >> 2] >> (8 * (g & 3))) & 0xFFu;
        if (oi != 0xFFu) {
            const int j = g * G + static_cast<int>(oi);  // channel within the half
            const uint32_t p = umma::smem_u32(dst + (((j >> 3) ^ (r & 7)) << 4) + (j & 7) * 2);
            float c = f16_to_f32(umma::ld_shared_u16(p));
            if (a.C > 0 && c != 0.0f && fabsf(c) < 6.103515625e-05f)
                c = __uint_as_float(static_cast<uint32_t>(
                        cent[((static_cast<size_t>(h) * a.max_chunks + chunk) * a.C + id) * D + kb * 64 + j]) << 16);
            umma::st_shared_u16(p, f32_to_f16(__fadd_rn(f16_to_f32(static_cast<uint16_t>(hd.ov[g >> 1] >> (16 * (g & 1)))), c)));
        }
    }
}

// Adds the two fp16 halves of a packed pair to two fp32 sums (sm_100-family
// mixed-precision add: the fp16 value is widened exactly).
__device__ __forceinline__ void add_f16x2_to(uint32_t p, float &s0, float &s1) {
    asm("{\n\t.reg .f16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "add.rn.f32.f16 %0, h0, %0;\n\tadd.rn.f32.f16 %1, h1, %1;\n\t}"
        : "+f"(s0), "+f"(s1)
        : "r"(p));
}

// P = exp2(s * scale_log2 - m) for 32 logits of one row, rounded to fp16
// and packed in pairs (column 2k in the low half of pk[k]), ready to be
// written over the row's S columns in tensor memory.  The row sum adds the
// same fp16 values the PV product uses, so the weights of O are normalised
// exactly (a one-slot cache returns V_hat unchanged).  Columns at or past
// nvalid (relative to c0) give 0.
__device__ __forceinline__ void softmax_chunk(const uint32_t (&v)[32], int c0, int nvalid, uint64_t sl2,
                                              uint64_t nm2, uint32_t (&pk)[16], float (&acc)[4]) {
    const bool full = c0 + 32 <= nvalid;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        float y0, y1;
        up2(fma2(pk2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1])), sl2, nm2), y0, y1);
        float p0 = ex2(y0), p1 = ex2(y1);
        if (!full) {
            p0 = c0 + 2 * k < nvalid ? p0 : 0.0f;
            p1 = c0 + 2 * k + 1 < nvalid ? p1 : 0.0f;
        }
        pk[k] = h2(p0, p1);
        add_f16x2_to(pk[k], acc[2 * (k & 1)], acc[2 * (k & 1) + 1]);
    }
}

// One producer role: the compressed stream it rebuilds and its buffers.
// Tile t goes to buffer t % kNbuf (QVG_TILE slots x D channels, 64-channel
// blocks of 128-byte swizzled lines); full[b] gets one arrival per slot
// thread, free[b] is committed by the MMAs that read the buffer.
struct Producer {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint8_t *ids;
    const uint16_t *cent;
    const uint16_t *raw;   // the current chunk's rows (raw tiles)
    const uint16_t *anch;  // the anchor arena (anchor tiles)
    const uint16_t *outv;  // outlier split side list, or NULL
    const uint8_t *outi;
    uint8_t *buf0;
    uint64_t *full, *freeb;
    bool psac;
    const int2 *tab;  // the CTA's tile table and its length
    int tab_n;
    uint8_t *pbuf;    // PSAC on the tensor core: the P_hat operand of each K buffer, or NULL
};

// Stage l of a cache tile reads the stage's rows: every compressed array is
// [L][H][...], so stage l of head h is row l * H + h (hl below).  A raw tile
// has stage 0 only.
template <int D, int BITS, int OUTL, bool RAW>
__device__ __forceinline__ void load_tile_half(const AttnWsArgs &a, const Producer &pr, int h, int hl,
                                               const TileInfo &ti, int r, int id, int kb, HalfData<BITS> &hd) {
    if (!RAW || ti.chunk >= 0)
        load_half<D, BITS, OUTL>(a, pr.codes, pr.scales, pr.cent, pr.outv, pr.outi, hl, ti.chunk, ti.base + r, id, kb, hd);
    else
        load_half_raw<D, BITS>(ti.chunk == -2 ? pr.anch : pr.raw, a.H, h, ti.base + r, kb, hd);
}

// One stage per buffer fill: with L stages, pseudo-tile u = t L + l holds
// stage l of tile t, rebuilt like a one-stage tile, and the S and PV
// products of the L pseudo-tiles accumulate into the same S_i and O_i in
// TMEM (K_hat = sum_l K_hat_l, so S = sum_l Q K_hat_l^T; likewise for V_hat):
// each stage is rounded to fp16 once, on its own values, and the stages are
// summed in fp32 by the tensor core.  Stages past 0 of a raw tile are zero.
// The loads of one 64-channel half are always in flight while the previous
// half is decoded (two register sets, A for the first half of a pseudo-tile
// and B for the second when D = 128); table entries and cluster ids run two
// pseudo-tiles ahead (ids are read for cache tiles only, whose slots
// t * QVG_TILE + r < n_slots <= capacity: in bounds).
// PSAC (K only): the slot's correction P_hat U^T is not added here; with the
// tile's last stage the slot writes P_hat = fp16(S_P p_k), k < 8, as row r
// of the tile's K = 16 operand (no swizzle: row r at (r / 8) * 256 +
// (r % 8) * 16, columns 8..15 zero), and the S product adds (Q U) P_hat^T on
// the tensor core.  Raw tiles and padding slots write zeros.
template <int D, int BITS, int OUTL, bool RAW, bool PSAC = false>
__device__ __forceinline__ void produce_fast(const AttnWsArgs &a, const Producer &pr, int h, int r, int tb,
                                             int n_tiles, volatile int *vfail, int L = 1) {
    constexpr int KB = D / 64, TB = KB * 16384;
    const int n_u = n_tiles * L;
    // tile, stage, cluster id and validity of pseudo-tile u
    auto info = [&](int u, TileInfo &ti, int &l, int &id, bool &v) {
        const int t = u / L;
        l = u - t * L;
        ti = tile_at<RAW>(a, pr.tab, pr.tab_n, tb, t);
        id = 0;
        if (a.C > 0 && ti.chunk >= 0)
            id = pr.ids[(static_cast<size_t>(l) * a.H + h) * a.cap + static_cast<size_t>(tb + t) * QVG_TILE + r];
        v = r < ti.nvalid && (ti.chunk >= 0 || l == 0);
    };
    TileInfo ti0{}, ti1{};
    int l0 = 0, l1 = 0, id0 = 0, id1 = 0;
    bool v0 = false, v1 = false;
    if (n_u > 0) info(0, ti0, l0, id0, v0);
    if (n_u > 1) info(1, ti1, l1, id1, v1);
    HalfData<BITS> A, B;
    if (v0) load_tile_half<D, BITS, OUTL, RAW>(a, pr, h, l0 * a.H + h, ti0, r, id0, 0, A);
    for (int u = 0; u < n_u; ++u) {
        const int b = u % kNbuf, use = u / kNbuf;
        uint8_t *T = pr.buf0 + b * TB + r * 128;
        const int hl0 = l0 * a.H + h;
        TileInfo ti2{};
        int l2 = 0, id2 = 0;
        bool v2 = false;
        if (u + 2 < n_u) info(u + 2, ti2, l2, id2, v2);
        const bool valid = v0, valid1 = u + 1 < n_u && v1;
        const bool last = l0 == L - 1;
        int2 pv = make_int2(0, 0);
        uint32_t ps = 0u;
        if constexpr (PSAC) {
            if (pr.pbuf && last && r < ti0.nvalid && ti0.chunk >= 0) {
                const size_t prow = static_cast<size_t>(h) * a.cap + ti0.base + r;
                pv = *reinterpret_cast<const int2 *>(a.psac_p + prow * QVG_PSAC_RANK);
                ps = a.psac_s[prow];
            }
        }
        if constexpr (KB == 2) {
            if (valid) load_tile_half<D, BITS, OUTL, RAW>(a, pr, h, hl0, ti0, r, id0, 1, B);
            if (use > 0 && !wait(&pr.freeb[b], (use - 1) & 1, vfail, a.wait_ns)) return;
            if (valid) {
                decode_store_half<BITS, OUTL != 0, (OUTL != 0 || PSAC)>(A, T, r);
                if constexpr (OUTL != 0) patch_outliers<D, BITS, OUTL>(a, pr.cent, A, hl0, ti0.chunk, id0, 0, T, r);
            } else {
                zero_line<OUTL != 0>(T);
            }
            if (valid1) load_tile_half<D, BITS, OUTL, RAW>(a, pr, h, l1 * a.H + h, ti1, r, id1, 0, A);
            if (valid) {
                decode_store_half<BITS, OUTL != 0, (OUTL != 0 || PSAC)>(B, T + 16384, r);
                if constexpr (OUTL != 0) patch_outliers<D, BITS, OUTL>(a, pr.cent, B, hl0, ti0.chunk, id0, 1, T + 16384, r);
            } else {
                zero_line<OUTL != 0>(T + 16384);
            }
        } else {
            B = A;
            if (valid1) load_tile_half<D, BITS, OUTL, RAW>(a, pr, h, l1 * a.H + h, ti1, r, id1, 0, A);
            if (use > 0 && !wait(&pr.freeb[b], (use - 1) & 1, vfail, a.wait_ns)) return;
            if (valid) {
                decode_store_half<BITS, OUTL != 0, (OUTL != 0 || PSAC)>(B, T, r);
                if constexpr (OUTL != 0) patch_outliers<D, BITS, OUTL>(a, pr.cent, B, hl0, ti0.chunk, id0, 0, T, r);
            } else {
                zero_line<OUTL != 0>(T);
            }
        }
        if constexpr (PSAC) {
            if (pr.pbuf && last) {
                const float S = f16_to_f32(static_cast<uint16_t>(ps));
                float pk[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    pk[k] = S * static_cast<float>(static_cast<int8_t>((pv.x >> (8 * k)) & 0xff));
                    pk[k + 4] = S * static_cast<float>(static_cast<int8_t>((pv.y >> (8 * k)) & 0xff));
                }
                *reinterpret_cast<uint4 *>(pr.pbuf + b * 4096 + (r >> 3) * 256 + (r & 7) * 16) =
                    make_uint4(h2(pk[0], pk[1]), h2(pk[2], pk[3]), h2(pk[4], pk[5]), h2(pk[6], pk[7]));
            }
        }
        umma::fence_proxy_async_smem();
        umma::mbar_arrive(&pr.full[b]);
        ti0 = ti1;
        l0 = l1;
        id0 = id1;
        v0 = v1;
        ti1 = ti2;
        l1 = l2;
        id1 = id2;
        v1 = v2;
    }
}

// The outlier-split variant, out of line so that its register allocation
// stays apart from the plain path's (inlined, both spill).
template <int D, int BITS, int NG>
__device__ __noinline__ void produce_fast_outl(const AttnWsArgs &a, const Producer &pr, int h, int r, int tb,
                                               int n_tiles, volatile int *vfail, int L) {
    const Producer prv = pr;  // the role's pointers in registers, read once
    produce_fast<D, BITS, NG, true>(a, prv, h, r, tb, n_tiles, vfail, L);
}

// The outlier split together with PSAC (every other case takes the fast
// producer, one stage per buffer fill).  Work runs in steps of one 32-channel quarter of the slot's row and one
// stage, in the order (tile, quarter, stage).  Each step's codes, scales,
// centroid slice and outlier entries are loaded one step ahead (register
// sets A and B); the next tile's stage ids, table entry and PSAC codes one
// tile ahead.  A quarter's stages accumulate in fp32 as
// acc = fl(acc + fl(S q + c)) -- S q is exact (an fp16 scale times a code
// of at most 4 bits), so one FMA gives the stage value -- with fl(o + c) at
// a channel the stage split off; after the last stage the PSAC term
// sum_k P_hat_k U_jk (fp32 FMA chain, ascending k) is added and the quarter
// is rounded to fp16 and stored.
template <int BITS>
struct QuarterData {
    uint32_t cw[BITS];  // 32 codes
    uint32_t s2[2];     // fp16 scales of the four 8-channel blocks, two per word
    uint4 cr[4];        // 32 bf16 centroid channels (a raw tile: the row itself)
    uint32_t oe;        // per 8-channel block (byte b): the element split off, 0xFF none
    uint2 ov;           // and its fp16 value (half b)
};

// Stage l's cluster id from four words of packed 8-bit ids (L <= 16).
__device__ __forceinline__ int stage_id(const uint32_t (&w)[4], int l) {
    uint32_t x = w[0];
    x = l >= 4 ? w[1] : x;
    x = l >= 8 ? w[2] : x;
    x = l >= 12 ? w[3] : x;
    return static_cast<int>((x >> (8 * (l & 3))) & 0xFFu);
}

template <int D>
__device__ __forceinline__ void load_stage_ids(const AttnWsArgs &a, const Producer &pr, int h, const TileInfo &ti,
                                               int r, uint32_t (&w)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = 0u;
    if (a.C == 0 || ti.chunk < 0 || r >= ti.nvalid) return;
    for (int l = 0; l < a.L; ++l) {
        const uint32_t v = pr.ids[(static_cast<size_t>(l) * a.H + h) * a.cap + ti.base + r];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (i == (l >> 2)) w[i] |= v << (8 * (l & 3));
    }
}

template <int D, int BITS, bool OUTL>
__device__ __forceinline__ void load_quarter(const AttnWsArgs &a, const Producer &pr, int h, const TileInfo &ti,
                                             int r, int id, int l, int qt, QuarterData<BITS> &qd) {
#pragma unroll
    for (int i = 0; i < BITS; ++i) qd.cw[i] = 0u;
    qd.s2[0] = qd.s2[1] = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) qd.cr[i] = make_uint4(0, 0, 0, 0);
    qd.oe = 0xFFFFFFFFu;
    qd.ov = make_uint2(0, 0);
    if (r >= ti.nvalid) return;
    if (ti.chunk < 0) {  // a raw row (the current chunk's or an anchor's), in stage 0
        if (l == 0) {
            const uint16_t *row =
                (ti.chunk == -2 ? pr.anch : pr.raw) + (static_cast<size_t>(ti.base + r) * a.H + h) * D + qt * 32;
#pragma unroll
            for (int i = 0; i < 4; ++i) qd.cr[i] = *reinterpret_cast<const uint4 *>(row + 8 * i);
        }
        return;
    }
    const int ng = D >> a.glog2;
    const size_t srow = (static_cast<size_t>(l) * a.H + h) * a.cap + ti.base + r;
    const uint8_t *cp = pr.codes + srow * (D * BITS / 8) + qt * (4 * BITS);
    if constexpr (BITS == 2) {
        const uint2 u = *reinterpret_cast<const uint2 *>(cp);
        qd.cw[0] = u.x;
        qd.cw[1] = u.y;
    } else {
        const uint4 u = *reinterpret_cast<const uint4 *>(cp);
        qd.cw[0] = u.x;
        qd.cw[1] = u.y;
        qd.cw[2] = u.z;
        qd.cw[3] = u.w;
    }
    if (a.group >= 32) {
        const uint32_t s0 = pr.scales[srow * ng + ((qt * 32) >> a.glog2)];
        qd.s2[0] = qd.s2[1] = s0 | (s0 << 16);
    } else {
#pragma unroll
        for (int b = 0; b < 4; ++b)
            qd.s2[b >> 1] |= static_cast<uint32_t>(pr.scales[srow * ng + ((qt * 32 + 8 * b) >> a.glog2)]) << (16 * (b & 1));
    }
    if (a.C > 0) {
        const uint16_t *crow =
            pr.cent + ((static_cast<size_t>(l) * a.H + h) * a.max_chunks + ti.chunk) * a.C * D + static_cast<size_t>(id) * D +
            qt * 32;
#pragma unroll
        for (int i = 0; i < 4; ++i) qd.cr[i] = *reinterpret_cast<const uint4 *>(crow + 8 * i);
    }
    if constexpr (OUTL) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int gi = (qt * 32 + 8 * b) >> a.glog2;
            const int oi = pr.outi[srow * ng + gi];
            const int e = gi * a.group + oi - (qt * 32 + 8 * b);
            if (oi != 0xFF && e >= 0 && e < 8) {
                qd.oe = (qd.oe & ~(0xFFu << (8 * b))) | (static_cast<uint32_t>(e) << (8 * b));
                const uint32_t o = pr.outv[srow * ng + gi];
                if (b < 2)
                    qd.ov.x |= o << (16 * b);
                else
                    qd.ov.y |= o << (16 * (b - 2));
            }
        }
    }
}

// acc (16 packed fp32 pairs) += this stage's values of the quarter.
template <int BITS, bool OUTL>
__device__ __forceinline__ void accumulate_quarter(const QuarterData<BITS> &qd, uint64_t (&acc)[16]) {
    constexpr uint32_t M = (1u << BITS) - 1u, MAGIC = 0x4B000000u;
    constexpr float E23 = 8388608.0f, HALF = static_cast<float>(1 << (BITS - 1));
    const uint64_t P2 = pk2(1.0f, 1.0f / static_cast<float>(1 << BITS));
    const uint64_t N2 = pk2(-(E23 + HALF), -(E23 / static_cast<float>(1 << BITS) + HALF));
    const uint64_t ONE2 = pk2(1.0f, 1.0f);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t blk = qd.cw[(8 * b * BITS) / 32] >> ((8 * b * BITS) % 32);
        const float S = f16_to_f32(static_cast<uint16_t>(qd.s2[b >> 1] >> (16 * (b & 1))));
        const uint64_t S2 = pk2(S, S);
        const uint32_t c4[4] = {qd.cr[b].x, qd.cr[b].y, qd.cr[b].z, qd.cr[b].w};
        const uint32_t eo = (qd.oe >> (8 * b)) & 0xFFu;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t x = blk >> (2 * k * BITS);
            const uint64_t mag = pk2(__uint_as_float((x & M) | MAGIC), __uint_as_float((x & (M << BITS)) | MAGIC));
            uint64_t v2 = fma2(S2, fma2(mag, P2, N2),
                               pk2(__uint_as_float(c4[k] << 16), __uint_as_float(c4[k] & 0xffff0000u)));
            if (OUTL && (eo >> 1) == static_cast<uint32_t>(k)) {  // code 0 there: v = c, becomes fl(o + c)
                const float o = f16_to_f32(static_cast<uint16_t>((b < 2 ? qd.ov.x : qd.ov.y) >> (16 * (b & 1))));
                float v0, v1;
                up2(v2, v0, v1);
                if (eo & 1u)
                    v1 = __fadd_rn(o, v1);
                else
                    v0 = __fadd_rn(o, v0);
                v2 = pk2(v0, v1);
            }
            acc[4 * b + k] = fma2(acc[4 * b + k], ONE2, v2);
        }
    }
}

template <int D, int BITS, bool OUTL>
__device__ __noinline__ void produce_general(const AttnWsArgs &a, const Producer &pr, int h, int r, int tb,
                                             int n_tiles, volatile int *vfail) {
    constexpr int KB = D / 64, TB = KB * 16384, Q = D / 32;
    const int L = a.L, per_tile = Q * L;
    const long long total = static_cast<long long>(n_tiles) * per_tile;
    TileInfo ti{}, tn{};
    uint32_t idw[4], idn[4];
    float pk[QVG_PSAC_RANK];
    if (n_tiles > 0) {
        ti = tile_at<true>(a, pr.tab, pr.tab_n, tb, 0);
        load_stage_ids<D>(a, pr, h, ti, r, idw);
    }
    if (n_tiles > 1) {
        tn = tile_at<true>(a, pr.tab, pr.tab_n, tb, 1);
        load_stage_ids<D>(a, pr, h, tn, r, idn);
    }
    QuarterData<BITS> cur, nxt;
    if (total > 0) load_quarter<D, BITS, OUTL>(a, pr, h, ti, r, stage_id(idw, 0), 0, 0, cur);
    uint64_t acc[16];
    int t = 0, qt = 0, l = 0;
    for (long long u = 0; u < total; ++u) {
        if (qt == 0 && l == 0) {
            // start of tile t: its PSAC codes (used after the first quarter's stages)
            if (pr.psac && ti.chunk >= 0 && r < ti.nvalid) {
                const size_t prow = static_cast<size_t>(h) * a.cap + ti.base + r;
                const float pS = f16_to_f32(a.psac_s[prow]);
                const int2 pv = *reinterpret_cast<const int2 *>(a.psac_p + prow * QVG_PSAC_RANK);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    pk[k] = pS * static_cast<float>(static_cast<int8_t>((pv.x >> (8 * k)) & 0xff));
                    pk[k + 4] = pS * static_cast<float>(static_cast<int8_t>((pv.y >> (8 * k)) & 0xff));
                }
            }
        }
        // prefetch step u + 1
        int l1 = l + 1, q1 = qt, t1 = t;
        if (l1 == L) {
            l1 = 0;
            if (++q1 == Q) {
                q1 = 0;
                ++t1;
            }
        }
        if (u + 1 < total) {
            if (t1 == t)
                load_quarter<D, BITS, OUTL>(a, pr, h, ti, r, stage_id(idw, l1), l1, q1, nxt);
            else
                load_quarter<D, BITS, OUTL>(a, pr, h, tn, r, stage_id(idn, l1), l1, q1, nxt);
        }
        if (l == 0) {
#pragma unroll
            for (int k = 0; k < 16; ++k) acc[k] = 0ull;
        }
        accumulate_quarter<BITS, OUTL>(cur, acc);
        if (l == L - 1) {
            const int b = t % kNbuf, use = t / kNbuf;
            uint8_t *T = pr.buf0 + b * TB + r * 128;
            if (qt == 0 && use > 0 && !wait(&pr.freeb[b], (use - 1) & 1, vfail, a.wait_ns)) return;
            float v[32];
#pragma unroll
            for (int k = 0; k < 16; ++k) up2(acc[k], v[2 * k], v[2 * k + 1]);
            if (pr.psac && ti.chunk >= 0 && r < ti.nvalid) {
                const float *U = a.psac_basis + ((static_cast<size_t>(ti.chunk) * a.H + h) * D + qt * 32) * QVG_PSAC_RANK;
#pragma unroll 4
                for (int e = 0; e < 32; ++e) {
                    const float4 u0 = *reinterpret_cast<const float4 *>(U + e * QVG_PSAC_RANK);
                    const float4 u1 = *reinterpret_cast<const float4 *>(U + e * QVG_PSAC_RANK + 4);
                    float corr = 0.0f;
                    corr = fmaf(pk[0], u0.x, corr);
                    corr = fmaf(pk[1], u0.y, corr);
                    corr = fmaf(pk[2], u0.z, corr);
                    corr = fmaf(pk[3], u0.w, corr);
                    corr = fmaf(pk[4], u1.x, corr);
                    corr = fmaf(pk[5], u1.y, corr);
                    corr = fmaf(pk[6], u1.z, corr);
                    corr = fmaf(pk[7], u1.w, corr);
                    v[e] = v[e] + corr;
                }
            }
            const int kb = qt >> 1, c0 = (qt & 1) * 4;
#pragma unroll
            for (int x = 0; x < 4; ++x)
                *reinterpret_cast<uint4 *>(T + kb * 16384 + (((c0 + x) ^ (r & 7)) << 4)) =
                    make_uint4(h2(v[8 * x], v[8 * x + 1]), h2(v[8 * x + 2], v[8 * x + 3]),
                               h2(v[8 * x + 4], v[8 * x + 5]), h2(v[8 * x + 6], v[8 * x + 7]));
            if (qt == Q - 1) {
                umma::fence_proxy_async_smem();
                umma::mbar_arrive(&pr.full[b]);
            }
        }
        cur = nxt;
        if (t1 != t) {  // next tile: shift the tile state, fetch the one after
            ti = tn;
#pragma unroll
            for (int i = 0; i < 4; ++i) idw[i] = idn[i];
            if (t1 + 1 < n_tiles) {
                tn = tile_at<true>(a, pr.tab, pr.tab_n, tb, t1 + 1);
                load_stage_ids<D>(a, pr, h, tn, r, idn);
            }
        }
        t = t1;
        qt = q1;
        l = l1;
    }
}

}  // namespace ws

// Warp roles (16 warps):
//   0-3, 4-7   softmax + epilogue of query tile i = 0 / 1 (thread = query row);
//              lane 0 of warp 5i issues the tcgen05.mma of tile i, and warp 0
//              owns the TMEM allocation
//   8-11       K producers: rebuild the 128-slot K_hat tile (thread = slot)
//   12-15      V producers: the same for V_hat
// Both producers write a tile as [64-channel block][slot][64 channels] with
// the 128-byte swizzle: K-major for the S = Q K_hat^T product (N = slots,
// K = channels) and, read through an MN-major descriptor, the B operand of
// O += P V_hat (N = channels, K = slots), so V needs no transpose.  K and V
// tiles rotate through kNbuf buffers each.
// P_i(t) is written in fp16 over the first 64 columns of S_i(t) in TMEM and
// is the A operand of PV_i(t), read from TMEM.  Once the group's four warps
// have written P_i(t), its issuer issues PV_i(t) and then S_i(t + 1); the
// tensor pipe runs one thread's MMAs in issue order, so S_i(t + 1)
// overwrites P_i(t) only after PV_i(t) has read it, and the commit that
// reports S_i(t + 1) also reports PV_i(t): once group i sees S_i(t + 1), O_i
// is settled and may be rescaled.  Issuing holds the issuing thread until
// the tensor pipe takes the MMA, but here the whole group waits for
// S_i(t + 1) at that point anyway.  The two groups run in step: the
// tensor pipe's N = 128 products lose about 40 % of their rate while other
// warps stream TMEM loads and stores, and a group's softmax alone on its
// sub-partitions is latency-bound, so overlapping one group's products
// with the other's softmax (issue turns) measured slower.
// mbarriers (phase = tile index / kNbuf for the buffers, tile index else):
//   kfull/vfull  producers -> issuers   tile written (one arrival per slot)
//   kfree/vfree  MMA commits -> producer tile consumed (S_0 and S_1 / PV_0 and PV_1;
//                S_0 / PV_0 alone when query tile 1 is past Nq)
//   sfull[i]     MMA commit -> group i   S_i(t) ready (and PV_i(t - 1) done)
//   pfull[i]     group i -> its issuer   P_i(t) in TMEM, O_i rescaled (one arrival per warp)
//   ofull[i]     MMA commit -> group i   the last PV_i done (epilogue)
// MODE 0: one-stage caches without the outlier split or PSAC, no raw tiles;
// MODE 1: no outlier split or PSAC, with raw bf16 tiles (the current chunk,
//         anchor chunks) or several stages (one buffer fill per stage);
// MODE 2: the outlier split (out-of-line producers: per-stage fills
//         without PSAC, else the general producer, which sums the stages and
//         adds PSAC itself);
// MODE 3: PSAC on K without the outlier split (raw tiles and stages allowed):
//         the correction runs on the tensor core as S_i += (Q_i U_c) P_hat^T,
//         one K = 16 product after each tile's S batch.  Q_i U_c (fp16, 128 x 8, computed
//         in fp32 by the softmax threads when a chunk c starts) and P_hat
//         (written by the K producers) are no-swizzle K-major operands of
//         4 KB, zero in columns 8..15; the tile table is cut to 2048 entries
//         to make room.
// Separate instantiations keep the out-of-line producers' call sites, which
// cost the plain kernel 7 % when present, out of modes 0 and 1.
// LS >= 1: LS stages per tile, one buffer fill each, known at compile time
// (with LS = 1 every pseudo-tile index is a tile index; LS = 2 serves
// two-stage QVG-Pro caches, 3.90 -> 3.81 ms against the run-time count);
// LS = 0: a.L stages.
template <int D, int BITS, bool TOP1, int MODE, int LS>
__global__ void __launch_bounds__(ws::kThreads, 1) k_attention_ws(AttnWsArgs a) {
    using namespace ws;
    constexpr int KB = D / 64;
    constexpr int TB = KB * 16384;  // one 128 x D fp16 tile
    constexpr bool PTC = MODE == 3;
    constexpr int kTab = PTC ? 2048 : kTabMax;
    extern __shared__ __align__(1024) uint8_t sm_raw[];
    uint8_t *sm = sm_raw + ((1024u - (umma::smem_u32(sm_raw) & 1023u)) & 1023u);
    uint8_t *Q0 = sm, *Q1 = Q0 + TB, *Kt0 = Q1 + TB, *Vt0 = Kt0 + kNbuf * TB;
    uint8_t *PA = Vt0 + kNbuf * TB, *PB = PA + 2 * 4096;  // MODE 3: Q_i U_c (two), P_hat (kNbuf)
    __shared__ uint64_t kfull[kNbuf], kfree[kNbuf], vfull[kNbuf], vfree[kNbuf], sfull[2], pfull[2], ofull[2], drain,
        never;
    __shared__ uint32_t tmem_base;
    __shared__ int fail;
    __shared__ int2 tile_tab[kTab];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hq = blockIdx.y, h = hq / a.grp, q0 = blockIdx.x * 256;
    // split z of gridDim.z takes cache tiles [tb, tb + n_tiles); every barrier
    // phase below counts tiles from tb
    const int n_all = a.n_ctiles + ceil_div(a.n_raw, QVG_TILE), z = blockIdx.z;
    const int tb = static_cast<int>(static_cast<long long>(n_all) * z / gridDim.z);
    const int n_tiles = static_cast<int>(static_cast<long long>(n_all) * (z + 1) / gridDim.z) - tb;
    // query tiles with at least one query row: a second tile past Nq issues
    // no products and runs no softmax
    const int n_grp = q0 + 128 < a.Nq ? 2 : 1;
    // buffer fills per tile: one per stage, except where a producer sums the
    // stages itself (the general producer of mode 2)
    const int n_stage = LS >= 1 ? LS : (MODE == 2 && a.psac_p) ? 1 : a.L;
    static_assert(MODE >= 0 && MODE <= 3 && (LS == 1 || MODE != 0), "attention mode");

    // Q tiles -> fp16 (exact for bf16 values in fp16's normal range), swizzled K-major
    for (int i = tid; i < 256 * (D / 8); i += kThreads) {
        const int rr = i / (D / 8), ci = i % (D / 8), kb = ci >> 3, c = ci & 7;
        const int r = rr & 127;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (q0 + rr < a.Nq) {
            v = bf16x8_to_f16(
                *reinterpret_cast<const uint4 *>(a.q + (static_cast<size_t>(q0 + rr) * a.Hq + hq) * D + ci * 8));
        }
        *reinterpret_cast<uint4 *>((rr < 128 ? Q0 : Q1) + kb * 16384 + r * 128 + ((c ^ (r & 7)) << 4)) = v;
    }
    for (int j = tid; j < min(n_tiles, kTab); j += kThreads) tile_tab[j] = tile_entry<MODE != 0>(a, tb + j);
    if constexpr (PTC) {
        for (int j = tid; j < (2 + kNbuf) * 4096 / 16; j += kThreads) reinterpret_cast<uint4 *>(PA)[j] = make_uint4(0, 0, 0, 0);
    }
    if (warp == 0) {
        umma::tmem_alloc(&tmem_base, 512);
        umma::tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < kNbuf; ++b) {
            umma::mbar_init(&kfull[b], 128);
            umma::mbar_init(&kfree[b], n_grp);
            umma::mbar_init(&vfull[b], 128);
            umma::mbar_init(&vfree[b], n_grp);
        }
        for (int i = 0; i < 2; ++i) {
            umma::mbar_init(&sfull[i], 1);
            umma::mbar_init(&pfull[i], 4);
            umma::mbar_init(&ofull[i], 1);
        }
        umma::mbar_init(&drain, n_grp);  // the issuing lanes
        umma::mbar_init(&never, 1);  // nothing arrives: the bounded-wait test hook
        umma::fence_barrier_init();
        fail = 0;
    }
    umma::fence_proxy_async_smem();
    umma::tc_fence_before();
    __syncthreads();
    umma::tc_fence_after();
    const uint32_t tmem = tmem_base;
    volatile int *vfail = &fail;

    if (warp < 4 * n_grp) {
        // ------------------------------------------------ softmax of tile i
        const int i = warp >> 2, r = tid & 127;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + i * 128 + lane_off, tO = tmem + 256 + i * 128 + lane_off;
        // the issuing lanes sit in warps 0 and 5, on two different
        // sub-partitions (warp w runs on sub-partition w % 4): on one they
        // shared its issue slots with two producer warps, and the kernel
        // took 4 % longer
        const bool issuer = (warp & 3) == i && lane == 0;
        const uint32_t idS = umma::idesc_f16(128, 128, 0), idO = umma::idesc_f16_bmn(128, D, 0);
        const uint32_t qa = umma::smem_u32(i ? Q1 : Q0), ka = umma::smem_u32(Kt0), va = umma::smem_u32(Vt0);
        const uint32_t pa = umma::smem_u32(PA + i * 4096), pb = umma::smem_u32(PB);
        // MODE 3: row r of Q_i U_c, fp32 FMAs in ascending channel order, to fp16
        int a_chunk = -1;
        auto psac_qu = [&](int c) {
            const float *U = a.psac_basis + (static_cast<size_t>(c) * a.H + h) * D * QVG_PSAC_RANK;
            const uint8_t *Qi = i ? Q1 : Q0;
            float acc[QVG_PSAC_RANK];
#pragma unroll
            for (int k = 0; k < QVG_PSAC_RANK; ++k) acc[k] = 0.0f;
#pragma unroll 1
            for (int ci = 0; ci < D / 8; ++ci) {
                const uint4 qv = *reinterpret_cast<const uint4 *>(Qi + (ci >> 3) * 16384 + r * 128 + (((ci & 7) ^ (r & 7)) << 4));
                const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float q = f16_to_f32(static_cast<uint16_t>(qw[e >> 1] >> (16 * (e & 1))));
                    const float4 u0 = *reinterpret_cast<const float4 *>(U + (ci * 8 + e) * QVG_PSAC_RANK);
                    const float4 u1 = *reinterpret_cast<const float4 *>(U + (ci * 8 + e) * QVG_PSAC_RANK + 4);
                    acc[0] = fmaf(q, u0.x, acc[0]);
                    acc[1] = fmaf(q, u0.y, acc[1]);
                    acc[2] = fmaf(q, u0.z, acc[2]);
                    acc[3] = fmaf(q, u0.w, acc[3]);
                    acc[4] = fmaf(q, u1.x, acc[4]);
                    acc[5] = fmaf(q, u1.y, acc[5]);
                    acc[6] = fmaf(q, u1.z, acc[6]);
                    acc[7] = fmaf(q, u1.w, acc[7]);
                }
            }
            *reinterpret_cast<uint4 *>(PA + i * 4096 + (r >> 3) * 256 + (r & 7) * 16) =
                make_uint4(h2(acc[0], acc[1]), h2(acc[2], acc[3]), h2(acc[4], acc[5]), h2(acc[6], acc[7]));
            umma::fence_proxy_async_smem();
            a_chunk = c;
        };
        if constexpr (PTC) {
            // the first chunk's Q_i U, complete before this group's first S product
            if (n_tiles > 0) {
                const int c0 = tile_at<true>(a, tile_tab, kTab, tb, 0).chunk;
                if (c0 >= 0) psac_qu(c0);
            }
            asm volatile("bar.sync %0, 128;" ::"r"(1 + i) : "memory");
        }
        // S_i(t) = Q_i K(t)^T into TMEM columns [128 i, 128 i + 128) once K(t)
        // is written (rolled issue loops: a descriptor's low 14 bits are the
        // shared address / 16, which these offsets never carry out of)
        // (stage l of tile t is K buffer fill u = t n_stage + l; the stages
        // accumulate into S_i, and the PSAC product follows the last one)
        auto issue_S = [&](int t) -> bool {
            const uint64_t dq = umma::desc_sw128(qa);
            for (int l = 0; l < n_stage; ++l) {
                const int u = t * n_stage + l, b = u % kNbuf;
                if (!ws::wait(&kfull[b], (u / kNbuf) & 1, vfail, a.wait_ns)) return false;
                umma::tc_fence_after();
                const uint64_t dk = umma::desc_sw128(ka + b * TB);
#pragma unroll 1
                for (int s = 0; s < D / 16; ++s) {
                    const uint32_t off16 = ((s >> 2) * 16384 + (s & 3) * 32) >> 4;
                    umma::mma_f16(tmem + i * 128, dq + off16, dk + off16, idS, (l | s) != 0);
                }
                if (l == n_stage - 1) {
                    if constexpr (PTC)
                        umma::mma_f16(tmem + i * 128, umma::desc_noswz(pa, 128, 256),
                                      umma::desc_noswz(pb + b * 4096, 128, 256), idS, 1u);
                    umma::mma_commit(&sfull[i]);
                }
                umma::mma_commit(&kfree[b]);
            }
            return true;
        };
        bool live = true;
        if (issuer && n_tiles > 0) {
            live = issue_S(0);
            // test hook: with S_i(0) in flight, wait on a barrier that nothing
            // completes; the bound runs out, every role stops, and the drain
            // below waits for the MMA
            if (live && a.inject && !ws::wait(&never, 0, vfail, a.wait_ns)) live = false;
        }
        live = __all_sync(0xffffffffu, live);
        float m_used = -INFINITY, l_sum = 0.0f, best = -INFINITY;
        int best_slot = 0;
        for (int t = 0; t < n_tiles && live; ++t) {
            const TileInfo ti = tile_at<MODE != 0>(a, tile_tab, kTab, tb, t);
            live = __all_sync(0xffffffffu, ws::wait(&sfull[i], t & 1, vfail, a.wait_ns));
            if (!live) break;
            umma::tc_fence_after();
            // row maximum of the raw logits (the scale is positive), scaled
            // once; the top-1 variant keeps one in-order chain so that ties
            // resolve to the lowest slot
            float rmax = -INFINITY;
            int targ = 0;
            if constexpr (TOP1) {
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    uint32_t v[32];
                    umma::tmem_ld32(tS + c0, v);
                    umma::tmem_ld_wait_regs(v);
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
                    umma::tmem_ld_wait_regs(v);
                    if (c0 + 32 <= ti.nvalid) {
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            m4[k & 3] = max3(m4[k & 3], __uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
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
                    best_slot = (tb + t) * QVG_TILE + targ;
                }
            }
            float corr = 1.0f;
            bool rescale = false;
            if (tmax > m_used + kRescale) {
                corr = ex2(m_used - tmax);
                rescale = t > 0;
                m_used = tmax;
            }
            // PV_i(t - 1) is done (reported with S_i(t)): O_i may be rescaled
            if (__any_sync(0xffffffffu, rescale)) {
                const float f = rescale ? corr : 1.0f;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t v[32];
                    umma::tmem_ld32(tO + c0, v);
                    umma::tmem_ld_wait_regs(v);
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * f);
                    umma::tmem_st32(tO + c0, v);
                }
            }
            const uint64_t sl2 = pk2(a.scale_log2, a.scale_log2), nm2 = pk2(-m_used, -m_used);
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            // P_i(t) over S_i(t): chunk c0 of S (columns [c0, c0 + 32)) becomes
            // columns [c0 / 2, c0 / 2 + 16), which hold logits already read
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t v[32], pk[16];
                umma::tmem_ld32(tS + c0, v);
                umma::tmem_ld_wait_regs(v);
                softmax_chunk(v, c0, ti.nvalid, sl2, nm2, pk, acc);
                umma::tmem_st16(tS + c0 / 2, pk);
            }
            l_sum = l_sum * corr + ((acc[0] + acc[1]) + (acc[2] + acc[3]));
            if constexpr (PTC) {
                // S_i(t + 1) is issued after this group's P_i(t): Q_i U of its
                // chunk goes in now (S_i(t), the last reader, has completed)
                if (t + 1 < n_tiles) {
                    const int c1 = tile_at<true>(a, tile_tab, kTab, tb, t + 1).chunk;
                    if (c1 >= 0 && c1 != a_chunk) psac_qu(c1);
                }
            }
            umma::tmem_st_wait();
            umma::tc_fence_before();
            __syncwarp();
            if (lane == 0) umma::mbar_arrive(&pfull[i]);
            if (issuer) {
                // O_i += P_i(t) V(t), P_i from TMEM (columns [128 i, 128 i + 64)),
                // once all four warps have written P_i(t), one product per
                // stage of V(t); then S_i(t + 1)
                bool ok = ws::wait(&pfull[i], t & 1, vfail, a.wait_ns);
                for (int l = 0; ok && l < n_stage; ++l) {
                    const int u = t * n_stage + l, b = u % kNbuf;
                    ok = ws::wait(&vfull[b], (u / kNbuf) & 1, vfail, a.wait_ns);
                    if (!ok) break;
                    umma::tc_fence_after();
                    const uint64_t dv = umma::desc_sw128_mn(va + b * TB, 16384);
#pragma unroll 1
                    for (int s = 0; s < 8; ++s)
                        umma::mma_f16_ts(tmem + 256 + i * 128, tmem + i * 128 + s * 8, dv + ((s * 2048) >> 4), idO,
                                         (t | l | s) != 0);
                    umma::mma_commit(&vfree[b]);
                }
                if (ok) {
                    if (t + 1 < n_tiles)
                        ok = issue_S(t + 1);
                    else
                        umma::mma_commit(&ofull[i]);
                }
                live = ok;
            }
            live = __all_sync(0xffffffffu, live);
        }
        // epilogue: O_i / l
        bool ok = live && !*vfail && n_tiles > 0 && ws::wait(&ofull[i], 0, vfail, a.wait_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            umma::tc_fence_after();
            const int qi = q0 + i * 128 + r;
            const float inv = 1.0f / l_sum;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t v[32];
                umma::tmem_ld32(tO + c0, v);
                umma::tmem_ld_wait_regs(v);
                if (qi < a.Nq) {
                    // split z writes its own [Nq][Hq][D] slice (z = 0 without a split)
                    const size_t o = ((static_cast<size_t>(z) * a.Nq + qi) * a.Hq + hq) * D + c0;
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
                const size_t li = (static_cast<size_t>(z) * a.Hq + hq) * a.Nq + qi;
                if (a.lse) a.lse[li] = (m_used + log2f(l_sum)) * 0.69314718055994531f;
                if constexpr (TOP1) {
                    a.top1[li] = best_slot;
                    if (a.best) a.best[li] = best;
                }
            }
        }
        // every MMA this group issued completes before TMEM is released
        if (issuer) {
            umma::mma_commit(&drain);
            umma::mbar_wait(&drain, 0, kWaitNs);
        }
    } else if (warp >= 8) {
        // ------------------------------------------------ K / V producers (thread = slot)
        const bool isv = warp >= 12;
        const Producer pr{isv ? a.vcodes : a.kcodes, isv ? a.vscales : a.kscales, isv ? a.vids : a.kids,
                          isv ? a.vcent : a.kcent, isv ? a.vraw : a.kraw, isv ? a.vanch : a.kanch,
                          isv ? a.voutv : a.koutv,
                          isv ? a.vouti : a.kouti, isv ? Vt0 : Kt0, isv ? vfull : kfull,
                          isv ? vfree : kfree,
                          !isv && a.psac_p != nullptr, tile_tab, kTab, PTC && !isv ? PB : nullptr};
        if constexpr (MODE == 0) {
            produce_fast<D, BITS, 0, false>(a, pr, h, tid & 127, tb, n_tiles, vfail);
        } else if constexpr (MODE == 3) {
            // one call site for both roles (two inlined copies of the producer
            // loop cost 60 %, as the roles' code then competes for the
            // instruction cache); the V role has no P_hat buffer and skips
            // the PSAC part at run time
            produce_fast<D, BITS, 0, true, true>(a, pr, h, tid & 127, tb, n_tiles, vfail, n_stage);
        } else if constexpr (MODE == 1) {
            produce_fast<D, BITS, 0, true>(a, pr, h, tid & 127, tb, n_tiles, vfail, n_stage);
        } else {
            // the outlier split: one stage per fill through the fast producer
            // when PSAC is off, else the general producer, which sums the
            // stages and adds the PSAC term itself (n_stage = 1)
            if (!a.psac_p) {
                const int ng = 64 / a.group;  // 1, 2, 4 or 8 (groups of 8 ... 64 channels)
                if (ng == 1)
                    produce_fast_outl<D, BITS, 1>(a, pr, h, tid & 127, tb, n_tiles, vfail, n_stage);
                else if (ng == 2)
                    produce_fast_outl<D, BITS, 2>(a, pr, h, tid & 127, tb, n_tiles, vfail, n_stage);
                else if (ng == 4)
                    produce_fast_outl<D, BITS, 4>(a, pr, h, tid & 127, tb, n_tiles, vfail, n_stage);
                else
                    produce_fast_outl<D, BITS, 8>(a, pr, h, tid & 127, tb, n_tiles, vfail, n_stage);
            }
            else if (pr.outi)
                produce_general<D, BITS, true>(a, pr, h, tid & 127, tb, n_tiles, vfail);
            else
                produce_general<D, BITS, false>(a, pr, h, tid & 127, tb, n_tiles, vfail);
        }
    }
    __syncwarp();
    umma::tc_fence_before();
    __syncthreads();
    if (tid == 0 && *vfail) raise_error(a.err, QVG_ERR_TIMEOUT);
    if (warp == 0) {
        umma::tc_fence_after();
        umma::tmem_dealloc(tmem, 512);
    }
}

template <int D, int BITS, bool TOP1, int MODE, int LS>
static qvg_status attn_ws_t(const AttnWsArgs &a, int a_splits, cudaStream_t st) {
    constexpr size_t smem = (2 + 2 * ws::kNbuf) * (D / 64) * 16384 + (MODE == 3 ? (2 + ws::kNbuf) * 4096 : 0) + 1024;
    {
        static std::atomic<uint64_t> done{0};
        const qvg_status s = smem_limit_once(done, reinterpret_cast<const void *>(k_attention_ws<D, BITS, TOP1, MODE, LS>),
                                             static_cast<int>(smem));
        if (s != QVG_OK) return s;
    }
    dim3 grid(ceil_div(a.Nq, 256), a.Hq, a_splits);
    k_attention_ws<D, BITS, TOP1, MODE, LS><<<grid, ws::kThreads, smem, st>>>(a);
    QVG_LAUNCH_CHECK();
    return QVG_OK;
}

template <int D, int BITS, int MODE, int LS>
static qvg_status attn_ws_m(const AttnWsArgs &a, int splits, cudaStream_t st) {
    return a.top1 ? attn_ws_t<D, BITS, true, MODE, LS>(a, splits, st) : attn_ws_t<D, BITS, false, MODE, LS>(a, splits, st);
}

template <int D, int BITS>
qvg_status attn_ws(const AttnWsArgs &a, int splits, cudaStream_t st) {
    const bool one = a.L == 1;
    if (a.kouti) return one ? attn_ws_m<D, BITS, 2, 1>(a, splits, st) : attn_ws_m<D, BITS, 2, 0>(a, splits, st);
    if (a.psac_p) return one ? attn_ws_m<D, BITS, 3, 1>(a, splits, st) : attn_ws_m<D, BITS, 3, 0>(a, splits, st);
    if (a.L == 2) return attn_ws_m<D, BITS, 1, 2>(a, splits, st);
    if (!one) return attn_ws_m<D, BITS, 1, 0>(a, splits, st);
    if (a.n_raw > 0 || a.chunk_anchor) return attn_ws_m<D, BITS, 1, 1>(a, splits, st);
    return attn_ws_m<D, BITS, 0, 1>(a, splits, st);
}

}  // namespace qvg
