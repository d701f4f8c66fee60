// compress.cu -- write path of the compressed KV cache (sm_103a).
//
// Quant VideoGen notes, "Semantic-Aware Smoothing": per chunk and head,
// k-means over the chunk's tokens, subtract each token's centroid, quantise
// the residual per group; "Progressive Residual Quantization": repeat on the
// dequantisation error for L stages.  QuantWM write-up, QSAC: weight the
// clustering distance per channel by history-query activity; PSAC: project
// the remaining key error on the top-8 query eigenvectors and store it as
// INT8.
//
// Kernels (one chunk, all heads per launch):
//   k_kmeans_init     seeded systematic pick of C tokens as first centroids
//   k_centroid_norms  ||c||_w^2 for the assignment score
//   k_kmeans_assign_tc score(c) = ||c||_w^2 - 2 x.(w*c) on the tensor cores,
//                     argmin with the two best re-scored exactly (lowest c on ties)
//   k_kmeans_update   stable order of a head's tokens by cluster, then the
//                     members summed in token order -> bf16 centroid + norm
//   k_residual_quant  r = x - c_id, per-group scale, codes, packing, stage
//                     residual for the next stage, PSAC INT8 projection
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "umma.cuh"


namespace qvg {

// ---------------------------------------------------------------------------
// k-means initialisation.  Reading (the pages leave the start open): a seeded
// systematic sample, one token in each of C equal strata of the chunk's
// raster order: idx_c = floor((c * 2^32 + u) * N / (C * 2^32)), with u the
// top 32 bits of the first SplitMix64 output (Steele, Lea, Flood 2014) from
// state seed ^ (chunk << 40) ^ (head << 20) ^ stage.
__device__ __forceinline__ uint64_t splitmix64_first(uint64_t state) {
    uint64_t z = state + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

template <int D>
__global__ void k_kmeans_init(const uint16_t *__restrict__ g, int N, int H, int C, int Ce,
                              uint64_t seed, int chunk, int stage, uint16_t *__restrict__ cent,
                              size_t hs, const float *__restrict__ w, float *__restrict__ cnorm) {
    constexpr int E = D / 32;  // channels per lane
    pdl_wait();
    pdl_trigger();
    const int h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x * (blockDim.x >> 5) + warp;
    if (c >= C) return;
    const uint64_t st = seed ^ (static_cast<uint64_t>(chunk) << 40) ^
                        (static_cast<uint64_t>(h) << 20) ^ static_cast<uint64_t>(stage);
    const uint64_t u = splitmix64_first(st) >> 32;
    uint16_t *dst = cent + static_cast<size_t>(h) * hs + static_cast<size_t>(c) * D + lane * E;
    float v[E];
    if (c < Ce) {
        const uint64_t num = ((static_cast<uint64_t>(c) << 32) + u) * static_cast<uint64_t>(N);
        const int idx = static_cast<int>(num / (static_cast<uint64_t>(Ce) << 32));
        const uint16_t *src = g + (static_cast<size_t>(idx) * H + h) * D + lane * E;
        if constexpr (E == 4) {
            const uint2 x = *reinterpret_cast<const uint2 *>(src);
            *reinterpret_cast<uint2 *>(dst) = x;
            v[0] = __uint_as_float(x.x << 16); v[1] = __uint_as_float(x.x & 0xffff0000u);
            v[2] = __uint_as_float(x.y << 16); v[3] = __uint_as_float(x.y & 0xffff0000u);
        } else {
            const uint32_t x = *reinterpret_cast<const uint32_t *>(src);
            *reinterpret_cast<uint32_t *>(dst) = x;
            v[0] = __uint_as_float(x << 16); v[1] = __uint_as_float(x & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) { dst[e] = 0; v[e] = 0.0f; }
    }
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float wj = w ? w[h * D + lane * E + e] : 1.0f;
        s = fmaf(wj * v[e], v[e], s);
    }
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) cnorm[h * C + c] = s;
}

// ||c||_w^2 (fp32) for every centroid; one warp per (head, centroid).
template <int D>
__global__ void k_centroid_norms(const uint16_t *__restrict__ cent, size_t hs, int H, int C,
                                 const float *__restrict__ w, float *__restrict__ cnorm) {
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= H * C) return;
    const int h = gw / C, c = gw % C;
    const uint16_t *row = cent + static_cast<size_t>(h) * hs + static_cast<size_t>(c) * D;
    float s = 0.0f;
    for (int j = lane; j < D; j += 32) {
        const float v = bf16_to_f32(row[j]);
        const float wj = w ? w[h * D + j] : 1.0f;
        s = fmaf(wj * v, v, s);
    }
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) cnorm[h * C + c] = s;
}

// ---------------------------------------------------------------------------
// Assignment on the tensor cores.  A CTA owns one head's centroids (staged
// once in shared memory) and walks several 128-token tiles of that head:
//   F_t[128 x Np] = [X_t | e_t] [B | b]^T,  f_c = x.c - ||c||_w^2/2 - ||x||_w^2/2
// with B = the centroids (bf16, exact) or, with QSAC weights, the weighted
// centroids w*c as a bf16 pair hi + lo (|w c - hi - lo| <= 2^-18 |w c|), and
// one extra K=16 block: e_t = (-1, -1, -1, -x1, -x2, -x3, 0...) per token,
// b = (n1, n2, n3, 1, 1, 1, 0...) per centroid, where x1+x2+x3 and n1+n2+n3
// are ||x||_w^2 / 2 and ||c||_w^2 / 2 split into three bf16 parts (exact to
// 2^-24).  So f_c = -d_c / 2 with d_c = sum_j w_j (x_j - c_j)^2, accumulated in
// fp32 in tensor memory by tcgen05.mma (M=128, N=Np = Ce rounded up to 16).
// Token tiles arrive by TMA (a tensor map over the stage's bf16 [N][H][d]
// operand, 128-byte swizzle, zero fill past N) into NA buffers, the
// centroids likewise once per launch; completion is counted on an mbarrier
// per buffer, and the MMA of tile k+1 runs while the epilogue of tile k reads
// the other accumulator.
//
// Epilogue, thread = token row (the four warp groups take interleaved
// 32-column chunks).  For f <= 0 a larger f has a smaller bit pattern as an
// unsigned integer, so the best clusters are the smallest keys
// (bits(f) with the low 4 bits replaced by the column's place in the
// thread's chain): three unsigned min/max per column keep the two best of
// each of four chains.  A slightly positive f (d within rounding of 0) ranks
// first as well.  The chains and groups are merged in (score, index) order,
// ties to the lower cluster; each warp then finishes 8 rows.
//
// Exactness: the tensor core sums K = D + 16 exact products in steps of 16,
// so the fp32 accumulation makes at most ~25 roundings of at most 2^-23
// (truncation) each, <= 2^-18 of the sum of |terms|; the hi/lo split of w*c
// adds 2^-18 (QSAC), the norm splits 2^-24 and the key truncation 2^-19 |f|.
// With sum w|x c| <= ||x||_w ||c||_w <= (||x||_w^2 + ||c||_w^2) / 2 this
// bounds the error of d_c = -2 f_c by
//   E_c <= 2^-16 (||x||_w^2 + ||c||_w^2) <= 2^-16 (3 ||x||_w^2 + 2 d_c)
// (2^-15 with QSAC), since ||c||_w <= ||x||_w + sqrt(d_c).  The computed
// best b is the exact argmin (no tie possible) when d_c - d_b > E_c + E_b
// for every other c; that margin grows with d_c, so the second best s
// decides it, and with a factor two to spare the test is
//   d_s - d_b > tau (3 ||x||_w^2 + d_s + d_b),  tau = 2^-14 (2^-13 with QSAC).
// Otherwise the two candidates are re-scored with the direct sum: the 32
// lanes of a warp each take D/32 consecutive channels of the row (fp32,
// ascending), the partial sums are added by an xor butterfly, and the smaller
// distance wins (ties to the lower index).  ||x||_w^2 comes from
// k_row_norms, run once per stage.
// Every wait is bounded; on expiry the CTA records QVG_ERR_TIMEOUT.
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s

constexpr int kAssignThreads = 512;
constexpr int kAssignGroups = kAssignThreads / 128;  // warp groups sharing the columns
constexpr float kAssignTau = 1.0f / 16384.0f;  // doubled with QSAC

// v = p0 + p1 + p2 in bf16 parts (each the rounding of what is left)
__device__ __forceinline__ void split3(float v, uint16_t &p0, uint16_t &p1, uint16_t &p2) {
    p0 = f32_to_bf16(v);
    const float r1 = v - bf16_to_f32(p0);
    p1 = f32_to_bf16(r1);
    p2 = f32_to_bf16(r1 - bf16_to_f32(p1));
}
__device__ __forceinline__ uint32_t bf16pair(uint16_t lo, uint16_t hi) {
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}
constexpr uint16_t kBf16One = 0x3f80, kBf16MinusOne = 0xbf80;

// (score, index) order: lower score, then lower index
__device__ __forceinline__ bool sc_less(float a, int ia, float b, int ib) { return a < b || (a == b && ia < ib); }
// merge the ordered pair (ov, oi) <= (pv, pi) into (best, second)
__device__ __forceinline__ void merge2(float &bv, int &bi, float &sv, int &si, float ov, int oi, float pv, int pi) {
    if (sc_less(ov, oi, bv, bi)) {
        if (sc_less(bv, bi, pv, pi)) {
            sv = bv;
            si = bi;
        } else {
            sv = pv;
            si = pi;
        }
        bv = ov;
        bi = oi;
    } else if (sc_less(ov, oi, sv, si)) {
        sv = ov;
        si = oi;
    }
}

template <int D, int P>
__global__ void __launch_bounds__(kAssignThreads, 1) k_kmeans_assign_tc(const __grid_constant__ CUtensorMap tm_x,
                                                            const __grid_constant__ CUtensorMap tm_c,
                                                            const uint16_t *__restrict__ g, int N, int H,
                                                            const uint16_t *__restrict__ cent, size_t hs,
                                                            int Ce, int Np, const float *__restrict__ cnorm,
                                                            int C, const float *__restrict__ w,
                                                            const float *__restrict__ xnorm,
                                                            int32_t *__restrict__ ids, int *err,
                                                            uint64_t wait_ns, int inject) {
    constexpr int KB = D / 64;                       // 64-element K blocks
    constexpr int AB = KB * 128 * 128;               // one token tile
    constexpr int NA = P == 1 ? 3 : 2;               // token tile buffers
    constexpr int E = D / 32;                        // channels per lane in the re-scoring
    extern __shared__ __align__(1024) uint8_t sm_raw[];
    // swizzle atoms need a 1024-byte aligned base (the launch adds 1 KB slack)
    uint8_t *sm = sm_raw + ((1024u - (umma::smem_u32(sm_raw) & 1023u)) & 1023u);
    uint8_t *As = sm;                                // NA x KB x [128 rows x 128 B]
    uint8_t *Ax = As + NA * AB;                      // NA x extra K block of the tokens (4 KB)
    uint8_t *Bs = Ax + NA * 4096;                    // P x KB x [Np rows x 128 B]
    uint8_t *Bx = Bs + static_cast<size_t>(P) * KB * Np * 128;  // extra K block of the centroids
    __shared__ uint64_t bar_mma[2], bar_a[NA], bar_drain, bar_never, bar_cent;
    __shared__ uint32_t tmem_base;
    __shared__ float xs[kAssignGroups][128][2];  // each warp group's two best scores per row
    __shared__ int xk[kAssignGroups][128][2];    // ... and their clusters
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = warp >> 2;       // warp group: 32-column chunks grp, grp + G, ... (G groups)
    const int h = blockIdx.y;
    const int n_tiles = ceil_div(N, 128);
    const int t0 = blockIdx.x, tstep = gridDim.x;
    const int my_tiles = t0 < n_tiles ? ceil_div(n_tiles - t0, tstep) : 0;
    const uint32_t ncols = Np <= 32 ? 32 : (Np <= 64 ? 64 : (Np <= 128 ? 128 : 256));
    const uint16_t *ch = cent + static_cast<size_t>(h) * hs;

    if (warp == 0) {
        umma::tmem_alloc(&tmem_base, 2 * ncols);
        umma::tmem_relinquish();
    }
    if (tid == 0) {
        umma::mbar_init(&bar_mma[0], 1);
        umma::mbar_init(&bar_mma[1], 1);
        umma::mbar_init(&bar_drain, 1);
        umma::mbar_init(&bar_never, 1);  // nothing arrives: the bounded-wait test hook
        umma::mbar_init(&bar_cent, 1);
        // per tile: the TMA's arrival (with its byte count) and one per thread
        // once its part of the extra K block is written
        for (int i = 0; i < NA; ++i) umma::mbar_init(&bar_a[i], kAssignThreads + 1);
        umma::tma_prefetch_map(&tm_x);
        if (P == 1) umma::tma_prefetch_map(&tm_c);
        umma::fence_barrier_init();
    }
    __syncthreads();

    // token tile k -> buffer k % NA: thread 0's TMA arrives on bar_a with the
    // tile's bytes, and each thread arrives once more after its part of the
    // extra K block (core matrix layout: row r, K half kh at (r/8)*256 +
    // kh*128 + (r%8)*16); n_issued counts thread 0's tile copies (for the drain)
    int n_issued = 0;
    auto load_tokens = [&](int k) {
        if (tid == 0) {
            const int n0 = (t0 + k * tstep) * 128;
            uint8_t *dst = As + (k % NA) * AB;
            umma::mbar_arrive_expect_tx(&bar_a[k % NA], AB);
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) umma::tma_load_3d(dst + kb * 16384, &tm_x, kb * 64, h, n0, &bar_a[k % NA]);
            n_issued = k + 1;
        }
    };
    auto load_norms = [&](int k) {
        const int n0 = (t0 + k * tstep) * 128;
        if (tid < 256) {
            const int r = tid >> 1, kh = tid & 1;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (kh == 0) {
                const float xh = n0 + r < N ? 0.5f * xnorm[static_cast<size_t>(h) * N + n0 + r] : 0.0f;
                uint16_t p0, p1, p2;
                split3(-xh, p0, p1, p2);
                v = make_uint4(bf16pair(kBf16MinusOne, kBf16MinusOne), bf16pair(kBf16MinusOne, p0), bf16pair(p1, p2), 0u);
            }
            *reinterpret_cast<uint4 *>(Ax + (k % NA) * 4096 + (r >> 3) * 256 + kh * 128 + (r & 7) * 16) = v;
            umma::fence_proxy_async_smem();
        }
        umma::mbar_arrive(&bar_a[k % NA]);
    };
    auto load_tile = [&](int k) {
        load_tokens(k);
        load_norms(k);
    };

    // before the previous kernel has finished: only the token tiles (this
    // stage's input, complete before the kernels in between began); their
    // norms may come from the kernel just before (the first assignment of a
    // stage follows the row norms), so they are read after the wait
    for (int k = 0; k < NA - 1 && k < my_tiles; ++k) load_tokens(k);
    pdl_wait();
    pdl_trigger();
    for (int k = 0; k < NA - 1 && k < my_tiles; ++k) load_norms(k);
    // centroids (or weighted hi/lo pair) -> swizzled K-major bf16, once; the
    // plain centroids by TMA (rows past C read 0; rows Ce .. C-1, unused
    // clusters, get a huge norm below)
    if constexpr (P == 1) {
        if (tid == 0) {
            umma::mbar_arrive_expect_tx(&bar_cent, KB * Np * 128);
#pragma unroll
            for (int kb = 0; kb < KB; ++kb)
                umma::tma_load_3d(Bs + static_cast<size_t>(kb) * Np * 128, &tm_c, kb * 64, 0, h, &bar_cent);
        }
    } else {
        for (int i = tid; i < Np * (D / 8); i += kAssignThreads) {
            const int r = i / (D / 8), ci = i % (D / 8), kb = ci >> 3, c = ci & 7;
            uint4 v = make_uint4(0, 0, 0, 0), v2 = make_uint4(0, 0, 0, 0);
            if (r < Ce) {
                v = *reinterpret_cast<const uint4 *>(ch + static_cast<size_t>(r) * D + ci * 8);
                uint32_t in[4] = {v.x, v.y, v.z, v.w}, hi[4], lo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint32_t hpair = 0, lpair = 0;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int j = ci * 8 + 2 * k + half;
                        const float cv = bf16_to_f32(static_cast<uint16_t>(in[k] >> (16 * half)));
                        const float wv = w[h * D + j] * cv;
                        const uint16_t hb = f32_to_bf16(wv);
                        const uint16_t lb = f32_to_bf16(wv - bf16_to_f32(hb));
                        hpair |= static_cast<uint32_t>(hb) << (16 * half);
                        lpair |= static_cast<uint32_t>(lb) << (16 * half);
                    }
                    hi[k] = hpair;
                    lo[k] = lpair;
                }
                v = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                v2 = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            const size_t off = static_cast<size_t>(kb) * Np * 128 + r * 128 + ((c ^ (r & 7)) << 4);
            *reinterpret_cast<uint4 *>(Bs + off) = v;
            *reinterpret_cast<uint4 *>(Bs + static_cast<size_t>(KB) * Np * 128 + off) = v2;
        }
    }
    // extra K block of the centroids; padded columns get a huge norm (f far
    // below any real column)
    for (int i = tid; i < 2 * Np; i += kAssignThreads) {
        const int c = i >> 1, kh = i & 1;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (kh == 0) {
            const float nrm = c < Ce ? cnorm[h * C + c] : 2.0e38f;
            uint16_t p0, p1, p2;
            split3(0.5f * nrm, p0, p1, p2);
            v = make_uint4(bf16pair(p0, p1), bf16pair(p2, kBf16One), bf16pair(kBf16One, kBf16One), 0u);
        }
        *reinterpret_cast<uint4 *>(Bx + (c >> 3) * 256 + kh * 128 + (c & 7) * 16) = v;
    }
    // the centroids have landed (every thread reads them in the re-scoring)
    bool c_ok = true;
    if (P == 1) c_ok = umma::mbar_wait(&bar_cent, 0, wait_ns);
    umma::fence_proxy_async_smem();
    umma::tc_fence_before();
    const bool cent_ok = __syncthreads_and(c_ok);
    umma::tc_fence_after();
    const uint32_t tmem = tmem_base;
    const uint32_t idesc = umma::idesc_f16(128, Np, 1);
    const uint32_t b0 = umma::smem_u32(Bs);
    auto issue = [&](int k) {
        const uint32_t a0 = umma::smem_u32(As + (k % NA) * AB);
#pragma unroll 1
        for (int p = 0; p < P; ++p)
#pragma unroll 1
            for (int s = 0; s < D / 16; ++s) {
                const uint64_t ad = umma::desc_sw128(a0 + (s >> 2) * 16384 + (s & 3) * 32);
                const uint64_t bd = umma::desc_sw128(b0 + (p * KB + (s >> 2)) * Np * 128 + (s & 3) * 32);
                umma::mma_f16(tmem + (k & 1) * ncols, ad, bd, idesc, (p | s) != 0);
            }
        umma::mma_f16(tmem + (k & 1) * ncols, umma::desc_noswz(umma::smem_u32(Ax + (k % NA) * 4096), 128, 256),
                      umma::desc_noswz(umma::smem_u32(Bx), 128, 256), idesc, 1u);
        umma::mma_commit(&bar_mma[k & 1]);
    };
    bool ok = cent_ok;
    int n_waited = 0;  // thread 0: tile copies it has waited for
    if (tid == 0 && my_tiles > 0 && ok) {
        if (umma::mbar_wait(&bar_a[0], 0, wait_ns)) {
            n_waited = 1;
            umma::tc_fence_after();
            issue(0);
        } else {
            ok = false;
        }
        // test hook: with tile 0's MMA in flight, wait on a barrier that
        // nothing completes, so that the bound runs out and the drain below
        // has an MMA to wait for
        if (ok && inject && !umma::mbar_wait(&bar_never, 0, wait_ns)) ok = false;
    }
    ok = __syncthreads_and(ok);
    for (int k = 0; ok && k < my_tiles; ++k) {
        const int t = t0 + k * tstep;
        const int buf = k % NA;
        // (1) with three buffers, tile k+1 is already loaded: start its MMA now
        // (its accumulator's previous tile, k-1, ended at the last barrier)
        if (NA == 3 && tid == 0 && k + 1 < my_tiles) {
            if (umma::mbar_wait(&bar_a[(k + 1) % NA], ((k + 1) / NA) & 1, wait_ns)) {
                n_waited = k + 2;
                umma::tc_fence_after();
                issue(k + 1);
            } else {
                ok = false;
            }
        }
        // (2) refill the buffer of tile k - 1 (its epilogue ended at the last barrier)
        if (k + NA - 1 < my_tiles) load_tile(k + NA - 1);
        // (3) epilogue of tile k (every thread also observes tile k's copy: the
        // re-scoring reads rows of it)
        if (!umma::mbar_wait(&bar_mma[k & 1], (k >> 1) & 1, wait_ns)) ok = false;
        if (ok && !umma::mbar_wait(&bar_a[buf], (k / NA) & 1, wait_ns)) ok = false;
        ok = __all_sync(0xffffffffu, ok);  // the TMEM loads below are warp-collective
        umma::tc_fence_after();
        const int r = (warp & 3) * 32 + lane;
        const uint8_t *Ab = As + buf * AB;
        // ||x||_w^2 of the row this lane finishes later (issued before the scan)
        const int fr = 8 * warp + (lane >> 2), fn = t * 128 + fr;
        const float xn_pre = fn < N ? xnorm[static_cast<size_t>(h) * N + fn] : 0.0f;
        uint32_t b1[4], b2[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) b1[q] = b2[q] = 0xffffffffu;
        if (ok) {
            // a thread's columns: chunk m = 0, 1 of 32 at grp*32 + 128 m (Np <= 256);
            // both loads in flight before the one wait
            const uint32_t trow = tmem + (k & 1) * ncols + (static_cast<uint32_t>((warp & 3) * 32) << 16);
            const int ca0 = grp * 32, ca1 = grp * 32 + 128;
            uint32_t acc[2][32];
            if (ca0 < Np) umma::tmem_ld32(trow + ca0, acc[0]);
            if (ca1 < Np) umma::tmem_ld32(trow + ca1, acc[1]);
            umma::tmem_ld_wait_regs(acc[0]);
            umma::reg_fence32(acc[1]);
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int c0 = m ? ca1 : ca0;
                if (c0 >= Np) continue;
                // columns past Np were not written by the MMA: masked in a partial chunk
                const bool full = c0 + 32 <= Np;
#pragma unroll
                for (int kk = 0; kk < 32; ++kk) {
                    uint32_t key = (acc[m][kk] & ~0xfu) | static_cast<uint32_t>((m << 3) | (kk >> 2));
                    if (!full && c0 + kk >= Np) key = 0xffffffffu;
                    const uint32_t hi = max(b1[kk & 3], key);
                    b1[kk & 3] = min(b1[kk & 3], key);
                    b2[kk & 3] = min(b2[kk & 3], hi);
                }
            }
        }
        // keys -> (d, cluster): d = -2 f; an empty slot scores +inf
        float bv[4], sv[4];
        int bi[4], si[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            auto dec = [&](uint32_t key, float &d, int &c) {
                if (key == 0xffffffffu) {
                    d = INFINITY;
                    c = 0x7fffffff;
                } else {
                    d = -2.0f * __uint_as_float(key & ~0xfu);
                    c = grp * 32 + 128 * static_cast<int>((key >> 3) & 1u) + 4 * static_cast<int>(key & 7u) + q;
                }
            };
            dec(b1[q], bv[q], bi[q]);
            dec(b2[q], sv[q], si[q]);
        }
#pragma unroll
        for (int q = 1; q < 4; ++q) merge2(bv[0], bi[0], sv[0], si[0], bv[q], bi[q], sv[q], si[q]);
        xs[grp][r][0] = bv[0];
        xs[grp][r][1] = sv[0];
        xk[grp][r][0] = bi[0];
        xk[grp][r][1] = si[0];
        __syncthreads();
        // finalisation: warp W takes rows 8W .. 8W+7; the four lanes 4l .. 4l+3
        // hold the four groups' pairs of row 8W + l and merge them by xor
        // shuffles, so every lane ends with the row's two best
        {
            const int gq = lane & 3, n = fn;
            float b1 = xs[gq][fr][0], b2 = xs[gq][fr][1];
            int a1 = xk[gq][fr][0], a2 = xk[gq][fr][1];
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1) {
                const float ob1 = __shfl_xor_sync(0xffffffffu, b1, o), ob2 = __shfl_xor_sync(0xffffffffu, b2, o);
                const int oa1 = __shfl_xor_sync(0xffffffffu, a1, o), oa2 = __shfl_xor_sync(0xffffffffu, a2, o);
                merge2(b1, a1, b2, a2, ob1, oa1, ob2, oa2);
            }
            int arg = a1 == 0x7fffffff ? 0 : a1;
            const int arg2 = (a2 == 0x7fffffff || !(b2 < INFINITY)) ? -1 : a2;
            const int j0 = lane * E, kb = j0 >> 6, e0 = j0 & 63, c8 = e0 >> 3, boff = (e0 & 7) * 2;
            auto ld_row = [&](const uint8_t *base, size_t kb_stride, int row, float (&v)[E]) {
                const uint8_t *pp = base + kb * kb_stride + row * 128 + ((c8 ^ (row & 7)) << 4) + boff;
                if constexpr (E == 4) {
                    const uint2 u = *reinterpret_cast<const uint2 *>(pp);
                    v[0] = __uint_as_float(u.x << 16);
                    v[1] = __uint_as_float(u.x & 0xffff0000u);
                    v[2] = __uint_as_float(u.y << 16);
                    v[3] = __uint_as_float(u.y & 0xffff0000u);
                } else {
                    const uint32_t u = *reinterpret_cast<const uint32_t *>(pp);
                    v[0] = __uint_as_float(u << 16);
                    v[1] = __uint_as_float(u & 0xffff0000u);
                }
            };
            float wl[E];
#pragma unroll
            for (int e = 0; e < E; ++e) wl[e] = w ? w[h * D + j0 + e] : 1.0f;
            const float xn = xn_pre;
            const bool flag = ok && gq == 0 && n < N && arg2 >= 0 &&
                              !(b2 - b1 > (P == 1 ? kAssignTau : 2.0f * kAssignTau) *
                                              (3.0f * xn + fmaxf(b1, 0.0f) + fmaxf(b2, 0.0f)));
            // warp-cooperative exact re-scoring of the flagged rows
            unsigned m = __ballot_sync(0xffffffffu, flag);
            while (m) {
                const int l = __ffs(m) - 1;
                m &= m - 1;
                const int rr = 8 * warp + (l >> 2);
                const int ca = __shfl_sync(0xffffffffu, arg, l), cb = __shfl_sync(0xffffffffu, arg2, l);
                float xv[E], va[E], vb[E];
                ld_row(Ab, 16384, rr, xv);
                if constexpr (P == 1) {
                    ld_row(Bs, static_cast<size_t>(Np) * 128, ca, va);
                    ld_row(Bs, static_cast<size_t>(Np) * 128, cb, vb);
                } else {
                    const uint16_t *pa = ch + static_cast<size_t>(ca) * D + j0, *pb = ch + static_cast<size_t>(cb) * D + j0;
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        va[e] = bf16_to_f32(pa[e]);
                        vb[e] = bf16_to_f32(pb[e]);
                    }
                }
                float da = 0.0f, db = 0.0f;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float fa = xv[e] - va[e], fb = xv[e] - vb[e];
                    da = fmaf(wl[e] * fa, fa, da);
                    db = fmaf(wl[e] * fb, fb, db);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    da += __shfl_xor_sync(0xffffffffu, da, o);
                    db += __shfl_xor_sync(0xffffffffu, db, o);
                }
                if (lane == l && (db < da || (db == da && cb < ca))) arg = cb;
            }
            if (ok && gq == 0 && n < N) ids[static_cast<size_t>(h) * N + n] = arg;
        }
        // (4) with two buffers, tile k+1's loads were issued in (2): start its MMA
        if (NA == 2 && tid == 0 && k + 1 < my_tiles) {
            if (umma::mbar_wait(&bar_a[(k + 1) % NA], ((k + 1) / NA) & 1, wait_ns)) {
                n_waited = k + 2;
                umma::tc_fence_after();
                issue(k + 1);
            } else {
                ok = false;
            }
        }
        umma::tc_fence_before();
        ok = __syncthreads_and(ok);
        umma::tc_fence_after();
    }
    if (!ok) {
        // a wait ran out and the assignment is incomplete: every row of this
        // CTA's tiles gets cluster 0, so that the kernels after this one read
        // valid ids (the call's results are undefined; its status is TIMEOUT)
        if (tid == 0) raise_error(err, QVG_ERR_TIMEOUT);
        for (int k = 0; k < my_tiles; ++k)
            for (int r = tid; r < 128; r += kAssignThreads) {
                const int n = (t0 + k * tstep) * 128 + r;
                if (n < N) ids[static_cast<size_t>(h) * N + n] = 0;
            }
    }
    // every MMA issued by thread 0 completes before TMEM is released (at the
    // default bound, whatever the pipeline's waits were given)
    if (tid == 0 && my_tiles > 0) {
        umma::mma_commit(&bar_drain);
        umma::mbar_wait(&bar_drain, 0, kWaitNs);
        // tile copies issued but never waited for (a wait ran out)
        for (int j = n_waited; j < n_issued; ++j)
            umma::mbar_wait(&bar_a[j % NA], static_cast<uint32_t>(j / NA) & 1u, kWaitNs);
    }
    umma::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        umma::tc_fence_after();
        umma::tmem_dealloc(tmem, 2 * ncols);
    }
}

template <typename T> struct RowLoad;
template <> struct RowLoad<uint16_t> {
    template <int E>
    __device__ static void load(const uint16_t *p, float (&v)[E]) {
        if constexpr (E == 4) {
            const uint2 u = *reinterpret_cast<const uint2 *>(p);
            v[0] = __uint_as_float(u.x << 16);
            v[1] = __uint_as_float(u.x & 0xffff0000u);
            v[2] = __uint_as_float(u.y << 16);
            v[3] = __uint_as_float(u.y & 0xffff0000u);
        } else {
            const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
            v[0] = __uint_as_float(u << 16);
            v[1] = __uint_as_float(u & 0xffff0000u);
        }
    }
};
template <> struct RowLoad<float> {
    template <int E>
    __device__ static void load(const float *p, float (&v)[E]) {
        if constexpr (E == 4) {
            const float4 u = *reinterpret_cast<const float4 *>(p);
            v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
        } else {
            const float2 u = *reinterpret_cast<const float2 *>(p);
            v[0] = u.x; v[1] = u.y;
        }
    }
};

// ---------------------------------------------------------------------------
// Update, one kernel: each CTA (S = gridDim.x per head) first orders the head's
// token indices by cluster in shared memory, stably (ascending token index
// inside each cluster).  Warp w owns a contiguous range of tokens: pass 1
// counts its tokens per cluster (warp match: the lowest lane of each group of
// equal ids adds the group size), pass 2 turns the per-warp counts of each
// cluster into offsets (earlier warps first) and scans the cluster totals,
// pass 3 walks the range again and places each token at its cluster's start
// + the offset of its warp + its rank among the earlier equal ids of the
// warp.  CTA x then finalises the contiguous cluster range
// [x Ce / S, (x + 1) Ce / S), whose members are contiguous in
// that order; the slice is cut into one equal run of positions per warp, so
// one very large cluster (the smallest-norm centroid collects the tiny
// residuals of a later stage) is summed by many warps.  Each warp sums the
// members' stage input over its run in order (fp32, eight row loads in
// flight); a cluster that lies inside the run is finalised at once, a
// cluster cut by the run's ends leaves a partial sum in shared memory, and
// the warp holding the cluster's first member adds the partials in warp
// order.  Finalising divides by the count, rounds to bf16 and writes the
// centroid and its weighted norm; an empty cluster keeps its centroid.
// Deterministic, with no atomic accumulation of values.  A diagonal weight
// leaves the minimiser at the plain mean.
constexpr int kUpdThreads = 1024;
// CTAs per head: about one per SM over all heads, 2..16
inline int update_splits(int H, int n_sm) { return std::max(2, std::min(16, n_sm / std::max(1, H))); }

template <int D, typename TIn>
__global__ void __launch_bounds__(kUpdThreads) k_kmeans_update(const TIn *__restrict__ xin, int N, int H,
                                                              const int32_t *__restrict__ ids,
                                                              uint16_t *__restrict__ cent, size_t hs, int Ce,
                                                              const float *__restrict__ w,
                                                              float *__restrict__ cnorm, int C,
                                                              float *__restrict__ means) {
    constexpr int W = kUpdThreads / 32;
    constexpr int E = D / 32;
    extern __shared__ __align__(16) uint16_t order[];          // [N] token indices, by cluster
    __shared__ int cnt[QVG_MAX_CLUSTERS + 1];                   // cluster start positions
    __shared__ int wc[W][QVG_MAX_CLUSTERS];                    // per-warp counts, then offsets
    const int h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t *hid = ids + static_cast<size_t>(h) * N;
    const int span = ceil_div(ceil_div(N, W), 32) * 32;        // tokens per warp, whole batches
    const int n_beg = warp * span, n_end = min(N, n_beg + span);
    for (int i = tid; i < W * QVG_MAX_CLUSTERS; i += kUpdThreads) (&wc[0][0])[i] = 0;
    pdl_wait();  // the assignment that wrote ids has finished
    pdl_trigger();
    __syncthreads();
    // pass 1: per-warp counts (an id outside [0, Ce) -- which the assignment
    // never writes -- counts as no member, so no access leaves the tables)
    for (int b0 = n_beg; b0 < n_end; b0 += 32) {
        const int n = b0 + lane;
        int c = n < n_end ? hid[n] : -1;
        c = static_cast<unsigned>(c) < static_cast<unsigned>(Ce) ? c : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, c);
        if (c >= 0 && (peers & ((1u << lane) - 1u)) == 0) wc[warp][c] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // pass 2: per-cluster offsets of the warps, then the exclusive scan of the totals
    if (tid < Ce) {
        int run = 0;
        for (int w2 = 0; w2 < W; ++w2) {
            const int t = wc[w2][tid];
            wc[w2][tid] = run;
            run += t;
        }
        cnt[tid] = run;
    }
    __syncthreads();
    if (warp == 0) {
        int v[8], tot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = lane * 8 + i;
            v[i] = c < Ce ? cnt[c] : 0;
            tot += v[i];
        }
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int acc = incl - tot;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = lane * 8 + i;
            if (c < Ce) cnt[c] = acc;  // each cluster's first position
            acc += v[i];
        }
        if (lane == 31) cnt[Ce] = incl;
    }
    __syncthreads();
    // pass 3: placement in token order
    for (int b0 = n_beg; b0 < n_end; b0 += 32) {
        const int n = b0 + lane;
        int c = n < n_end ? hid[n] : -1;
        c = static_cast<unsigned>(c) < static_cast<unsigned>(Ce) ? c : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, c);
        const unsigned before = peers & ((1u << lane) - 1u);
        if (c >= 0) order[cnt[c] + wc[warp][c] + __popc(before)] = static_cast<uint16_t>(n);
        __syncwarp();
        if (c >= 0 && before == 0) wc[warp][c] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // this CTA's clusters and its warps' runs of the sorted order; wc is free
    // again and holds the partial sums, two rows per warp ([0]: the run's
    // first cluster, begun before the run; [1]: its last, going on after it)
    float (*part)[2][D] = reinterpret_cast<float (*)[2][D]>(&wc[0][0]);
    static_assert(sizeof(float) * W * 2 * D <= sizeof(int) * W * QVG_MAX_CLUSTERS, "partials fit in wc");
    const int c_lo = static_cast<int>(static_cast<long long>(Ce) * blockIdx.x / gridDim.x);
    const int c_hi = static_cast<int>(static_cast<long long>(Ce) * (blockIdx.x + 1) / gridDim.x);
    const int p_lo = cnt[c_lo], M = cnt[c_hi] - p_lo;
    auto run_beg = [&](int w2) { return p_lo + static_cast<int>(static_cast<long long>(M) * w2 / W); };
    const int a = run_beg(warp), b = run_beg(warp + 1);
    auto finalise = [&](int c, const float (&acc)[E]) {
        const float cntf = static_cast<float>(cnt[c + 1] - cnt[c]);
        uint16_t *row = cent + static_cast<size_t>(h) * hs + static_cast<size_t>(c) * D + lane * E;
        float nrm = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float mean = __fdiv_rn(acc[e], cntf);
            if (means) means[(static_cast<size_t>(h) * C + c) * D + lane * E + e] = mean;
            const uint16_t cb = f32_to_bf16(mean);
            row[e] = cb;
            const float cv = bf16_to_f32(cb);
            const float wj = w ? w[h * D + lane * E + e] : 1.0f;
            nrm = fmaf(wj * cv, cv, nrm);
        }
        for (int o = 16; o > 0; o >>= 1) nrm += __shfl_xor_sync(0xffffffffu, nrm, o);
        if (lane == 0) cnorm[h * C + c] = nrm;
    };
    if (means) {  // an empty cluster keeps its centroid: that is its fp32 value too
        for (int i = tid; i < (c_hi - c_lo) * D; i += kUpdThreads) {
            const int c = c_lo + i / D, j = i % D;
            if (cnt[c + 1] == cnt[c])
                means[(static_cast<size_t>(h) * C + c) * D + j] =
                    bf16_to_f32(cent[static_cast<size_t>(h) * hs + static_cast<size_t>(c) * D + j]);
        }
    }
    int split_c = -1;  // a cluster that starts in this run and goes on after it
    if (a < b) {
        int c = c_lo;
        while (cnt[c + 1] <= a) ++c;
        for (int pos = a; pos < b; ++c) {
            if (cnt[c + 1] <= pos) continue;  // empty cluster
            const int end = min(b, cnt[c + 1]);
            float acc[E];
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = 0.0f;
            for (int i0 = pos; i0 < end; i0 += 8) {
                int nn[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) nn[q] = i0 + q < end ? static_cast<int>(order[i0 + q]) : -1;
                float v[8][E];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (nn[q] >= 0)
                        RowLoad<TIn>::template load<E>(xin + (static_cast<size_t>(nn[q]) * H + h) * D + lane * E, v[q]);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (nn[q] >= 0)
#pragma unroll
                        for (int e = 0; e < E; ++e) acc[e] += v[q][e];
            }
            const bool head = cnt[c] >= a, tail = cnt[c + 1] <= b;
            if (head && tail) {
                finalise(c, acc);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) part[warp][head ? 1 : 0][lane * E + e] = acc[e];
                if (head) split_c = c;
            }
            pos = end;
        }
    }
    __syncthreads();
    if (split_c >= 0) {  // add the later runs' partials of split_c, in warp order
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = part[warp][1][lane * E + e];
        for (int w2 = warp + 1; w2 < W; ++w2) {
            const int a2 = run_beg(w2), b2 = run_beg(w2 + 1);
            if (a2 >= cnt[split_c + 1]) break;
            if (a2 < b2)
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] += part[w2][0][lane * E + e];
        }
        finalise(split_c, acc);
    }
}

// ---------------------------------------------------------------------------
// Residual quantisation of one stage, thread = (token, head) row x 32-channel
// block: D / 32 adjacent lanes (TPR) share a row, so each load or store
// instruction of a warp covers 8 (d = 128) or 16 (d = 64) whole rows, and a
// block of 256 threads takes consecutive tokens of one head; the grid runs
// over the heads first, so the blocks in flight cover every head of a token
// range and read the token-major input in whole DRAM pages.  Pass 1 forms
// r = x - c (kept in registers) and each 8-channel block's amax; a group's
// amax is combined over its blocks in channel order and, for a group wider
// than 32 channels, over the row's lanes by xor shuffles (every lane of the
// group gets the same result), and its scale is computed once.  Pass 2
// quantises and packs; only when the next stage or PSAC needs the
// reconstruction error does a third pass re-read the block (from L1).
// Writes codes, fp16 scales and the cluster id; optionally the
// next stage's input X_{l+1} = X_l - deq (fp32 and its bf16 rounding, the
// next clustering operand); optionally (last stage of a key chunk with
// PSAC) the INT8 projection of X_{L+1} on the basis U, an fp32 FMA chain in
// ascending channel order -- run block after block by the row's lanes in
// turn, each continuing the chain of the one before (handed on by shuffle).
// OUTL (outlier split): pass 1 also keeps, per group, the second-largest
// |r| and the signed value and channel of the largest.  The largest is an
// outlier exactly when it is strictly above the second: for G <= 100 the
// group's linear-interpolation 99th percentile lies strictly between the
// two.  The scale then comes from the second-largest (the largest of the
// values that remain; equal to the largest when nothing is split off), the
// outlier's code is 0 and its stage value is fp16(r) + c.
template <typename TIn>
__device__ __forceinline__ void load32(const TIn *p, float (&v)[32]);
template <>
__device__ __forceinline__ void load32<uint16_t>(const uint16_t *p, float (&v)[32]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p + 8 * i);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[8 * i + 2 * k] = __uint_as_float(w4[k] << 16);
            v[8 * i + 2 * k + 1] = __uint_as_float(w4[k] & 0xffff0000u);
        }
    }
}
template <>
__device__ __forceinline__ void load32<float>(const float *p, float (&v)[32]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 u = *reinterpret_cast<const float4 *>(p + 4 * i);
        v[4 * i] = u.x;
        v[4 * i + 1] = u.y;
        v[4 * i + 2] = u.z;
        v[4 * i + 3] = u.w;
    }
}

// Group statistics of a run of channels: amax m, second-largest m2, and the
// signed value rv and row channel ix of the first largest.
struct GStat {
    float m, m2, rv;
    int ix;
};
// a's channels come before b's: the combined statistics are those of a
// sequential pass over a then b
__device__ __forceinline__ GStat gmerge(const GStat &a, const GStat &b) {
    if (b.m > a.m) return GStat{b.m, fmaxf(a.m, b.m2), b.rv, b.ix};
    return GStat{a.m, fmaxf(a.m2, b.m), a.rv, a.ix};
}

// DELTA: the call writes the next stage's input or the PSAC projection
// (delta_out or psacU set); without it the kernel ends after the codes.
template <int D, int BITS, typename TIn, bool OUTL, bool DELTA>
__global__ void __launch_bounds__(256, DELTA ? 2 : 3) k_residual_quant(
    const TIn *__restrict__ xin, int N, int H, const uint16_t *__restrict__ cent, size_t hs, int C,
    const int32_t *__restrict__ ids, int group, int mode, uint8_t *__restrict__ codes,
    uint16_t *__restrict__ scales, uint8_t *__restrict__ ids_out, size_t shs,
    float *__restrict__ delta_out, uint16_t *__restrict__ gbf_out, const float *__restrict__ psacU,
    int8_t *__restrict__ psac_p, uint16_t *__restrict__ psac_s, size_t phs, uint16_t *__restrict__ outl_val,
    uint8_t *__restrict__ outl_idx) {
    constexpr int NB = D * BITS / 8, CB = 32 * BITS / 8;  // code bytes per row / per 32-channel block
    constexpr int TPR = D / 32, RPB = 256 / TPR;           // lanes per row, rows per block
    pdl_wait();  // the final assignment (which reads this stage's operand) has finished
    pdl_trigger();
    const int lane = threadIdx.x & 31, cb = lane % TPR, h = blockIdx.x;
    const int n_row = blockIdx.y * RPB + threadIdx.x / TPR;
    // every lane takes part in the shuffles below; a row past N repeats row
    // N - 1 and stores nothing
    const bool live = n_row < N;
    const int n = live ? n_row : N - 1;
    const int glog = __ffs(group) - 1;  // groups are powers of two: shifts, not divisions
    const int ng = D >> glog;
    // (an id outside [0, C) never comes from the assignment; clamped so that
    // no access leaves the centroid table)
    const unsigned uid = C > 0 ? static_cast<unsigned>(ids[static_cast<size_t>(h) * N + n]) : 0u;
    const int id = uid < static_cast<unsigned>(C) ? static_cast<int>(uid) : max(C - 1, 0);
    const size_t trow = static_cast<size_t>(n) * H + h;  // token-major row of the stage buffers
    const TIn *xr = xin + trow * D + cb * 32;
    const uint16_t *cr = C > 0 ? cent + static_cast<size_t>(h) * hs + static_cast<size_t>(id) * D + cb * 32 : nullptr;
    // pass 1: r = x - c for the lane's 32 channels (kept for pass 2) and the
    // statistics of each 8-channel block
    float r[32];
    {
        float x[32], c[32];
        load32<TIn>(xr, x);
        if (C > 0) load32<uint16_t>(cr, c);
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = C > 0 ? __fsub_rn(x[e], c[e]) : x[e];
    }
    GStat st8[4];
#pragma unroll
    for (int b8 = 0; b8 < 4; ++b8) {
        float m = 0.0f, m2 = 0.0f, rv = 0.0f;
        int ix = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float a = fabsf(r[8 * b8 + e]);
            if constexpr (OUTL) {
                if (a > m) {
                    m2 = m;
                    m = a;
                    rv = r[8 * b8 + e];
                    ix = e;
                } else {
                    m2 = fmaxf(m2, a);
                }
            } else {
                m = fmaxf(m, a);
            }
        }
        st8[b8] = GStat{m, m2, rv, cb * 32 + 8 * b8 + ix};
    }
    // each 8-channel block's group statistics: groups of 8, 16 or 32
    // channels lie inside the lane's block; wider ones span 2 or 4 lanes
    GStat gs8[4];
    const GStat zero{0.0f, 0.0f, 0.0f, 0};
    if (group <= 32) {
        const int g8log = glog - 3;  // 1, 2 or 4 blocks per group (log2: 0, 1, 2)
#pragma unroll
        for (int b8 = 0; b8 < 4; ++b8) {
            GStat acc = zero;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if ((k >> g8log) == (b8 >> g8log)) acc = OUTL ? gmerge(acc, st8[k]) : GStat{fmaxf(acc.m, st8[k].m), 0.0f, 0.0f, 0};
            gs8[b8] = acc;
        }
    } else {
        GStat acc = zero;
#pragma unroll
        for (int k = 0; k < 4; ++k) acc = OUTL ? gmerge(acc, st8[k]) : GStat{fmaxf(acc.m, st8[k].m), 0.0f, 0.0f, 0};
        // lanes cb ^ o (o < group / 32) of the row hold the group's other blocks
        for (int o = 1; o < (group >> 5); o <<= 1) {
            GStat pt;
            pt.m = __shfl_xor_sync(0xffffffffu, acc.m, o);
            if constexpr (OUTL) {
                pt.m2 = __shfl_xor_sync(0xffffffffu, acc.m2, o);
                pt.rv = __shfl_xor_sync(0xffffffffu, acc.rv, o);
                pt.ix = __shfl_xor_sync(0xffffffffu, acc.ix, o);
                acc = (cb & o) ? gmerge(pt, acc) : gmerge(acc, pt);  // the lower channels first
            } else {
                acc.m = fmaxf(acc.m, pt.m);
            }
        }
#pragma unroll
        for (int b8 = 0; b8 < 4; ++b8) gs8[b8] = acc;
    }
    // scales (and the outlier entries) of each block's group, computed once
    // per group; the lane with the group's first block writes them
    const size_t srow = static_cast<size_t>(h) * shs + n;
    float Sb[4], ib[4], ob[4];
    int ocb[4];
    uint16_t sbits[4], obits[4];
    auto group_scale = [&](int b8) {
        const GStat &g = gs8[b8];
        sbits[b8] = group_scale_f16(OUTL ? g.m2 : g.m, BITS, mode);
        Sb[b8] = f16_to_f32(sbits[b8]);
        ib[b8] = Sb[b8] > 0.0f ? __fdiv_rn(1.0f, Sb[b8]) : 0.0f;
        ocb[b8] = -1;
        ob[b8] = 0.0f;
        obits[b8] = 0;
        if constexpr (OUTL) {
            if (g.m > g.m2) {
                ocb[b8] = g.ix;
                obits[b8] = f32_to_f16(fminf(fmaxf(g.rv, -65504.0f), 65504.0f));
                ob[b8] = f16_to_f32(obits[b8]);
            }
        }
    };
    if (group >= 32) {
        group_scale(0);
#pragma unroll
        for (int b8 = 1; b8 < 4; ++b8) {
            Sb[b8] = Sb[0];
            ib[b8] = ib[0];
            ob[b8] = ob[0];
            ocb[b8] = ocb[0];
            sbits[b8] = sbits[0];
            obits[b8] = obits[0];
        }
    } else {
#pragma unroll
        for (int b8 = 0; b8 < 4; ++b8) group_scale(b8);
    }
#pragma unroll
    for (int b8 = 0; b8 < 4; ++b8) {
        const int ch = cb * 32 + 8 * b8, gi = ch >> glog;
        if (live && (ch & (group - 1)) == 0) {
            scales[srow * ng + gi] = sbits[b8];
            if constexpr (OUTL) {
                outl_val[srow * ng + gi] = obits[b8];
                outl_idx[srow * ng + gi] = static_cast<uint8_t>(ocb[b8] < 0 ? 0xFF : ocb[b8] - gi * group);
            }
        }
    }
    if (ids_out && live && cb == 0) ids_out[srow] = static_cast<uint8_t>(id);  // no ids without centroids (C = 0)
    // pass 2: the codes, clamp(rint(r / S)) as quant_code_rcp (common.cuh)
    // gives them -- rint(r fl(1 / S)), with the division redone, after the
    // loop, for the rare element whose product lies within |y| 2^-21 of a
    // half-integer; an outlier's code is 0
    constexpr float kQmax = static_cast<float>((1 << (BITS - 1)) - 1);
    uint32_t pw[CB / 4];
#pragma unroll
    for (int k = 0; k < CB / 4; ++k) pw[k] = 0u;
    uint32_t near = 0u;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const int b8 = e >> 3;
        int q = 0;
        if (!(OUTL && cb * 32 + e == ocb[b8]) && Sb[b8] > 0.0f) {
            const float y = __fmul_rn(r[e], ib[b8]);
            const float t = rintf(y);
            if (0.5f - fabsf(y - t) <= fabsf(y) * 0x1p-21f) near |= 1u << e;
            q = static_cast<int>(fminf(fmaxf(t, -kQmax - 1.0f), kQmax));
        }
        pw[(e * BITS) / 32] |= static_cast<uint32_t>(q + (1 << (BITS - 1))) << ((e * BITS) % 32);
    }
    if (near) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
            if ((near >> e) & 1u) {
                const float t = rintf(__fdiv_rn(r[e], Sb[e >> 3]));
                const int q = static_cast<int>(fminf(fmaxf(t, -kQmax - 1.0f), kQmax));
                const int wi = (e * BITS) / 32, sh = (e * BITS) % 32;
                pw[wi] = (pw[wi] & ~(((1u << BITS) - 1u) << sh)) | (static_cast<uint32_t>(q + (1 << (BITS - 1))) << sh);
            }
    }
    if (live) {
        uint8_t *cdst = codes + srow * NB + cb * CB;
        if constexpr (CB == 8)
            *reinterpret_cast<uint2 *>(cdst) = make_uint2(pw[0], pw[1]);
        else
            *reinterpret_cast<uint4 *>(cdst) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
    }
    // the stage's reconstruction error X - (S q + c) (or the outlier's fp16
    // value + c): the next stage's input and the PSAC operand
    if constexpr (!DELTA) return;
    float dl[32];
    {
        float x[32], c[32];
        load32<TIn>(xr, x);
        if (C > 0) load32<uint16_t>(cr, c);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int q = static_cast<int>((pw[(e * BITS) / 32] >> ((e * BITS) % 32)) & ((1u << BITS) - 1u)) -
                          (1 << (BITS - 1));
            const bool is_out = OUTL && cb * 32 + e == ocb[e >> 3];
            const float rh = is_out ? ob[e >> 3] : __fmul_rn(Sb[e >> 3], static_cast<float>(q));
            const float deq = C > 0 ? __fadd_rn(rh, c[e]) : rh;
            dl[e] = __fsub_rn(x[e], deq);
        }
    }
    if (live && delta_out) {
        float4 *dp = reinterpret_cast<float4 *>(delta_out + trow * D + cb * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) dp[i] = make_float4(dl[4 * i], dl[4 * i + 1], dl[4 * i + 2], dl[4 * i + 3]);
        if (gbf_out) {
            uint4 *gp = reinterpret_cast<uint4 *>(gbf_out + trow * D + cb * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t w4[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    w4[k] = static_cast<uint32_t>(f32_to_bf16(dl[8 * i + 2 * k])) |
                            (static_cast<uint32_t>(f32_to_bf16(dl[8 * i + 2 * k + 1])) << 16);
                gp[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
        }
    }
    if (psacU) {
        // the projection chain over the row's channels in ascending order:
        // lane block j continues the chain of blocks 0 .. j - 1
        const float *Uh = psacU + static_cast<size_t>(h) * D * QVG_PSAC_RANK;
        const int row_lane0 = lane - cb;
        float P[QVG_PSAC_RANK];
#pragma unroll
        for (int k = 0; k < QVG_PSAC_RANK; ++k) P[k] = 0.0f;
#pragma unroll 1
        for (int j = 0; j < TPR; ++j) {
            if (cb == j) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float4 u0 = *reinterpret_cast<const float4 *>(Uh + (cb * 32 + e) * QVG_PSAC_RANK);
                    const float4 u1 = *reinterpret_cast<const float4 *>(Uh + (cb * 32 + e) * QVG_PSAC_RANK + 4);
                    const float de = dl[e];
                    P[0] = fmaf(de, u0.x, P[0]);
                    P[1] = fmaf(de, u0.y, P[1]);
                    P[2] = fmaf(de, u0.z, P[2]);
                    P[3] = fmaf(de, u0.w, P[3]);
                    P[4] = fmaf(de, u1.x, P[4]);
                    P[5] = fmaf(de, u1.y, P[5]);
                    P[6] = fmaf(de, u1.z, P[6]);
                    P[7] = fmaf(de, u1.w, P[7]);
                }
            }
#pragma unroll
            for (int k = 0; k < QVG_PSAC_RANK; ++k) P[k] = __shfl_sync(0xffffffffu, P[k], row_lane0 + j);
        }
        if (live && cb == 0) {
            float pa = 0.0f;
#pragma unroll
            for (int k = 0; k < QVG_PSAC_RANK; ++k) pa = fmaxf(pa, fabsf(P[k]));
            const uint16_t psb = f32_to_f16(fminf(__fdiv_rn(pa, 127.0f), 65504.0f));
            const float pSp = f16_to_f32(psb);
            uint32_t pq[2] = {0u, 0u};
#pragma unroll
            for (int k = 0; k < QVG_PSAC_RANK; ++k) {
                int qp = 0;
                if (pSp > 0.0f) {
                    float t = rintf(__fdiv_rn(P[k], pSp));
                    t = fminf(fmaxf(t, -127.0f), 127.0f);
                    qp = static_cast<int>(t);
                }
                pq[k >> 2] |= (static_cast<uint32_t>(qp) & 0xffu) << (8 * (k & 3));
            }
            *reinterpret_cast<uint2 *>(psac_p + (static_cast<size_t>(h) * phs + n) * QVG_PSAC_RANK) =
                make_uint2(pq[0], pq[1]);
            psac_s[static_cast<size_t>(h) * phs + n] = psb;
        }
    }
}

__global__ void k_chunk_table(int chunk, int slot0, int N, int32_t *chunk_start, int32_t *chunk_len,
                              int32_t *tile_chunk, int32_t *chunk_anchor, int anchor_row) {
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) {
        chunk_start[chunk] = slot0;
        chunk_len[chunk] = N;
        if (chunk_anchor) chunk_anchor[chunk] = anchor_row;
    }
    const int t0 = slot0 / QVG_TILE, nt = ceil_div(N, QVG_TILE);
    for (int t = threadIdx.x; t < nt; t += blockDim.x) tile_chunk[t0 + t] = chunk;
}

// ---------------------------------------------------------------------------
// Launchers.

static int sm_count() { return sm_count_current(); }

// cuTensorMapEncodeTiled from the driver (looked up once; no link to libcuda).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

// 3-D bf16 tensor map (dims d0 innermost .. d2, byte strides of dims 1 and 2),
// boxes of box0 x box1 x box2 elements with the 128-byte swizzle, zero fill
// outside the tensor.  A host-side description only: nothing is allocated.
static bool bf16_tensor_map(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                            uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1, uint32_t box2) {
    const auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1, stride2};
    const cuuint32_t box[3] = {box0, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

qvg_status launch_kmeans_init(const uint16_t *g, int N, int H, int d, int C, int Ce, uint64_t seed,
                              int chunk, int stage, uint16_t *cent, size_t hs, const float *w, float *cnorm,
                              cudaStream_t st) {
    dim3 grid(ceil_div(C, 8), H);
    const cudaError_t e = d == 64 ? launch_pdl(k_kmeans_init<64>, grid, dim3(256), 0, st, g, N, H, C, Ce, seed,
                                               chunk, stage, cent, hs, w, cnorm)
                                  : launch_pdl(k_kmeans_init<128>, grid, dim3(256), 0, st, g, N, H, C, Ce, seed,
                                               chunk, stage, cent, hs, w, cnorm);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        note_cuda_error(e);
        return QVG_ERR_CUDA;
    }
    return QVG_OK;
}

qvg_status launch_centroid_norms(const uint16_t *cent, size_t hs, int H, int C, int d,
                                 const float *w, float *cnorm, cudaStream_t st) {
    const int warps = H * C, blocks = ceil_div(warps * 32, 256);
    if (d == 64)
        k_centroid_norms<64><<<blocks, 256, 0, st>>>(cent, hs, H, C, w, cnorm);
    else
        k_centroid_norms<128><<<blocks, 256, 0, st>>>(cent, hs, H, C, w, cnorm);
    QVG_LAUNCH_CHECK();
    return QVG_OK;
}

template <int D, int P>
static qvg_status assign_tc_impl(const uint16_t *g, int N, int H, const uint16_t *cent, size_t hs, int Ce,
                                 const float *cnorm, int C, const float *w, const float *xnorm, int32_t *ids,
                                 cudaStream_t st) {
    const int Np = std::max(16, ceil_div(Ce, 16) * 16);
    constexpr int KB = D / 64, NA = P == 1 ? 3 : 2;
    const size_t smem = NA * (static_cast<size_t>(KB) * 128 * 128 + 4096) + static_cast<size_t>(P) * KB * Np * 128 +
                        static_cast<size_t>(Np) * 32 + 1024;
    {
        // the largest request of this instantiation (Np = 256), once per device
        static std::atomic<uint64_t> done{0};
        const size_t most = NA * (static_cast<size_t>(KB) * 128 * 128 + 4096) +
                            static_cast<size_t>(P) * KB * QVG_MAX_CLUSTERS * 128 + QVG_MAX_CLUSTERS * 32 + 1024;
        const qvg_status s = smem_limit_once(done, reinterpret_cast<const void *>(k_kmeans_assign_tc<D, P>),
                                             static_cast<int>(most));
        if (s != QVG_OK) return s;
    }
    // one CTA per SM in total, spread over the heads; each walks
    // ceil(tiles / ctas_per_head) token tiles of its head
    const int n_tiles = ceil_div(N, 128);
    const int per_head = std::max(1, std::min(n_tiles, sm_count() / std::max(1, H)));
    dim3 grid(per_head, H);
    // the stage operand [N][H][D] in boxes of (64 channels, 1 head, 128 tokens);
    // this chunk's centroids [H][C][D] (head stride hs) in boxes of (64, Np, 1)
    CUtensorMap tm_x, tm_c;
    if (!bf16_tensor_map(&tm_x, g, D, H, N, D * 2ull, static_cast<uint64_t>(H) * D * 2, 64, 1, 128) ||
        (P == 1 && !bf16_tensor_map(&tm_c, cent, D, C, H, D * 2ull, hs * 2, 64, Np, 1)))
        return QVG_ERR_CUDA;
    if (P != 1) tm_c = tm_x;  // (unused: the weighted centroids are staged by the threads)
    const cudaError_t e = launch_pdl(k_kmeans_assign_tc<D, P>, grid, dim3(kAssignThreads), smem, st, tm_x, tm_c, g,
                                     N, H, cent, hs, Ce, Np, cnorm, C, w, xnorm, ids, device_error_word(),
                                     wait_limit_ns(), wait_inject());
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        note_cuda_error(e);
        return QVG_ERR_CUDA;
    }
    return QVG_OK;
}

qvg_status launch_kmeans_assign(const uint16_t *g, int N, int H, int d, const uint16_t *cent,
                                size_t hs, int Ce, const float *cnorm, int C, const float *w,
                                const float *xnorm, int32_t *ids, cudaStream_t st) {
    if (d == 64)
        return w ? assign_tc_impl<64, 2>(g, N, H, cent, hs, Ce, cnorm, C, w, xnorm, ids, st)
                 : assign_tc_impl<64, 1>(g, N, H, cent, hs, Ce, cnorm, C, w, xnorm, ids, st);
    return w ? assign_tc_impl<128, 2>(g, N, H, cent, hs, Ce, cnorm, C, w, xnorm, ids, st)
             : assign_tc_impl<128, 1>(g, N, H, cent, hs, Ce, cnorm, C, w, xnorm, ids, st);
}

// ||x||_w^2 per (token, head) row of the clustering operand: a warp takes
// kNormRows consecutive rows with all their loads in flight, each row D/32
// consecutive channels per lane (fp32, ascending) and an xor-butterfly sum.
constexpr int kNormRows = 4;

template <int D>
__global__ void __launch_bounds__(256) k_row_norms(const uint16_t *__restrict__ g, int N, int H,
                                                   const float *__restrict__ w, float *__restrict__ xnorm) {
    constexpr int E = D / 32;
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const long long row0 = (static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * kNormRows;
    const long long rows = static_cast<long long>(N) * H;
    if (row0 >= rows) return;
    float v[kNormRows][E];
#pragma unroll
    for (int i = 0; i < kNormRows; ++i)
        if (row0 + i < rows) RowLoad<uint16_t>::template load<E>(g + static_cast<size_t>(row0 + i) * D + lane * E, v[i]);
#pragma unroll
    for (int i = 0; i < kNormRows; ++i) {
        if (row0 + i >= rows) break;
        const int n = static_cast<int>((row0 + i) / H), h = static_cast<int>((row0 + i) % H);
        float sx = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float wj = w ? w[h * D + lane * E + e] : 1.0f;
            sx = fmaf(wj * v[i][e], v[i][e], sx);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sx += __shfl_xor_sync(0xffffffffu, sx, o);
        if (lane == 0) xnorm[static_cast<size_t>(h) * N + n] = sx;
    }
}

qvg_status launch_row_norms(const uint16_t *g, int N, int H, int d, const float *w, float *xnorm,
                            cudaStream_t st) {
    const long long rows = static_cast<long long>(N) * H;
    const unsigned blocks = static_cast<unsigned>((rows + 8 * kNormRows - 1) / (8 * kNormRows));
    const cudaError_t e = d == 64 ? launch_pdl(k_row_norms<64>, dim3(blocks), dim3(256), 0, st, g, N, H, w, xnorm)
                                  : launch_pdl(k_row_norms<128>, dim3(blocks), dim3(256), 0, st, g, N, H, w, xnorm);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        note_cuda_error(e);
        return QVG_ERR_CUDA;
    }
    return QVG_OK;
}

qvg_status launch_kmeans_update(const void *xin, bool xin_f32, int N, int H, int d,
                                const int32_t *ids, uint16_t *cent, size_t hs, int Ce, int C, const float *w,
                                float *cnorm, float *means, cudaStream_t st) {
    const size_t smem = static_cast<size_t>(N) * sizeof(uint16_t);
    dim3 grid(update_splits(H, sm_count()), H);
#define QVG_UPD(D_, T_)                                                                                     \
    do {                                                                                                    \
        static std::atomic<uint64_t> done{0};                                                               \
        const qvg_status as = smem_limit_once(done, reinterpret_cast<const void *>(k_kmeans_update<D_, T_>), \
                                              131072);                                                      \
        if (as != QVG_OK) return as;                                                                        \
        const cudaError_t le = launch_pdl(k_kmeans_update<D_, T_>, grid, dim3(kUpdThreads), smem, st,        \
                                          static_cast<const T_ *>(xin), N, H, ids, cent, hs, Ce, w, cnorm, C, \
                                          means);                                                           \
        if (le != cudaSuccess) {                                                                            \
            (void)cudaGetLastError();                                                                       \
            note_cuda_error(le);                                                                            \
            return QVG_ERR_CUDA;                                                                            \
        }                                                                                                   \
    } while (0)
    if (d == 64) {
        if (xin_f32) QVG_UPD(64, float); else QVG_UPD(64, uint16_t);
    } else {
        if (xin_f32) QVG_UPD(128, float); else QVG_UPD(128, uint16_t);
    }
#undef QVG_UPD
    QVG_LAUNCH_CHECK();
    return QVG_OK;
}

template <int D, int BITS, bool OUTL>
static cudaError_t rq_launch(const void *xin, bool f32, int N, int H, const uint16_t *cent, size_t hs,
                             int C, const int32_t *ids, int group, int mode, uint8_t *codes,
                             uint16_t *scales, uint8_t *ids_out, size_t shs, float *delta_out,
                             uint16_t *gbf_out, const float *U, int8_t *pp, uint16_t *ps, size_t phs,
                             uint16_t *ov, uint8_t *oi, cudaStream_t st) {
    // block (x, y): head x, tokens [y RPB, (y + 1) RPB), RPB = 256 / (D / 32)
    // -- the heads vary fastest, so the blocks in flight read whole token rows
    // [h = 0 .. H) of the token-major input (N <= 65535: y fits the grid)
    const dim3 grid(H, static_cast<unsigned>(ceil_div(std::max(N, 1), 256 / (D / 32))));
#define QVG_RQ(T_, DL_)                                                                                   \
    launch_pdl(k_residual_quant<D, BITS, T_, OUTL, DL_>, grid, dim3(256), 0, st, static_cast<const T_ *>(xin), N, \
               H, cent, hs, C, ids, group, mode, codes, scales, ids_out, shs, delta_out, gbf_out, U, pp, ps, phs, \
               ov, oi)
    const bool delta = delta_out != nullptr || U != nullptr;
    cudaError_t e;
    if (f32)
        e = delta ? QVG_RQ(float, true) : QVG_RQ(float, false);
    else
        e = delta ? QVG_RQ(uint16_t, true) : QVG_RQ(uint16_t, false);
#undef QVG_RQ
    return e;
}

template <int D, int BITS>
static void rq_dispatch(const void *xin, bool f32, int N, int H, const uint16_t *cent, size_t hs,
                        int C, const int32_t *ids, int group, int mode, uint8_t *codes,
                        uint16_t *scales, uint8_t *ids_out, size_t shs, float *delta_out,
                        uint16_t *gbf_out, const float *U, int8_t *pp, uint16_t *ps, size_t phs,
                        uint16_t *ov, uint8_t *oi, cudaStream_t st) {
    const cudaError_t e =
        ov ? rq_launch<D, BITS, true>(xin, f32, N, H, cent, hs, C, ids, group, mode, codes, scales, ids_out, shs,
                                      delta_out, gbf_out, U, pp, ps, phs, ov, oi, st)
           : rq_launch<D, BITS, false>(xin, f32, N, H, cent, hs, C, ids, group, mode, codes, scales, ids_out, shs,
                                       delta_out, gbf_out, U, pp, ps, phs, ov, oi, st);
    if (e != cudaSuccess) note_cuda_error(e);
}

qvg_status launch_residual_quant(const void *xin, bool xin_f32, int N, int H, int d,
                                 const uint16_t *cent, size_t hs, int C, const int32_t *ids,
                                 int bits, int group, int mode, uint8_t *codes, uint16_t *scales,
                                 uint8_t *ids_out, size_t shs, float *delta_out,
                                 uint16_t *gbf_out, const float *U, int8_t *pp, uint16_t *ps,
                                 size_t phs, uint16_t *ov, uint8_t *oi, cudaStream_t st) {
    if (d == 64 && bits == 2)
        rq_dispatch<64, 2>(xin, xin_f32, N, H, cent, hs, C, ids, group, mode, codes, scales, ids_out, shs, delta_out, gbf_out, U, pp, ps, phs, ov, oi, st);
    else if (d == 64)
        rq_dispatch<64, 4>(xin, xin_f32, N, H, cent, hs, C, ids, group, mode, codes, scales, ids_out, shs, delta_out, gbf_out, U, pp, ps, phs, ov, oi, st);
    else if (bits == 2)
        rq_dispatch<128, 2>(xin, xin_f32, N, H, cent, hs, C, ids, group, mode, codes, scales, ids_out, shs, delta_out, gbf_out, U, pp, ps, phs, ov, oi, st);
    else
        rq_dispatch<128, 4>(xin, xin_f32, N, H, cent, hs, C, ids, group, mode, codes, scales, ids_out, shs, delta_out, gbf_out, U, pp, ps, phs, ov, oi, st);
    QVG_LAUNCH_CHECK();
    return QVG_OK;
}

qvg_status launch_chunk_table(int chunk, int slot0, int N, int32_t *chunk_start, int32_t *chunk_len,
                              int32_t *tile_chunk, int32_t *chunk_anchor, int anchor_row, cudaStream_t st) {
    const cudaError_t e = launch_pdl(k_chunk_table, dim3(1), dim3(256), 0, st, chunk, slot0, N, chunk_start,
                                     chunk_len, tile_chunk, chunk_anchor, anchor_row);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        note_cuda_error(e);
        return QVG_ERR_CUDA;
    }
    return QVG_OK;
}

}  // namespace qvg
