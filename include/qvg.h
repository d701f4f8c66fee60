/*
 * qvg.h -- C ABI of libqvg: 2-bit / 4-bit compression of an autoregressive
 * video model's KV cache (Quant VideoGen, "QVG" / "QVG-Pro") with the QuantWM
 * extensions (QSAC, PSAC), and attention that reads the compressed cache
 * directly.  One GPU (NVIDIA GB300, sm_103a).
 *
 * Sources cited below by page title and section:
 *   [QVG]  Quant VideoGen: Auto-Regressive Long Video Generation via 2-Bit
 *          KV-Cache Quantization (papernotes.org notes, ICML 2026).
 *   [P1]   The 2-bit quantisation trap in video generation (cloud.baidu.com).
 *   [QWM]  QuantWM write-up (loncent.com): QSAC and PSAC.
 *   [P2]   Temporally stable 2-bit KV-cache compression for video world models, in practice (hmyw.cn): section 3.3 (temporal anchors), section 3.4
 *          (outlier separation).
 *
 * Conventions for every call:
 *   - Buffers are device pointers owned by the caller unless stated; the
 *     library never allocates device memory and never frees caller memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Only qvg_get_status synchronises.
 *   - Every call returns a qvg_status.  Argument errors are found on the
 *     host before anything is launched and leave all buffers untouched.
 *     A failed launch returns QVG_ERR_CUDA.  Errors found on the device
 *     (an exceeded wait bound) are latched in a per-device status word and
 *     reported by qvg_get_status(stream).
 *   - bf16 / fp16 values travel as their 16-bit patterns (uint16_t).
 *   - Layouts are row-major; "[a][b][c]" lists dimensions outermost first.
 *   - Thread safety: calls on different streams, from any host threads, may
 *     run concurrently as long as they do not write the same buffers.  Each
 *     call works on the device current on its host thread.  Library state:
 *     the per-device error word, the no-alloc scratch
 *     (qvg_compress_chunk_noalloc), and per-device launch set-up tables
 *     (each kernel's shared-memory limit, the SM count, the error word's
 *     address), each entry made once per device by the first call that
 *     needs it and published atomically, so first calls may race and one
 *     process may drive several devices.  Per host thread: the last CUDA
 *     error (qvg_last_cuda_error) and the wait settings of
 *     qvg_debug_set_wait.
 */
#ifndef QVG_H
#define QVG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QVG_OK = 0,
    QVG_ERR_INVALID_ARG = 1, /* a pointer, size or layout argument is wrong   */
    QVG_ERR_UNSUPPORTED = 2, /* valid, but outside what the kernels implement  */
    QVG_ERR_CUDA = 3,        /* a CUDA launch or runtime call failed           */
    QVG_ERR_TIMEOUT = 4,     /* a device-side wait exceeded its bound          */
    QVG_ERR_WORKSPACE = 5,   /* workspace missing or smaller than required     */
    QVG_ERR_CAPACITY = 6     /* the cache has no room for another chunk        */
} qvg_status;

/* qvg_params.flags */
#define QVG_QSAC 1            /* weight the clustering distance by qsac_w        */
#define QVG_PSAC 2            /* store the rank-8 key-error projection            */
#define QVG_GIVEN_CENTROIDS 4 /* start k-means from centroids the caller wrote   */
                              /* into this chunk's centroid slot                 */
#define QVG_OUTLIER 8         /* outlier split in the residual quantiser: per    */
                              /* group, a value above the group's P99 is kept   */
                              /* in fp16 (G <= 64; see outl_val below)           */
#define QVG_KEEP_MEANS 16     /* qvg_compress_chunk leaves each stage's fp32     */
                              /* centroid means in the workspace (see there)     */

#define QVG_TILE 128      /* chunks start at multiples of this many token slots */
#define QVG_PSAC_RANK 8   /* PSAC subspace rank ([QWM] PSAC: top-8 directions)  */
#define QVG_MAX_CLUSTERS 256
#define QVG_CACHE_NBUF 14

/* Output element types of qvg_decompress / qvg_attention. */
#define QVG_OUT_F32 0
#define QVG_OUT_BF16 1

/*
 * Method parameters ([QVG] "training strategy": the hyperparameters are the
 * cluster count C, the residual stage count L and the bit width b; the group
 * size G is that of the per-group quantiser, [P1] section 2 and [QVG]
 * "core tension").
 *   C          clusters per (chunk, head, stage), 0..256; 0 = plain per-group
 *              quantisation without centroid (the RTN baseline of [QVG]
 *              "main results").  C > N clusters a chunk of N tokens with N.
 *   L          progressive residual stages, >= 1 ([QVG] "Progressive
 *              Residual Quantization").  L = 1 is QVG, L > 1 QVG-Pro.
 *   bits       2 or 4.
 *   group      G: channels per quantisation group; head_dim % G == 0,
 *              G >= head_dim / 32.
 *   iters      Lloyd iterations (assign + update) before the final assign.
 *   scale_mode 0: S = max|r| / (2^{b-1} - 1)  ([QVG] "core tension");
 *              1: S = max|r| / 2, codes in [-2, 1]  ([P1] section 2; bits = 2).
 *   flags      QVG_QSAC | QVG_PSAC | QVG_GIVEN_CENTROIDS | QVG_OUTLIER |
 *              QVG_KEEP_MEANS.
 *   anchor_every  temporal anchors ([P2] section 3.3: the first frames of
 *              each window are kept at high precision so that errors do not
 *              pile up from window to window): 0 = none; k > 0 = chunk c of
 *              a cache (0-based) with c % k == 0 is stored as its bf16 K/V
 *              in the cache's anchor arena instead of being compressed.
 *   seed       k-means initialisation seed.
 * A cache must always be used with the C, L, bits and group it was sized for.
 */
typedef struct {
    int32_t C;
    int32_t L;
    int32_t bits;
    int32_t group;
    int32_t iters;
    int32_t scale_mode;
    int32_t flags;
    int32_t anchor_every;
    uint64_t seed;
} qvg_params;

/*
 * One compressed tensor (K or V) of one layer: an arena of token slots that
 * grows chunk by chunk ([QVG] "overall framework": the cache is processed
 * chunk by chunk; [P1] section 1: the cache grows linearly with frames).
 * Every buffer is caller-allocated device memory of the size that
 * qvg_cache_bytes reports, 16-byte aligned (the kernels read it with vector
 * loads; a misaligned buffer is refused with QVG_ERR_INVALID_ARG before any
 * launch).  Chunks start at slot multiples of QVG_TILE; the
 * slots between a chunk's end and the next multiple are padding.
 *   codes      uint8 [L][H][capacity][d*bits/8]  packed offset-binary codes:
 *              element j of a row at bits (j*bits)%8 of byte (j*bits)/8,
 *              value q + 2^{bits-1} ([QVG] "algorithm-system co-design":
 *              packed INT representation).
 *   scales     fp16  [L][H][capacity][d/G]       per-group scales.
 *   ids        uint8 [L][H][capacity]            cluster of each token.
 *   cent       bf16  [L][H][max_chunks][C][d]    centroids ([QVG] "overall
 *              framework": centroids kept in BF16).
 *   chunk_start int32 [max_chunks]  first slot of each chunk.
 *   chunk_len   int32 [max_chunks]  tokens in each chunk.
 *   tile_chunk  int32 [capacity/QVG_TILE] chunk owning each slot tile.
 *   psac_p     int8  [H][capacity][8]  PSAC projection codes (K only, or NULL).
 *   psac_s     fp16  [H][capacity]     PSAC per-token scales (or NULL).
 *   psac_basis fp32  [max_chunks][H][d][8] basis each chunk was encoded with
 *              (or NULL).
 *   outl_val   fp16  [L][H][capacity][d/G]  outlier split ([P2] section 3.4,
 *              "outlier separation"; with QVG_OUTLIER, else NULL): per group
 *              of a stage's residual, the value above the group's 99th
 *              percentile of |r| (linear interpolation; for G <= 100 at most
 *              the largest), fp16, saturated at 65504.  The group's scale and
 *              codes come from the other values; the outlier's code is 0 and
 *              it is rebuilt as outl_val + centroid.
 *   outl_idx   uint8 [L][H][capacity][d/G]  its channel within the group,
 *              0xFF when no value lies above the percentile (0 in outl_val).
 *   anchor     bf16  [A][H][d]  anchor chunks' K or V as given (with
 *              anchor_every > 0, else NULL).  Anchor chunk c starts at row
 *              (c / anchor_every) * S, S = capacity / max_chunks rounded up
 *              to QVG_TILE, and A = ceil(max_chunks / anchor_every) * S; an
 *              anchor chunk longer than S is refused (QVG_ERR_CAPACITY).  Its
 *              token slots in the other buffers are reserved but unused.
 *   chunk_anchor int32 [max_chunks]  first anchor row of each chunk, -1 for
 *              a compressed chunk (with anchor_every > 0, else NULL).
 * n_chunks and n_tokens are host-side counters that qvg_compress_chunk
 * advances; set both to 0 for an empty cache.  A cache can be saved and
 * restored by copying its buffers and these two counters.
 */
typedef struct {
    int32_t H;
    int32_t d;
    int32_t capacity_tokens; /* multiple of QVG_TILE */
    int32_t max_chunks;
    int32_t n_chunks;
    int32_t n_tokens;        /* first free slot (a multiple of QVG_TILE) */
    uint8_t *codes;
    uint16_t *scales;
    uint8_t *ids;
    uint16_t *cent;
    int32_t *chunk_start;
    int32_t *chunk_len;
    int32_t *tile_chunk;
    int8_t *psac_p;
    uint16_t *psac_s;
    float *psac_basis;
    uint16_t *outl_val;
    uint8_t *outl_idx;
    uint16_t *anchor;
    int32_t *chunk_anchor;
} qvg_cache;

/* Text for a status code (static storage; never NULL). */
const char *qvg_status_string(qvg_status s);

/*
 * Bytes of each cache buffer, in the order codes, scales, ids, cent,
 * chunk_start, chunk_len, tile_chunk, psac_p, psac_s, psac_basis, outl_val,
 * outl_idx, anchor, chunk_anchor (out_sizes has QVG_CACHE_NBUF entries).
 * The PSAC entries are 0 unless p->flags has QVG_PSAC, the outlier entries
 * 0 unless QVG_OUTLIER, the anchor entries 0 unless p->anchor_every > 0.  capacity_tokens must be a positive multiple of
 * QVG_TILE.  The total is the compressed footprint; [P1] section 1 gives
 * the uncompressed one, 2 (K and V) x layers x heads x head_dim x tokens x
 * bytes per element.
 */
qvg_status qvg_cache_bytes(const qvg_params *p, int32_t H, int32_t d,
                           int32_t capacity_tokens, int32_t max_chunks,
                           size_t out_sizes[QVG_CACHE_NBUF]);

/* Operations for qvg_workspace_size. */
#define QVG_OP_COMPRESS 0
#define QVG_OP_ATTENTION 1
#define QVG_OP_PSAC_BASIS 2

/*
 * Scratch bytes an operation needs for a chunk of n tokens (compress) or n
 * queries (attention), H KV heads, head_dim d and Hq query heads.  The
 * caller allocates it (256-byte aligned) and passes it to the call; its
 * contents need no initialisation and are dead after the call completes.
 * For attention it is 0 when n queries already fill the GPU (the cache is
 * then not split) and otherwise enough for the largest split the current
 * device's SM count can call for.
 */
qvg_status qvg_workspace_size(const qvg_params *p, int32_t op, int32_t n,
                              int32_t H, int32_t d, int32_t Hq, size_t *bytes);

/*
 * Compress one chunk of N new tokens and append it to `cache`
 * ([QVG] "overall framework", "Semantic-Aware Smoothing", "Progressive
 * Residual Quantization"; [QWM] QSAC and PSAC).  For each KV head and each
 * stage l = 1..L:
 *   k-means over the chunk's tokens: seeded init, p->iters Lloyd iterations,
 *   one final assignment (distance sum_j w_j (x_j - c_j)^2, w = qsac_w with
 *   QVG_QSAC, else 1; ties to the lowest cluster);
 *   residual r = X_l - C_id; per-group quantisation of r with fp16 scales
 *   (with QVG_OUTLIER, first splitting off each group's value above its
 *   P99 into the fp16 side list, [P2] section 3.4);
 *   X_{l+1} = X_l - (S q + C_id).
 * With QVG_PSAC, the remaining key error E = X_{L+1} is projected on the
 * rank-8 basis and stored as INT8 per token with one fp16 scale.
 * With p->anchor_every = k > 0, chunk n_chunks is an anchor when
 * n_chunks % k == 0 ([P2] section 3.3): its bf16 K or V is copied into the
 * anchor arena as given, and nothing else is computed for it.
 *   x_bf16     bf16 [N][H][d] device, the chunk's K or V (token-major),
 *              16-byte aligned.
 *   N          1 .. 65535 tokens.
 *   qsac_w     fp32 [H][d] device per-channel weights (required with QVG_QSAC,
 *              else ignored); positive and finite.
 *   psac_basis fp32 [H][d][8] device, 16-byte aligned (required with
 *              QVG_PSAC, else ignored); copied into the cache's per-chunk
 *              basis slot.
 *   cache      appended in place: the chunk occupies slots
 *              [n_tokens, n_tokens + N); n_chunks += 1 and n_tokens advances to
 *              the next multiple of QVG_TILE.  With QVG_GIVEN_CENTROIDS the
 *              caller has written all L stages' starting centroids into the
 *              new chunk's centroid slot (index n_chunks).
 *   workspace  device scratch of at least qvg_workspace_size(QVG_OP_COMPRESS).
 *              With QVG_KEEP_MEANS (and C > 0, iters >= 1) its first
 *              L*H*C*d*4 bytes hold, after the call, fp32 [L][H][C][d]: each
 *              stage's centroids of its last Lloyd update before the bf16
 *              rounding (the member mean in fp32; an empty cluster's kept
 *              centroid), for checking the update against a reference.
 * Returns QVG_ERR_CAPACITY when the chunk does not fit, in the slots or (an
 * anchor chunk) in its anchor rows; nothing is written then.
 */
qvg_status qvg_compress_chunk(const qvg_params *p, const void *x_bf16,
                              int32_t N, const float *qsac_w,
                              const float *psac_basis, qvg_cache *cache,
                              void *workspace, size_t ws_bytes, void *stream);

/*
 * Size of the fixed device scratch behind qvg_compress_chunk_noalloc: 32 MiB,
 * reserved on every device that loads the library, until the process exits.
 */
#define QVG_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * qvg_compress_chunk without a caller workspace (the pages have no
 * counterpart: this serves callers that cannot allocate device memory, such
 * as code inside a framework whose memory pool owns the whole device and
 * forbids further cudaMalloc calls, or code that must not risk the
 * device-wide synchronisation of cudaMalloc / cudaFree).  Same arguments,
 * results and errors as qvg_compress_chunk, which it calls; the workspace is
 * a fixed scratch array of QVG_NOALLOC_SCRATCH_BYTES inside the library.
 *   - Checks its arguments and the cache's capacity first, in the order
 *     and with the codes of qvg_compress_chunk; then returns
 *     QVG_ERR_WORKSPACE, before anything is launched, when
 *     qvg_workspace_size(QVG_OP_COMPRESS) for this call exceeds the scratch
 *     (for example L > 1 or PSAC on large chunks: use qvg_compress_chunk).
 *   - The first call on a device, made with that device current, looks up
 *     the scratch's device address (cudaGetSymbolAddress); make that first
 *     call before any stream capture.  It allocates nothing, ever.
 *   - Every call on a device shares the one scratch array, which keeps the
 *     last call's contents; nothing in it needs to start at zero.  Calls
 *     whose work overlaps on the GPU (different streams, or different host
 *     threads without ordering) race on the scratch: order them.
 */
qvg_status qvg_compress_chunk_noalloc(const qvg_params *p, const void *x_bf16,
                                      int32_t N, const float *qsac_w,
                                      const float *psac_basis, qvg_cache *cache,
                                      void *stream);

/*
 * Rebuild ntok token slots starting at slot tok0 ([QVG] "overall
 * framework": X_hat = S_X * X_INT + C_i, summed over stages per
 * "Progressive Residual Quantization"; with PSAC data present, plus the
 * correction P_hat U^T of [QWM] PSAC).  Stages are summed in fp32 in stage
 * order.  With QVG_OUTLIER, a value split off from its group is rebuilt as
 * its fp16 copy plus the centroid ([P2] section 3.4); an anchor chunk's
 * slots give its stored bf16 K/V ([P2] section 3.3).
 *   out      [ntok][H][d] fp32 or bf16 (out_dtype), 4-byte aligned (16-byte
 *            for fp32 and 8-byte for bf16 take vector stores); the caller's
 *            device buffer.  Padding slots give 0.
 * Errors: QVG_ERR_INVALID_ARG for tok0 < 0, ntok < 0, tok0 + ntok past
 * n_tokens or a misaligned out; ntok = 0 does nothing.
 */
qvg_status qvg_decompress(const qvg_params *p, const qvg_cache *cache,
                          int32_t tok0, int32_t ntok, void *out,
                          int32_t out_dtype, void *stream);

/*
 * Attention of Nq query tokens over every token in the compressed K and V
 * caches, reading codes, scales, ids and centroids directly and never
 * writing a reconstructed K or V to memory ([QVG] "algorithm-system
 * co-design": dequantisation fused with attention):
 *   O = softmax(scale * Q K_hat^T) V_hat, K_hat including the PSAC
 *   correction when the K cache holds PSAC data.
 *   q_bf16   bf16 [Nq][Hq][d], 16-byte aligned; query head hq reads KV head
 *            hq / (Hq / H).
 *   scale    softmax scale; <= 0 selects 1/sqrt(d).
 *   out      [Nq][Hq][d] fp32 or bf16, 16-byte aligned.
 *   lse      fp32 [Hq][Nq] natural-log log-sum-exp of the scaled logits, or NULL.
 *   top1     int32 [Hq][Nq] slot of the largest logit (lowest on ties), or NULL.
 *   workspace, ws_bytes  optional device scratch (256-byte aligned).  When
 *            ceil(Nq / 256) * Hq work units cannot occupy every SM (a few
 *            queries, as in decoding), a workspace of at least
 *            qvg_workspace_size(QVG_OP_ATTENTION, Nq, H, d, Hq) lets the call
 *            split the cache over more CTAs: each split writes its
 *            normalised fp32 output, log-sum-exp and best logit there, and a
 *            second kernel merges them (weights e^{lse_split - max}).  With no
 *            workspace, or a smaller one, the call runs unsplit; the results
 *            agree within fp32 rounding of the merge.
 * No mask: every cached token precedes the queries.  k and v must hold the
 * same chunks.  Errors: QVG_ERR_INVALID_ARG for a misaligned q_bf16 or out
 * (Nq > 0), QVG_ERR_WORKSPACE for a misaligned workspace.
 */
qvg_status qvg_attention(const qvg_params *p, const void *q_bf16, int32_t Nq,
                         int32_t Hq, const qvg_cache *k, const qvg_cache *v,
                         float scale, void *out, int32_t out_dtype, float *lse,
                         int32_t *top1, void *workspace, size_t ws_bytes,
                         void *stream);

/*
 * Attention of one autoregressive step: the Nq queries of the chunk being
 * generated attend to every token of the compressed cache (the earlier
 * chunks) and to the chunk's own n_cur tokens, whose K/V are still raw bf16
 * ([QVG] research background: chunk-by-chunk generation in which each chunk
 * attends to the cached K/V of the chunks before it; within a chunk there is
 * no mask).  The keys are the concatenation [K_hat ; K_cur] and the values
 * [V_hat ; V_cur], in one softmax:
 *   O = softmax(scale * Q [K_hat ; K_cur]^T) [V_hat ; V_cur].
 *   k_cur_bf16, v_cur_bf16  bf16 [n_cur][H][d], 16-byte aligned (the layout
 *            qvg_compress_chunk takes, so the same buffers are compressed
 *            into the cache after the step); read only, owned by the caller.
 *   n_cur    >= 0; 0 gives qvg_attention.  The cache may be empty (first
 *            chunk) when n_cur > 0.
 *   top1     current-chunk token j is reported as slot k->n_tokens + j, the
 *            slot it takes once the chunk is compressed into this cache.
 * The other arguments, the workspace rule and the outputs are those of
 * qvg_attention.  The raw rows are rounded to fp16 for the tensor core like
 * the reconstructed ones (exact inside fp16's normal range).
 * Errors: QVG_ERR_INVALID_ARG for n_cur < 0, a missing or misaligned raw
 * buffer, or no keys at all.
 */
qvg_status qvg_attention_ar(const qvg_params *p, const void *q_bf16, int32_t Nq,
                            int32_t Hq, const qvg_cache *k, const qvg_cache *v,
                            const void *k_cur_bf16, const void *v_cur_bf16,
                            int32_t n_cur, float scale, void *out,
                            int32_t out_dtype, float *lse, int32_t *top1,
                            void *workspace, size_t ws_bytes, void *stream);

/*
 * History-query statistics ([QWM] QSAC: per-channel activity of history
 * queries; PSAC: their second-moment matrix).  For KV head h, the query
 * heads hq with hq / (Hq/H) == h are pooled:
 *   M[h] (+)= sum over the n tokens and those heads of q q^T   fp32 [H][d][d]
 *   count (+)= n * Hq / H                                      int64 [1]
 *   w[h][j] = M[h][j][j] / count  (mean q_j^2, the QSAC weight) fp32 [H][d]
 * accumulate = 0 overwrites M and count, 1 adds to them.
 */
qvg_status quantwm_query_stats(const void *q_hist_bf16, int32_t n, int32_t Hq,
                               int32_t H, int32_t d, int32_t accumulate,
                               float *M, float *w, int64_t *count,
                               void *stream);

/*
 * PSAC basis ([QWM] PSAC: eigendecomposition of the history-query second
 * moment, top-8 eigenvectors as the principal subspace).  Jacobi
 * eigendecomposition of M[h] / count per head; outputs sorted by eigenvalue,
 * descending, each vector's largest-magnitude component made positive:
 *   U        fp32 [H][d][rank]  column k = k-th eigenvector
 *   eigvals  fp32 [H][rank]     eigenvalues of M / count
 *   energy_frac fp32 [H]        sum of the top-rank eigenvalues / trace
 * rank must be QVG_PSAC_RANK; d is 64 or 128.
 */
qvg_status quantwm_psac_basis(const float *M, const int64_t *count, int32_t H,
                              int32_t d, int32_t rank, float *U,
                              float *eigvals, float *energy_frac,
                              void *stream);

/*
 * Name of the CUDA error behind the latest QVG_ERR_CUDA returned to the
 * calling host thread ("cudaSuccess" if none); static storage.
 */
const char *qvg_last_cuda_error(void);

/*
 * Synchronise with `stream` (NULL: with the whole current device), then
 * return and clear the current device's latched device-side error (QVG_OK
 * if none).  The word is per device, so an error raised by work on another
 * stream that has completed is reported too; work still running elsewhere
 * may latch one after the read.  Returns QVG_ERR_CUDA when the
 * synchronisation reports a CUDA error.
 */
qvg_status qvg_get_status(void *stream);

/*
 * Device-side waits, a test hook for the failure path (the pages have no
 * counterpart).  Every wait of a kernel on a barrier (the k-means
 * assignment's tile and MMA hand-offs, the attention pipeline's) is bounded;
 * when the bound runs out the kernel stops its work, waits at the default
 * bound for the tensor-core work it has issued, frees its tensor memory,
 * latches QVG_ERR_TIMEOUT in the device word and returns, leaving the
 * context usable.  This call sets, for the kernels that the calling host
 * thread launches afterwards:
 *   limit_ns  the bound of those waits in nanoseconds; 0 restores the
 *             default of 2 s.
 *   inject    1: each such kernel additionally waits once on a barrier that
 *             nothing completes, with tensor-core work in flight, so that
 *             the bound runs out (qvg_get_status then reports
 *             QVG_ERR_TIMEOUT and the call's outputs are undefined);
 *             0: no such wait.
 * Errors: QVG_ERR_INVALID_ARG for inject other than 0 or 1.
 */
qvg_status qvg_debug_set_wait(uint64_t limit_ns, int32_t inject);

#ifdef __cplusplus
}
#endif

#endif /* QVG_H */
