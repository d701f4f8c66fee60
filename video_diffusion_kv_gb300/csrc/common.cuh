// common.cuh -- device helpers shared by the libqvg kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "../../include/qvg.h"

namespace qvg {

// ---- number formats -------------------------------------------------------

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float f16_to_f32(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}
__device__ __forceinline__ uint16_t f32_to_f16(float f) {
    return __half_as_ushort(__float2half_rn(f));
}

// ---- per-group symmetric quantiser ----------------------------------------
// Quant VideoGen notes, "core tension": S = max|r| / (2^{b-1} - 1),
// q = round(r / S); page-1 toy quantiser (scale_mode 1): S = max|r| / 2,
// q clamped to [-2, 1].  The scale is stored as fp16 (saturated at 65504)
// and the codes use the stored value; IEEE division, round-half-even.  Each
// step is a separately rounded IEEE operation (no contraction), so the
// codes agree bit for bit with any other IEEE implementation of the same
// definition.

__device__ __forceinline__ uint16_t group_scale_f16(float amax, int bits, int mode) {
    const float den = mode == 0 ? static_cast<float>((1 << (bits - 1)) - 1) : 2.0f;
    float S = __fdiv_rn(amax, den);
    S = fminf(S, 65504.0f);
    return f32_to_f16(S);
}

// The code of r at the stored scale Sp: clamp(rint(fl(r / Sp)), -2^{b-1},
// 2^{b-1} - 1), 0 when Sp is 0 -- without a division per element: inv =
// fl(1 / Sp) (one division per group), y = fl(r inv).  With x = r / Sp
// exactly, |y - x| <= |x| 2^-23
// (two roundings of at most 2^-24 each) and |fl(x) - x| <= |x| 2^-24, so y
// and the IEEE quotient fl(x) round to the same integer unless a
// half-integer lies between them or on one of them, which needs y within
// |y| 2^-21 of a half-integer (a margin of more than twice the bound); those
// elements take the division.  y - rint(y) is exact (Sterbenz), and beyond
// 2^23 y is an integer and the clamp decides, so the code is bit for bit
// the one the division gives.
__device__ __forceinline__ int quant_code_rcp(float r, float Sp, float inv, int bits) {
    if (!(Sp > 0.0f)) return 0;
    const float qmax = static_cast<float>((1 << (bits - 1)) - 1);
    const float y = __fmul_rn(r, inv);
    float t = rintf(y);
    if (0.5f - fabsf(y - t) <= fabsf(y) * 0x1p-21f) t = rintf(__fdiv_rn(r, Sp));
    t = fminf(fmaxf(t, -qmax - 1.0f), qmax);
    return static_cast<int>(t);
}

// ---- sticky device error word --------------------------------------------
// One int per device (defined in api.cu; kernels get its address).  The
// first error wins; qvg_get_status reads and clears it.
__device__ __forceinline__ void raise_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Programmatic dependent launch (launch_pdl below): a kernel may run its
// prologue while the previous kernel of the stream finishes; pdl_wait()
// blocks until that kernel has completed and its writes are visible (a no-op
// for a normal launch), pdl_trigger() lets the next kernel start its own
// prologue.  Kernels here trigger only after their own wait, so two kernels
// back in the stream have always completed when a kernel starts.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace qvg

// ---- host-side launch plumbing (internal, not part of the ABI) ------------

namespace qvg {
// Records the CUDA error behind the latest QVG_ERR_CUDA of this host thread.
void note_cuda_error(cudaError_t e);
}

#define QVG_LAUNCH_CHECK()                                        \
    do {                                                          \
        const cudaError_t qvg_e_ = cudaPeekAtLastError();         \
        if (qvg_e_ != cudaSuccess) {                              \
            (void)cudaGetLastError();                             \
            ::qvg::note_cuda_error(qvg_e_);                       \
            return QVG_ERR_CUDA;                                  \
        }                                                         \
    } while (0)

namespace qvg {

// Launch with programmatic stream serialisation (see pdl_wait / pdl_trigger).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Device address of the current device's error word (looked up once per
// device, race-free), or NULL if the current device cannot be determined.
int *device_error_word();

// ---- per-device launch set-up -------------------------------------------
// Everything a launch needs to know about the device is looked up once per
// device (the device current on the calling host thread) and kept in tables
// indexed by device number; each entry is published atomically, so first
// calls may come from several host threads at once, and one process may
// drive several devices.
constexpr int kMaxDevices = 64;

// Multiprocessor count of the current device (152 if it cannot be read).
int sm_count_current();

// Raises `func`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device: `done` is the call site's bit mask of devices
// already set up (a function-local static at every call site).
qvg_status smem_limit_once(std::atomic<uint64_t> &done, const void *func, int bytes);

// Bound of the device-side waits of the kernels that the calling host thread
// launches next (nanoseconds), and whether those launches add one wait on a
// barrier that nothing arrives at (the bounded-wait test hook,
// qvg_debug_set_wait in qvg.h).
uint64_t wait_limit_ns();
int wait_inject();

// The argument checks of qvg_compress_chunk, in its order, without the
// workspace: QVG_OK and the workspace the call needs (*ws_need), or the
// first error.
qvg_status check_compress_args(const qvg_params *p, const void *x_bf16, int N, const float *qsac_w,
                               const float *psac_basis, const qvg_cache *cache, size_t *ws_need);

// Launchers implemented in the kernel translation units.  All return a
// qvg_status and only enqueue work on `st`.
qvg_status launch_kmeans_init(const uint16_t *g, int N, int H, int d, int C, int Ce,
                              uint64_t seed, int chunk, int stage,
                              uint16_t *cent, size_t cent_head_stride, const float *w, float *cnorm,
                              cudaStream_t st);
qvg_status launch_centroid_norms(const uint16_t *cent, size_t cent_head_stride, int H,
                                 int C, int d, const float *w, float *cnorm, cudaStream_t st);
// xnorm [H][N]: ||x||_w^2 per token (launch_row_norms, once per stage).
qvg_status launch_kmeans_assign(const uint16_t *g, int N, int H, int d,
                                const uint16_t *cent, size_t cent_head_stride, int Ce,
                                const float *cnorm, int C, const float *w, const float *xnorm,
                                int32_t *ids, cudaStream_t st);
qvg_status launch_row_norms(const uint16_t *g, int N, int H, int d, const float *w, float *xnorm,
                            cudaStream_t st);
// means (optional) [H][C][d]: the fp32 member means before the bf16
// rounding (an empty cluster: its kept centroid).
qvg_status launch_kmeans_update(const void *xin, bool xin_f32, int N, int H, int d,
                                const int32_t *ids, uint16_t *cent, size_t cent_head_stride, int Ce, int C,
                                const float *w, float *cnorm, float *means, cudaStream_t st);
qvg_status launch_residual_quant(const void *xin, bool xin_f32, int N, int H, int d,
                                 const uint16_t *cent, size_t cent_head_stride, int C,
                                 const int32_t *ids, int bits, int group, int mode,
                                 uint8_t *codes, uint16_t *scales, uint8_t *ids_out,
                                 size_t slot_head_stride, float *delta_out,
                                 uint16_t *gbf_out, const float *psac_U, int8_t *psac_p,
                                 uint16_t *psac_s, size_t psac_head_stride, uint16_t *outl_val,
                                 uint8_t *outl_idx, cudaStream_t st);
qvg_status launch_chunk_table(int chunk, int slot0, int N, int32_t *chunk_start,
                              int32_t *chunk_len, int32_t *tile_chunk, int32_t *chunk_anchor,
                              int anchor_row, cudaStream_t st);
qvg_status launch_decompress(const qvg_params *p, const qvg_cache *c, int tok0, int ntok,
                             void *out, int out_dtype, cudaStream_t st);
// Rows of the anchor arena reserved per anchor chunk: the capacity per
// chunk, rounded up to a whole tile.
inline int anchor_stride(int capacity_tokens, int max_chunks) {
    return ((capacity_tokens / max_chunks + QVG_TILE - 1) / QVG_TILE) * QVG_TILE;
}
qvg_status launch_attention_ws(const qvg_params *p, const uint16_t *q, int Nq, int Hq,
                               const qvg_cache *k, const qvg_cache *v, float scale_log2,
                               const uint16_t *k_cur, const uint16_t *v_cur, int n_cur,
                               void *out, int out_dtype, float *lse, int32_t *top1,
                               void *workspace, size_t ws_bytes, cudaStream_t st);
// Cache splits qvg_attention uses for Nq queries x Hq heads (n_tiles < 0:
// the most any cache length can need), and the workspace they take.
int attention_splits(int Nq, int Hq, int n_tiles);
size_t attention_split_bytes(int Nq, int Hq, int d, int splits);
qvg_status launch_query_stats(const uint16_t *q, int n, int Hq, int H, int d, int accumulate,
                              float *M, float *w, int64_t *count, cudaStream_t st);
qvg_status launch_psac_basis(const float *M, const int64_t *count, int H, int d, int rank,
                             float *U, float *eig, float *frac, cudaStream_t st);

}  // namespace qvg
