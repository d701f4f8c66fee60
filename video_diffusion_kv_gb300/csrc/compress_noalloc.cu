// compress_noalloc.cu -- chunk compression for callers that cannot allocate
// device memory.
//
// qvg_compress_chunk needs a caller-provided device workspace.  Some callers
// have no way to provide one: code running inside a framework whose memory
// pool owns the whole device and forbids further cudaMalloc calls, or code
// that must not risk the device-wide synchronisation cudaMalloc / cudaFree
// may perform.  qvg_compress_chunk_noalloc serves them from a fixed scratch
// array that lives in this file as a statically allocated __device__
// variable: it is reserved when the library's module is loaded on a device
// and held by every device that loads the library until the process exits.
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(QVG_NOALLOC_SCRATCH_BYTES);

// The scratch array.  In host code this name is only a host-side stand-in,
// never a device address: host code must use the address returned by
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_compress_scratch[kScratchBytes];

// Per-device address of g_compress_scratch, looked up on the first call made
// with that device current.
std::mutex g_setup_mutex;
void *g_scratch_ptr[64] = {};

qvg_status scratch_for_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return QVG_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_compress_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            (void)cudaGetLastError();
            qvg::note_cuda_error(e);
            return QVG_ERR_CUDA;
        }
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return QVG_OK;
}

}  // namespace

extern "C" qvg_status qvg_compress_chunk_noalloc(const qvg_params *p, const void *x_bf16, int32_t N,
                                                 const float *qsac_w, const float *psac_basis,
                                                 qvg_cache *cache, void *stream) {
    // argument, capacity and size errors first, in qvg_compress_chunk's order
    size_t need = 0;
    qvg_status s = qvg::check_compress_args(p, x_bf16, N, qsac_w, psac_basis, cache, &need);
    if (s != QVG_OK) return s;
    if (need > kScratchBytes) return QVG_ERR_WORKSPACE;  // beyond the fixed scratch: use qvg_compress_chunk
    void *scratch = nullptr;
    if ((s = scratch_for_current_device(&scratch)) != QVG_OK) return s;
    return qvg_compress_chunk(p, x_bf16, N, qsac_w, psac_basis, cache, scratch, kScratchBytes, stream);
}
