// quantwm.cu -- QuantWM history-query statistics and PSAC basis (sm_103a).
//
// QuantWM write-up, QSAC: the activity of history queries per channel weights
// the clustering distance (reading: activity = E[q_j^2]); PSAC: the top-8
// eigenvectors of the history-query second-moment matrix span the subspace in
// which the key error is corrected.
#include <algorithm>

#include "common.cuh"

namespace qvg {

// M[h] (+)= sum over tokens and the query heads of group h of q q^T, one CTA
// per 32x32 block of M[h]; fp32 accumulation over 64-token smem batches.
template <int D>
__global__ void __launch_bounds__(256) k_query_stats(const uint16_t *__restrict__ q, int n, int Hq,
                                                    int grp, int accumulate, float *__restrict__ M) {
    __shared__ float As[64][33];
    __shared__ float Bs[64][33];
    const int h = blockIdx.z, a0 = blockIdx.y * 32, b0 = blockIdx.x * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 warps: rows ty*4..ty*4+3
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const int rows = n * grp;
    for (int r0 = 0; r0 < rows; r0 += 64) {
        for (int i = threadIdx.x; i < 64 * 32; i += 256) {
            const int rr = i / 32, c = i % 32, r = r0 + rr;
            float va = 0.f, vb = 0.f;
            if (r < rows) {
                const int t = r / grp, hq = h * grp + r % grp;
                const uint16_t *qr = q + (static_cast<size_t>(t) * Hq + hq) * D;
                va = bf16_to_f32(qr[a0 + c]);
                vb = bf16_to_f32(qr[b0 + c]);
            }
            As[rr][c] = va;
            Bs[rr][c] = vb;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < 64; ++k) {
            const float bv = Bs[k][tx];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = fmaf(As[k][ty * 4 + i], bv, acc[i]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const size_t o = (static_cast<size_t>(h) * D + a0 + ty * 4 + i) * D + b0 + tx;
        M[o] = accumulate ? M[o] + acc[i] : acc[i];
    }
}

// count (+)= n * grp; w[h][j] = M[h][j][j] / count.  One CTA.
__global__ void k_stats_finalize(const float *__restrict__ M, int H, int D, int64_t add,
                                 int accumulate, float *__restrict__ w, int64_t *count) {
    __shared__ int64_t c;
    if (threadIdx.x == 0) c = (accumulate ? *count : 0) + add;
    __syncthreads();
    const float cf = static_cast<float>(c);
    for (int i = threadIdx.x; i < H * D; i += blockDim.x) {
        const int h = i / D, j = i % D;
        w[i] = M[(static_cast<size_t>(h) * D + j) * D + j] / cf;
    }
    __syncthreads();
    if (threadIdx.x == 0) *count = c;
}

qvg_status launch_query_stats(const uint16_t *q, int n, int Hq, int H, int d, int accumulate,
                              float *M, float *w, int64_t *count, cudaStream_t st) {
    const int grp = Hq / H;
    dim3 grid(d / 32, d / 32, H);
    if (d == 64)
        k_query_stats<64><<<grid, 256, 0, st>>>(q, n, Hq, grp, accumulate, M);
    else
        k_query_stats<128><<<grid, 256, 0, st>>>(q, n, Hq, grp, accumulate, M);
    QVG_LAUNCH_CHECK();
    k_stats_finalize<<<1, 1024, 0, st>>>(M, H, d, static_cast<int64_t>(n) * grp, accumulate, w, count);
    QVG_LAUNCH_CHECK();
    return QVG_OK;
}

// ---------------------------------------------------------------------------
// Jacobi eigendecomposition of M[h] / count, one CTA per head.  Parallel
// (round-robin) ordering: in each step the d/2 disjoint pairs of a
// tournament schedule are rotated at once, which for disjoint pairs is the
// same as rotating them one after another; d - 1 steps make a sweep.  Each
// rotation uses the stable angle of the textbook cyclic Jacobi method
// (Golub & Van Loan, "Matrix Computations"): theta = (a_qq - a_pp) /
// (2 a_pq), t = sign(theta) / (|theta| + sqrt(1 + theta^2)),
// c = 1/sqrt(1 + t^2), s = t c; A <- J^T A J, V <- V J.  Stops when the
// off-diagonal Frobenius norm falls below 1e-6 of ||A||_F (fp32) or after 40
// sweeps.
constexpr int JD = 128;  // maximum head_dim

// Round-robin schedule: position 0 keeps element 0 and positions 1 .. D-1
// rotate by one each step, so after `step` steps position i >= 1 holds
// ((i - 1 - step) mod (D - 1)) + 1; pair pi of the step is (position pi,
// position D - 1 - pi), ordered p < q.
template <int D>
__device__ __forceinline__ void jacobi_pair(int pi, int step, int &p, int &q) {
    auto at = [&](int i) { return i == 0 ? 0 : ((i - 1 - step) % (D - 1) + (D - 1)) % (D - 1) + 1; };
    p = at(pi);
    q = at(D - 1 - pi);
    if (p > q) {
        const int t = p;
        p = q;
        q = t;
    }
}

// Shared memory: A and V [D][D] fp32, the step's rotations and pairs.  The
// row update runs with consecutive threads on consecutive entries of a row
// (conflict-free); the column update with consecutive threads on different
// pairs of the same row (a column walk would put a warp in one bank).
template <int D>
__global__ void __launch_bounds__(512) k_psac_jacobi(const float *__restrict__ Min,
                                                    const int64_t *__restrict__ count, int r,
                                                    float *__restrict__ U, float *__restrict__ eig,
                                                    float *__restrict__ frac) {
    constexpr int HALF = D / 2;
    extern __shared__ float js[];
    float *A = js;                 // [D][D]
    float *V = A + D * D;          // [D][D]
    float *cs = V + D * D;         // [D/2]
    float *sn = cs + HALF;         // [D/2]
    int *pp = reinterpret_cast<int *>(sn + HALF);  // [D/2]
    int *qq = pp + HALF;                           // [D/2]
    __shared__ float red[16];
    __shared__ int done;
    __shared__ int top[QVG_PSAC_RANK];
    const int h = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
    const float inv = 1.0f / static_cast<float>(*count);
    for (int i = tid; i < D * D; i += nt) {
        A[i] = Min[static_cast<size_t>(h) * D * D + i] * inv;
        V[i] = (i / D == i % D) ? 1.0f : 0.0f;
    }
    __syncthreads();
    // ||A||_F
    float part = 0.f;
    for (int i = tid; i < D * D; i += nt) part += A[i] * A[i];
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if ((tid & 31) == 0) red[tid >> 5] = part;
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int i = 0; i < nt / 32; ++i) s += red[i];
        red[15] = s;
    }
    __syncthreads();
    const float fro2 = red[15];
    for (int sweep = 0; sweep < 40; ++sweep) {
        float off = 0.f;
        for (int i = tid; i < D * D; i += nt)
            if (i / D != i % D) off += A[i] * A[i];
        for (int o = 16; o > 0; o >>= 1) off += __shfl_xor_sync(0xffffffffu, off, o);
        __syncthreads();
        if ((tid & 31) == 0) red[tid >> 5] = off;
        __syncthreads();
        if (tid == 0) {
            float s = 0.f;
            for (int i = 0; i < nt / 32; ++i) s += red[i];
            done = s <= 1e-12f * fro2;
        }
        __syncthreads();
        if (done) break;
        for (int step = 0; step < D - 1; ++step) {
            if (tid < HALF) {
                int p, q;
                jacobi_pair<D>(tid, step, p, q);
                const float apq = A[p * D + q];
                float c = 1.f, s = 0.f;
                if (apq != 0.f) {
                    const float theta = (A[q * D + q] - A[p * D + p]) / (2.f * apq);
                    const float t = (theta >= 0.f ? 1.f : -1.f) / (fabsf(theta) + sqrtf(1.f + theta * theta));
                    c = 1.f / sqrtf(1.f + t * t);
                    s = t * c;
                }
                cs[tid] = c;
                sn[tid] = s;
                pp[tid] = p;
                qq[tid] = q;
            }
            __syncthreads();
            // rows: A <- J^T A
            for (int i = tid; i < HALF * D; i += nt) {
                const int pi = i / D, k = i % D;
                const int p = pp[pi], q = qq[pi];
                const float c = cs[pi], s = sn[pi];
                const float apk = A[p * D + k], aqk = A[q * D + k];
                A[p * D + k] = c * apk - s * aqk;
                A[q * D + k] = s * apk + c * aqk;
            }
            __syncthreads();
            // columns: A <- A J, V <- V J
            for (int i = tid; i < HALF * D; i += nt) {
                const int k = i / HALF, pi = i % HALF;
                const int p = pp[pi], q = qq[pi];
                const float c = cs[pi], s = sn[pi];
                const float akp = A[k * D + p], akq = A[k * D + q];
                A[k * D + p] = c * akp - s * akq;
                A[k * D + q] = s * akp + c * akq;
                const float vkp = V[k * D + p], vkq = V[k * D + q];
                V[k * D + p] = c * vkp - s * vkq;
                V[k * D + q] = s * vkp + c * vkq;
            }
            __syncthreads();
        }
    }
    // top-r eigenpairs by descending eigenvalue (lowest index on ties)
    if (tid == 0) {
        float tr = 0.f, sum = 0.f;
        for (int i = 0; i < D; ++i) tr += A[i * D + i];
        for (int k = 0; k < r; ++k) {
            int b = -1;
            for (int i = 0; i < D; ++i) {
                bool used = false;
                for (int m = 0; m < k; ++m) used |= (top[m] == i);
                if (used) continue;
                if (b < 0 || A[i * D + i] > A[b * D + b]) b = i;
            }
            top[k] = b;
            eig[h * r + k] = A[b * D + b];
            sum += A[b * D + b];
        }
        frac[h] = tr > 0.f ? sum / tr : 0.f;
    }
    __syncthreads();
    if (tid < r) {
        const int col = top[tid];
        int big = 0;
        for (int k = 1; k < D; ++k)
            if (fabsf(V[k * D + col]) > fabsf(V[big * D + col])) big = k;
        const float sg = V[big * D + col] < 0.f ? -1.f : 1.f;
        for (int k = 0; k < D; ++k) U[(static_cast<size_t>(h) * D + k) * r + tid] = sg * V[k * D + col];
    }
}

qvg_status launch_psac_basis(const float *M, const int64_t *count, int H, int d, int rank, float *U,
                             float *eig, float *frac, cudaStream_t st) {
    const size_t smem = (2 * static_cast<size_t>(d) * d + d) * sizeof(float) + d * sizeof(int);
    {
        static std::atomic<uint64_t> done128{0}, done64{0};
        const int most = static_cast<int>((2 * JD * JD + JD) * sizeof(float) + JD * sizeof(int));
        qvg_status s = smem_limit_once(done128, reinterpret_cast<const void *>(k_psac_jacobi<128>), most);
        if (s == QVG_OK) s = smem_limit_once(done64, reinterpret_cast<const void *>(k_psac_jacobi<64>), most);
        if (s != QVG_OK) return s;
    }
    if (d == 128)
        k_psac_jacobi<128><<<H, 512, smem, st>>>(M, count, rank, U, eig, frac);
    else if (d == 64)
        k_psac_jacobi<64><<<H, 512, smem, st>>>(M, count, rank, U, eig, frac);
    else
        return QVG_ERR_UNSUPPORTED;
    QVG_LAUNCH_CHECK();
    return QVG_OK;
}

}  // namespace qvg
