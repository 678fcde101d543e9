// subspace.cu -- the geometry behind the CCQ read: the dominant eigenspace of
// the key covariance Sigma_T = C / n - mu mu^T (mu = m / n) of a head's final
// state, and how much of a given key lies in it.
//
// The article's diagnosis (10100.com, "method": keys concentrate in a few
// dominant directions; a needle that must be retrieved lies off them, so a
// read that does not discount the dominant directions drowns it) is measured
// here on the state the forward produced: the top-k eigenvectors of Sigma_T
// by orthogonal (subspace) iteration, and for a key x the captured energy
// |U^T x|^2 / |x|^2.
//
// One CTA per head.  Sigma lives in shared memory (fp32, dk x dk); each
// iteration is W = Sigma V, then V = W R^-1 with R the Cholesky factor of
// W^T W (Cholesky-QR); at the end the Rayleigh-Ritz step diagonalises
// H = V^T Sigma V (k x k) by cyclic Jacobi and rotates V to the Ritz vectors,
// sorted by Ritz value.
#include <cuda_bf16.h>

#include "common.cuh"

namespace ccq {
namespace subspace {

constexpr int NTHREADS = 256;
constexpr int KMAX = 32;

template <int DK>
__global__ void __launch_bounds__(NTHREADS)
sigma_subspace_kernel(const float *__restrict__ C, const float *__restrict__ m, double n, int k,
                      int iters, float *__restrict__ U, float *__restrict__ ritz) {
    extern __shared__ float4 sm_f4[];  // 16-byte aligned (float2 / float4 reads below)
    float *sm = reinterpret_cast<float *>(sm_f4);
    float *Sig = sm;                    // [DK][DK]
    float *V = Sig + DK * DK;           // [DK][KMAX]
    float *Wm = V + DK * KMAX;          // [DK][KMAX]
    float *G = Wm + DK * KMAX;          // [KMAX][KMAX]  (W^T W, then R, then H)
    float *Q = G + KMAX * KMAX;         // [KMAX][KMAX]  (Jacobi rotations)
    float *mu = Q + KMAX * KMAX;        // [DK]
    const int tid = threadIdx.x, bh = blockIdx.x;
    const float *Cb = C + (size_t)bh * DK * DK;
    const float rn = (float)(1.0 / n);

    for (int i = tid; i < DK; i += NTHREADS) mu[i] = m[(size_t)bh * DK + i] * rn;
    __syncthreads();
    for (int x = tid; x < DK * DK; x += NTHREADS) {
        const int i = x / DK, j = x % DK;
        Sig[x] = Cb[x] * rn - mu[i] * mu[j];
    }
    // deterministic start: e_j plus a fixed spread over all coordinates
    for (int x = tid; x < DK * k; x += NTHREADS) {
        const int i = x / k, j = x % k;
        V[i * KMAX + j] = (i == j ? 1.f : 0.f) + 0.01f * (float)(((i * 7 + j * 13) % 17) - 8);
    }
    __syncthreads();

    // Wm = Sig V.  A thread forms a 2-row x 4-column block; Sig is symmetric,
    // so rows i0, i0+1 are read as column entries Sig[l][i0..i0+1] (one float2,
    // consecutive across lanes) and V[l][j0..j0+3] as one float4.
    auto matmul_sigma = [&]() {
        const int kq = (k + 3) / 4;
        for (int blk = tid; blk < (DK / 2) * kq; blk += NTHREADS) {
            const int i0 = 2 * (blk / kq), j0 = 4 * (blk % kq);
            float a[2][4] = {};
            for (int l = 0; l < DK; ++l) {
                const float2 sg = *reinterpret_cast<const float2 *>(&Sig[l * DK + i0]);
                const float4 v4 = *reinterpret_cast<const float4 *>(&V[l * KMAX + j0]);
                a[0][0] = fmaf(sg.x, v4.x, a[0][0]);
                a[0][1] = fmaf(sg.x, v4.y, a[0][1]);
                a[0][2] = fmaf(sg.x, v4.z, a[0][2]);
                a[0][3] = fmaf(sg.x, v4.w, a[0][3]);
                a[1][0] = fmaf(sg.y, v4.x, a[1][0]);
                a[1][1] = fmaf(sg.y, v4.y, a[1][1]);
                a[1][2] = fmaf(sg.y, v4.z, a[1][2]);
                a[1][3] = fmaf(sg.y, v4.w, a[1][3]);
            }
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (j0 + c < k) Wm[(i0 + r) * KMAX + j0 + c] = a[r][c];
        }
    };
    auto cholqr = [&]() {  // V = Wm R^-1, R^T R = Wm^T Wm
        for (int x = tid; x < k * k; x += NTHREADS) {
            const int a = x / k, b = x % k;
            float s = 0.f;
            for (int l = 0; l < DK; ++l) s += Wm[l * KMAX + a] * Wm[l * KMAX + b];
            G[a * KMAX + b] = s;
        }
        __syncthreads();
        if (tid < 32) {  // Cholesky, upper factor R in place; warp 0, lane b owns column b
            const int b = tid;
            for (int a = 0; a < k; ++a) {
                float d = G[a * KMAX + a];  // every lane forms the pivot (same reads)
                for (int l = 0; l < a; ++l) d -= G[l * KMAX + a] * G[l * KMAX + a];
                d = sqrtf(fmaxf(d, 1e-30f));
                if (b > a && b < k) {
                    float s = G[a * KMAX + b];
                    for (int l = 0; l < a; ++l) s -= G[l * KMAX + a] * G[l * KMAX + b];
                    G[a * KMAX + b] = s / d;
                }
                __syncwarp();
                if (b == a) G[a * KMAX + a] = d;
                __syncwarp();
            }
        }
        __syncthreads();
        // rows of V: v_i = w_i R^-1 (forward substitution along the row)
        for (int i = tid; i < DK; i += NTHREADS) {
            for (int b = 0; b < k; ++b) {
                float s = Wm[i * KMAX + b];
                for (int a = 0; a < b; ++a) s -= V[i * KMAX + a] * G[a * KMAX + b];
                V[i * KMAX + b] = s / G[b * KMAX + b];
            }
        }
        __syncthreads();
    };

    for (int x = tid; x < DK * k; x += NTHREADS) Wm[(x / k) * KMAX + x % k] = V[(x / k) * KMAX + x % k];
    __syncthreads();
    cholqr();
    for (int it = 0; it < iters; ++it) {
        matmul_sigma();
        __syncthreads();
        cholqr();
    }

    // ---- Rayleigh-Ritz: H = V^T Sig V (Wm = Sig V), Jacobi on H (thread 0)
    matmul_sigma();
    __syncthreads();
    for (int x = tid; x < k * k; x += NTHREADS) {
        const int a = x / k, b = x % k;
        float s = 0.f;
        for (int l = 0; l < DK; ++l) s += V[l * KMAX + a] * Wm[l * KMAX + b];
        G[a * KMAX + b] = s;
        Q[a * KMAX + b] = a == b ? 1.f : 0.f;
    }
    __syncthreads();
    if (tid < 32) {  // warp 0: lane l owns row / column l of each rotation's update
        const int l = tid;
        if (l == 0)
            for (int a = 0; a < k; ++a)  // symmetrise
                for (int b = a + 1; b < k; ++b) {
                    const float s = 0.5f * (G[a * KMAX + b] + G[b * KMAX + a]);
                    G[a * KMAX + b] = G[b * KMAX + a] = s;
                }
        __syncwarp();
        for (int sweep = 0; sweep < 30; ++sweep) {
            float off = 0.f;  // every lane forms the same sum (same reads, same order)
            for (int a = 0; a < k; ++a)
                for (int b = a + 1; b < k; ++b) off += G[a * KMAX + b] * G[a * KMAX + b];
            if (off < 1e-20f) break;
            for (int a = 0; a < k; ++a)
                for (int b = a + 1; b < k; ++b) {
                    const float hab = G[a * KMAX + b];
                    if (fabsf(hab) < 1e-30f) continue;  // warp-uniform
                    // plane rotation J (c, s) with (J^T H J)[a][b] = 0: the classical
                    // cyclic Jacobi method for symmetric matrices
                    const float tau = (G[b * KMAX + b] - G[a * KMAX + a]) / (2.f * hab);
                    const float t = (tau >= 0.f ? 1.f : -1.f) / (fabsf(tau) + sqrtf(1.f + tau * tau));
                    const float c = 1.f / sqrtf(1.f + t * t), s = t * c;
                    __syncwarp();  // every lane has read this rotation's inputs
                    if (l < k) {  // H <- H J: columns a and b, row l
                        const float x = G[l * KMAX + a], y = G[l * KMAX + b];
                        G[l * KMAX + a] = c * x - s * y;
                        G[l * KMAX + b] = s * x + c * y;
                    }
                    __syncwarp();
                    if (l < k) {  // H <- J^T H: rows a and b, column l
                        const float x = G[a * KMAX + l], y = G[b * KMAX + l];
                        G[a * KMAX + l] = c * x - s * y;
                        G[b * KMAX + l] = s * x + c * y;
                        const float qx = Q[l * KMAX + a], qy = Q[l * KMAX + b];  // Q <- Q J
                        Q[l * KMAX + a] = c * qx - s * qy;
                        Q[l * KMAX + b] = s * qx + c * qy;
                    }
                    __syncwarp();
                }
        }
    }
    __syncthreads();
    if (tid == 0) {
        // order by Ritz value, descending: a permutation stored in row 0 of Wm
        for (int a = 0; a < k; ++a) Wm[a] = (float)a;
        for (int a = 0; a < k; ++a)
            for (int b = a + 1; b < k; ++b)
                if (G[(int)Wm[b] * KMAX + (int)Wm[b]] > G[(int)Wm[a] * KMAX + (int)Wm[a]]) {
                    const float t = Wm[a];
                    Wm[a] = Wm[b];
                    Wm[b] = t;
                }
    }
    __syncthreads();
    for (int a = tid; a < k; a += NTHREADS) {
        const int pa = (int)Wm[a];
        ritz[(size_t)bh * k + a] = G[pa * KMAX + pa];
    }
    for (int x = tid; x < DK * k; x += NTHREADS) {  // U[:, a] = V Q[:, perm a]
        const int i = x / k, a = x % k, pa = (int)Wm[a];
        float s = 0.f;
        for (int l = 0; l < k; ++l) s += V[i * KMAX + l] * Q[l * KMAX + pa];
        U[((size_t)bh * DK + i) * k + a] = s;
    }
}

// align[bh, j] = |U^T x|^2 / |x|^2 for x = X[bh, j, :]; one warp per key.
template <typename TIn>
__global__ void __launch_bounds__(NTHREADS)
alignment_kernel(const float *__restrict__ U, const TIn *__restrict__ X, int dk, int k, int nx,
                 int BH, float *__restrict__ align) {
    const int warp = (blockIdx.x * NTHREADS + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= BH * nx) return;
    const int bh = warp / nx;
    const TIn *x = X + (size_t)warp * dk;
    const float *Ub = U + (size_t)bh * dk * k;
    float xx = 0.f;
    for (int i = lane; i < dk; i += 32) {
        const float xi = io<TIn>::load(x + i);
        xx += xi * xi;
    }
    xx = warp_sum(xx);
    float cap = 0.f;
    for (int a = 0; a < k; ++a) {
        float s = 0.f;
        for (int i = lane; i < dk; i += 32) s += Ub[i * k + a] * io<TIn>::load(x + i);
        s = warp_sum(s);
        cap += s * s;
    }
    if (lane == 0) align[warp] = xx > 0.f ? cap / xx : 0.f;
}

}  // namespace subspace

size_t sigma_subspace_smem(int dk) {
    using namespace subspace;
    return sizeof(float) * ((size_t)dk * dk + 2 * (size_t)dk * KMAX + 2 * KMAX * KMAX + dk);
}

cudaError_t launch_sigma_subspace(const float *C, const float *m, double n, int BH, int dk, int k,
                                  int iters, float *U, float *ritz, cudaStream_t st) {
    using namespace subspace;
    const size_t bytes = sigma_subspace_smem(dk);
    if (dk == 64) {
        cudaError_t e = cudaFuncSetAttribute(sigma_subspace_kernel<64>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)bytes);
        if (e != cudaSuccess) return e;
        sigma_subspace_kernel<64><<<BH, NTHREADS, bytes, st>>>(C, m, n, k, iters, U, ritz);
    } else {
        cudaError_t e = cudaFuncSetAttribute(sigma_subspace_kernel<128>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)bytes);
        if (e != cudaSuccess) return e;
        sigma_subspace_kernel<128><<<BH, NTHREADS, bytes, st>>>(C, m, n, k, iters, U, ritz);
    }
    return cudaGetLastError();
}

cudaError_t launch_alignment(const float *U, const void *X, bool bf16, int BH, int dk, int k,
                             int nx, float *align, cudaStream_t st) {
    using namespace subspace;
    const long long warps = (long long)BH * nx;
    const unsigned blocks = (unsigned)((warps * 32 + NTHREADS - 1) / NTHREADS);
    if (bf16)
        alignment_kernel<__nv_bfloat16><<<blocks, NTHREADS, 0, st>>>(
            U, static_cast<const __nv_bfloat16 *>(X), dk, k, nx, BH, align);
    else
        alignment_kernel<float><<<blocks, NTHREADS, 0, st>>>(U, static_cast<const float *>(X), dk,
                                                              k, nx, BH, align);
    return cudaGetLastError();
}

}  // namespace ccq
