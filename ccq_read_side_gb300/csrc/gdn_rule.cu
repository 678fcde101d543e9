// gdn_rule.cu -- second pass of the tensor-core Gated DeltaNet forward: the
// gated delta rule itself, reading the cleaned query qc that the first pass
// (tc_gla.cu, cleaned-query mode) wrote into the output tensor, and
// overwriting it with o.
//
// The Gated DeltaNet write (gist.science summary of 2606.01294, section 2,
// "integration": the backbone's own update), in d_k x d_v form,
//     S_t = alpha_t (S_{t-1} - beta_t k_t (k_t^T S_{t-1})) + beta_t k_t v_t^T,
// treats every column of S independently: column j only ever meets v_{t,j}
// and o_{t,j} = S_t[:, j] . qc_t.  So the d_v columns are split over a
// cluster of NC CTAs per (b, h), each keeping its dk x (dv / NC) slice of S
// in shared memory for the whole sequence.  Per chunk of L tokens (scalar
// cumulative log-decay g, Gam_il = exp(g_i - g_l)), the chunk form
//     Aw = strict_tril(beta_i Gam_il k_i . k_l),  Ag = tril(Gam_il qc_i . k_l)
//     U  = (I + Aw)^-1 (beta V - beta exp(g) (K S0))
//     O  = exp(g) (Qc S0) + Ag U
//     S <- exp(g_L) S0 + (K exp(g_L - g))^T U
// is evaluated for the CTA's columns; the L x L matrices are computed by
// every CTA of the cluster (they do not depend on S).
//
// qc and o share the output tensor: a cluster barrier after each chunk's
// loads guarantees that every CTA has read the chunk's qc rows before any CTA
// overwrites them with o.
#include <cuda_bf16.h>

#include "common.cuh"
#include "sm103.cuh"

namespace ccq {
namespace gdnrule {

constexpr int NC = 8;          // CTAs per (b, h)
constexpr int L = 16;          // tokens per chunk
constexpr int NTHREADS = 256;

template <typename TIn, int DK, int DV>
__global__ void __cluster_dims__(NC, 1, 1) __launch_bounds__(NTHREADS)
gdn_rule_kernel(const __grid_constant__ CcqParams p) {
    constexpr int W = DV / NC;  // columns of S in this CTA
    static_assert(L * L == NTHREADS, "one thread per (i, l) of the chunk's L x L matrices");
    static_assert(L * W <= NTHREADS, "one thread per (i, j) of the chunk's L x W tiles");
    __shared__ float sS[DK][W];
    __shared__ float sK[L][DK + 1], sQ[L][DK + 1];  // +1: conflict-free row-wise dots
    __shared__ float sV[L][W], sX[L][W], sU[L][W], sQS[L][W];
    __shared__ float sAw[L][L], sAg[L][L];
    __shared__ float sLa[L], sBeta[L], sG[L], sE[L], sD[L];

    const int tid = threadIdx.x;
    const uint32_t rank = sm103::cluster_ctarank();
    const int bh = blockIdx.x / NC;
    const int j0 = (int)rank * W;
    const int T = p.T;
    const TIn *gk = static_cast<const TIn *>(p.k) + (size_t)bh * T * DK;
    const TIn *gv = static_cast<const TIn *>(p.v) + (size_t)bh * T * DV;
    const TIn *gla = static_cast<const TIn *>(p.log_alpha) + (size_t)bh * T;
    const TIn *gbeta = static_cast<const TIn *>(p.beta) + (size_t)bh * T;
    TIn *go = static_cast<TIn *>(p.o) + (size_t)bh * T * DV;  // qc in, o out (DV == DK)

    for (int x = tid; x < DK * W; x += NTHREADS) {
        const int c = x / W, j = x % W;
        sS[c][j] = p.S0 ? p.S0[((size_t)bh * DK + c) * DV + j0 + j] : 0.f;
    }

    for (int c0 = 0; c0 < T; c0 += L) {
        const int Lc = min(L, T - c0);
        // ---- the chunk: K, qc (zero past the tail), this CTA's columns of V
        for (int x = tid; x < L * DK; x += NTHREADS) {
            const int i = x / DK, c = x % DK;
            const bool ok = i < Lc;
            sK[i][c] = ok ? io<TIn>::load(gk + (size_t)(c0 + i) * DK + c) : 0.f;
            sQ[i][c] = ok ? io<TIn>::load(go + (size_t)(c0 + i) * DV + c) : 0.f;
        }
        if (tid < L * W) {
            const int i = tid / W, j = tid % W;
            sV[i][j] = i < Lc ? io<TIn>::load(gv + (size_t)(c0 + i) * DV + j0 + j) : 0.f;
        }
        if (tid < L) {
            const bool ok = tid < Lc;
            sLa[tid] = ok ? io<TIn>::load(gla + c0 + tid) : 0.f;
            sBeta[tid] = ok ? io<TIn>::load(gbeta + c0 + tid) : 0.f;
        }
        __syncthreads();
        // every CTA of the cluster holds this chunk's qc: o may now overwrite it
        sm103::cluster_sync();

        // ---- scalar cumulative log-decay (zero past the tail)
        if (tid < 32) {
            float g = tid < L ? sLa[tid] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, g, o);
                if ((tid & 31) >= o) g += y;
            }
            if (tid < L) sG[tid] = g;
        }
        __syncthreads();
        const float gL = sG[L - 1];
        if (tid < L) {
            sE[tid] = expf(sG[tid]);
            sD[tid] = expf(gL - sG[tid]);
        }
        // ---- Aw_il = beta_i Gam_il k_i.k_l (l < i), Ag_il = Gam_il qc_i.k_l (l <= i)
        {
            const int i = tid / L, l = tid % L;
            float aw = 0.f, ag = 0.f;
            if (i < Lc && l <= i) {
                float kk = 0.f, qk = 0.f;
#pragma unroll 8
                for (int d = 0; d < DK; ++d) {
                    const float kl = sK[l][d];
                    kk += sK[i][d] * kl;
                    qk += sQ[i][d] * kl;
                }
                const float gam = expf(sG[i] - sG[l]);
                ag = gam * qk;
                if (l < i) aw = sBeta[i] * gam * kk;
            }
            sAw[i][l] = aw;
            sAg[i][l] = ag;
        }
        // ---- X = beta V - beta exp(g) (K S0);  QS = Qc S0  (this CTA's columns)
        if (tid < L * W) {
            const int i = tid / W, j = tid % W;
            float ks = 0.f, qs = 0.f;
#pragma unroll 8
            for (int c = 0; c < DK; ++c) {
                const float s = sS[c][j];
                ks += sK[i][c] * s;
                qs += sQ[i][c] * s;
            }
            sQS[i][j] = qs;
            sX[i][j] = sBeta[i] * (sV[i][j] - expf(sG[i]) * ks);
        }
        __syncthreads();
        // ---- U = (I + Aw)^-1 X, forward substitution down each column
        if (tid < W) {
            const int j = tid;
            for (int i = 0; i < L; ++i) {
                float u = sX[i][j];
                for (int l = 0; l < i; ++l) u -= sAw[i][l] * sU[l][j];
                sU[i][j] = u;
            }
        }
        __syncthreads();
        // ---- O = exp(g) QS + Ag U
        if (tid < L * W) {
            const int i = tid / W, j = tid % W;
            if (i < Lc) {
                float a = sE[i] * sQS[i][j];
                for (int l = 0; l <= i; ++l) a += sAg[i][l] * sU[l][j];
                io<TIn>::store(go + (size_t)(c0 + i) * DV + j0 + j, a);
            }
        }
        // ---- S <- exp(g_L) S + (K exp(g_L - g))^T U
        const float egL = expf(gL);
        for (int x = tid; x < DK * W; x += NTHREADS) {
            const int c = x / W, j = x % W;
            float a = egL * sS[c][j];
#pragma unroll
            for (int i = 0; i < L; ++i) a += sK[i][c] * sD[i] * sU[i][j];
            sS[c][j] = a;
        }
        __syncthreads();
    }
    if (p.S_out)
        for (int x = tid; x < DK * W; x += NTHREADS) {
            const int c = x / W, j = x % W;
            p.S_out[((size_t)bh * DK + c) * DV + j0 + j] = sS[c][j];
        }
}

}  // namespace gdnrule

// Second pass (after launch_tc_qclean): dk = dv = 128, bf16.
cudaError_t launch_gdn_rule(const CcqParams &p, cudaStream_t st) {
    using namespace gdnrule;
    if (p.B * p.H == 0 || p.T == 0) return cudaSuccess;
    gdn_rule_kernel<__nv_bfloat16, 128, 128><<<p.B * p.H * NC, NTHREADS, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ccq
