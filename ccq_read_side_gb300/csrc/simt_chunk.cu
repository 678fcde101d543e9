// simt_chunk.cu -- fp32 CUDA-core chunked CCQ forward (GLA and Gated DeltaNet).
//
// One CTA per (b, h); the carried state S (dk x dv), C (dk x dk), m (dk) and
// the token count live in shared memory in fp32 for the whole sequence.  The
// sequence is walked in chunks of up to 16 tokens.  Per chunk, with t_i the
// number of tokens seen after token i of the chunk:
//
//   CCQ read (Sigma_t q of the gist.science summary of 2606.01294, section 2,
//   written over a chunk):
//     A_ij = q_i . k_j (j <= i);   s_i = m0 . q_i + sum_{j<=i} A_ij  (= m_t . q_i)
//     P_i  = C0 q_i + sum_{j<=i} (A_ij - s_i/t_i) k_j - (s_i/t_i) m0  (= t_i Sigma_t q_i)
//     qc_i = q_i - (lambda_i / t_i) P_i
//   GLA write + read, per-channel cumulative log-decay Bc, R = Bc at the
//   chunk's last token:
//     Qt = qc * exp(Bc - R), Kh = K * exp(R - Bc), Sb = diag(exp R) S0
//     O = tril(Qt Kh^T) V + Qt Sb;   S <- Sb + Kh^T V
//   Gated DeltaNet (scalar cumulative log-decay g, Gam_ij = exp(g_i - g_j)):
//     U = (I + strict_tril(beta_i Gam_ij k_i.k_j))^-1 (beta V - beta exp(g) K S0)
//     O = exp(g) (Qc S0) + tril(Gam * Qc K^T) U
//     S <- exp(g_L) S0 + (K * exp(g_L - g))^T U
//   statistics: C += K^T K, m += sum K, n += tokens in the chunk.
//
// This is the fp32 kernel for fp32 inputs (and for any shape the tensor-core
// kernel does not take).  Its arithmetic is fp32 throughout.
#include <algorithm>

#include "common.cuh"

namespace ccq {

constexpr int SIMT_LMAX = 16;
constexpr int SIMT_THREADS = 256;

template <int DK, int DV, bool GDN>
struct SimtSmem {
    static constexpr int L = SIMT_LMAX;
    static constexpr int S = 0;                       // [DK][DV]
    static constexpr int C = S + DK * DV;             // [DK][DK] (symmetric)
    static constexpr int M = C + DK * DK;             // [DK]
    static constexpr int Q = M + DK;                  // [L][DK]
    static constexpr int K = Q + L * DK;              // [L][DK]
    static constexpr int V = K + L * DK;              // [L][DV]
    static constexpr int LA = V + L * DV;             // GLA [L][DK]; GDN la[L], beta[L], g[L]
    static constexpr int A = LA + (GDN ? 3 * L : L * DK);  // [L][L]
    static constexpr int QT = A + L * L;              // [L][DK]: qc, then (GLA) Qt
    static constexpr int X = QT + L * DK;             // GLA: KhT [DK][L]; GDN: X [L][DV]
    static constexpr int U = X + (GDN ? L * DV : DK * L);  // GDN: U [L][DV]; GLA: unused
    static constexpr int QS = U + (GDN ? L * DV : 0);  // GDN: Qc S0 [L][DV]
    static constexpr int AG = QS + (GDN ? L * DV : 0); // [L][L]
    static constexpr int AW = AG + L * L;             // GDN [L][L]
    static constexpr int GAM = AW + L * L;            // GLA: exp(R) [DK]
    static constexpr int TOK = GAM + DK;              // per-token scalars: s/t, lambda/t, eg, kd
    static constexpr int TOTAL = TOK + 4 * L;
    static constexpr size_t BYTES = sizeof(float) * TOTAL;
};

template <typename TIn, int DK, int DV, bool GDN>
__global__ void __launch_bounds__(SIMT_THREADS)
simt_chunk_kernel(CcqParams p) {
    using SM = SimtSmem<DK, DV, GDN>;
    constexpr int L = SM::L;
    extern __shared__ float smem[];
    float *sS = smem + SM::S, *sC = smem + SM::C, *sM = smem + SM::M;
    float *sQ = smem + SM::Q, *sK = smem + SM::K, *sV = smem + SM::V, *sLA = smem + SM::LA;
    float *sA = smem + SM::A, *sQt = smem + SM::QT, *sX = smem + SM::X, *sU = smem + SM::U;
    float *sQS = smem + SM::QS, *sAg = smem + SM::AG, *sAw = smem + SM::AW;
    float *sGam = smem + SM::GAM, *sTok = smem + SM::TOK;
    float *tok_s = sTok, *tok_a = sTok + L, *tok_e = sTok + 2 * L, *tok_d = sTok + 3 * L;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bh = blockIdx.x, h = bh % p.H;
    const int T = p.T;
    const int Lc_max = (p.chunk > 0 && p.chunk < L) ? p.chunk : L;
    const bool l2n = (p.flags & CCQ_FLAG_L2NORM_QK) != 0;

    const TIn *gq = reinterpret_cast<const TIn *>(p.q) + (size_t)bh * T * DK;
    const TIn *gk = reinterpret_cast<const TIn *>(p.k) + (size_t)bh * T * DK;
    const TIn *gv = reinterpret_cast<const TIn *>(p.v) + (size_t)bh * T * DV;
    const TIn *gla = reinterpret_cast<const TIn *>(p.log_alpha) + (size_t)bh * T * (GDN ? 1 : DK);
    const TIn *gbeta = GDN ? reinterpret_cast<const TIn *>(p.beta) + (size_t)bh * T : nullptr;
    TIn *go = reinterpret_cast<TIn *>(p.o) + (size_t)bh * T * DV;

    // ---- carried state
    for (int x = tid; x < DK * DV; x += SIMT_THREADS)
        sS[x] = p.S0 ? p.S0[(size_t)bh * DK * DV + x] : 0.f;
    for (int x = tid; x < DK * DK; x += SIMT_THREADS)
        sC[x] = p.C0 ? p.C0[(size_t)bh * DK * DK + x] : 0.f;
    for (int x = tid; x < DK; x += SIMT_THREADS) sM[x] = p.m0 ? p.m0[(size_t)bh * DK + x] : 0.f;
    double n = (double)p.t0;  // exact token count (identical in every thread)
    const float bl = p.lambda_in ? 0.f : p.b_lambda[h];
    const float *wl = p.lambda_in ? nullptr : p.w_lambda + (size_t)h * DK;
    __syncthreads();

    for (int c0 = 0; c0 < T; c0 += Lc_max) {
        const int Lc = min(Lc_max, T - c0);
        // ---- load the chunk (zero padding past Lc)
        for (int x = tid; x < L * DK; x += SIMT_THREADS) {
            int i = x / DK, c = x % DK;
            bool ok = i < Lc;
            sQ[x] = ok ? io<TIn>::load(gq + (size_t)(c0 + i) * DK + c) : 0.f;
            sK[x] = ok ? io<TIn>::load(gk + (size_t)(c0 + i) * DK + c) : 0.f;
            if (!GDN) sLA[x] = ok ? io<TIn>::load(gla + (size_t)(c0 + i) * DK + c) : 0.f;
        }
        for (int x = tid; x < L * DV; x += SIMT_THREADS) {
            int i = x / DV, c = x % DV;
            sV[x] = i < Lc ? io<TIn>::load(gv + (size_t)(c0 + i) * DV + c) : 0.f;
        }
        if (GDN && tid < L) {
            bool ok = tid < Lc;
            sLA[tid] = ok ? io<TIn>::load(gla + c0 + tid) : 0.f;
            sLA[L + tid] = ok ? io<TIn>::load(gbeta + c0 + tid) : 0.f;
        }
        __syncthreads();
        if (l2n) {  // warp per row: x / sqrt(|x|^2 + 1e-6)
            for (int r = warp; r < 2 * L; r += SIMT_THREADS / 32) {
                float *row = (r < L ? sQ : sK) + (r % L) * DK;
                float ss = 0.f;
                for (int c = lane; c < DK; c += 32) ss += row[c] * row[c];
                ss = warp_sum(ss);
                float sc = 1.0f / sqrtf(ss + 1e-6f);
                for (int c = lane; c < DK; c += 32) row[c] *= sc;
            }
            __syncthreads();
        }

        // ---- A_ij = q_i . k_j (j <= i)
        {
            int i = tid / L, j = tid % L;
            float a = 0.f;
            if (i < Lc && j <= i) {
                const float *qi = sQ + i * DK, *kj = sK + j * DK;
#pragma unroll 8
                for (int dd = 0; dd < DK; ++dd) {
                    int d = (dd + j) & (DK - 1);
                    a += qi[d] * kj[d];
                }
            }
            sA[tid] = a;
        }
        __syncthreads();

        // ---- per-token scalars: s_i / t_i, lambda_i / t_i
        for (int i = warp; i < Lc; i += SIMT_THREADS / 32) {
            float mq = 0.f, wq = 0.f;
            for (int c = lane; c < DK; c += 32) {
                float qv = sQ[i * DK + c];
                mq += sM[c] * qv;
                if (wl) wq += wl[c] * qv;
            }
            mq = warp_sum(mq);
            wq = warp_sum(wq);
            if (lane == 0) {
                float rs = 0.f;
                for (int j = 0; j <= i; ++j) rs += sA[i * L + j];
                float t = (float)(n + (double)(i + 1));
                float lam = p.lambda_in ? p.lambda_in[(size_t)bh * T + c0 + i]
                                        : 1.0f / (1.0f + expf(-(wq + bl)));
                if (p.lambda_out) p.lambda_out[(size_t)bh * T + c0 + i] = lam;
                tok_s[i] = (mq + rs) / t;
                tok_a[i] = lam / t;
            }
        }
        __syncthreads();

        // ---- P and qc: thread = channel c, tokens ig, ig + G, ...
        {
            constexpr int G = SIMT_THREADS / DK;
            constexpr int NT = L / G;
            const int c = tid % DK, ig = tid / DK;
            float acc[NT];
#pragma unroll
            for (int u = 0; u < NT; ++u) acc[u] = 0.f;
            for (int d = 0; d < DK; ++d) {
                float cdc = sC[d * DK + c];  // = C[c][d] (symmetric)
#pragma unroll
                for (int u = 0; u < NT; ++u) acc[u] += cdc * sQ[(ig + u * G) * DK + d];
            }
#pragma unroll
            for (int u = 0; u < NT; ++u) {
                int i = ig + u * G;
                if (i < Lc) {
                    float si = tok_s[i];
                    float a = acc[u];
                    for (int j = 0; j <= i; ++j) a += (sA[i * L + j] - si) * sK[j * DK + c];
                    a -= si * sM[c];
                    sQt[i * DK + c] = sQ[i * DK + c] - tok_a[i] * a;
                } else {
                    sQt[i * DK + c] = 0.f;
                }
            }
        }
        __syncthreads();

        if (!GDN) {
            // ---- per-channel decay: Qt = qc exp(Bc - R), Kh = K exp(R - Bc), gamma = exp(R)
            if (tid < DK) {
                const int c = tid;
                float R = 0.f;
                for (int i = 0; i < Lc; ++i) R += sLA[i * DK + c];
                float Bc = 0.f;
                for (int i = 0; i < L; ++i) {
                    if (i < Lc) {
                        Bc += sLA[i * DK + c];
                        sQt[i * DK + c] *= expf(Bc - R);
                        sX[c * L + i] = sK[i * DK + c] * expf(R - Bc);
                    } else {
                        sX[c * L + i] = 0.f;
                    }
                }
                sGam[c] = expf(R);
            }
            __syncthreads();
            // ---- Ag_ij = Qt_i . Kh_j (j <= i)
            {
                int i = tid / L, j = tid % L;
                float a = 0.f;
                if (i < Lc && j <= i) {
                    for (int c = 0; c < DK; ++c) a += sQt[i * DK + c] * sX[c * L + j];
                }
                sAg[tid] = a;
            }
            __syncthreads();
            // ---- O = tril(Ag) V + Qt (gamma S0)
            {
                constexpr int G = SIMT_THREADS / DV;
                constexpr int NT = L / G;
                const int jv = tid % DV, ig = tid / DV;
                float acc[NT];
#pragma unroll
                for (int u = 0; u < NT; ++u) acc[u] = 0.f;
                for (int c = 0; c < DK; ++c) {
                    float s = sS[c * DV + jv] * sGam[c];
#pragma unroll
                    for (int u = 0; u < NT; ++u) acc[u] += sQt[(ig + u * G) * DK + c] * s;
                }
#pragma unroll
                for (int u = 0; u < NT; ++u) {
                    int i = ig + u * G;
                    if (i < Lc) {
                        float a = acc[u];
                        for (int l = 0; l <= i; ++l) a += sAg[i * L + l] * sV[l * DV + jv];
                        io<TIn>::store(go + (size_t)(c0 + i) * DV + jv, a);
                    }
                }
            }
            __syncthreads();
            // ---- S <- gamma S + Kh^T V
            for (int x = tid; x < DK * DV; x += SIMT_THREADS) {
                int c = x / DV, jv = x % DV;
                float a = sGam[c] * sS[x];
#pragma unroll
                for (int i = 0; i < L; ++i) a += sX[c * L + i] * sV[i * DV + jv];
                sS[x] = a;
            }
        } else {
            // ---- scalar cumulative log-decay
            float *sLa = sLA, *sBeta = sLA + L, *sG = sLA + 2 * L;
            if (tid == 0) {
                float g = 0.f;
                for (int i = 0; i < L; ++i) {
                    g += sLa[i];  // zero past Lc
                    sG[i] = g;
                }
            }
            __syncthreads();
            const float gL = sG[L - 1];
            if (tid < L) {
                tok_e[tid] = expf(sG[tid]);
                tok_d[tid] = expf(gL - sG[tid]);
            }
            // ---- Aw_il = beta_i Gam_il k_i.k_l (l < i), Ag_il = Gam_il qc_i.k_l (l <= i)
            {
                int i = tid / L, l = tid % L;
                float aw = 0.f, ag = 0.f;
                if (i < Lc && l <= i) {
                    float kk = 0.f, qk = 0.f;
                    for (int dd = 0; dd < DK; ++dd) {
                        int d = (dd + l) & (DK - 1);
                        float kl = sK[l * DK + d];
                        kk += sK[i * DK + d] * kl;
                        qk += sQt[i * DK + d] * kl;
                    }
                    float gam = expf(sG[i] - sG[l]);
                    ag = gam * qk;
                    if (l < i) aw = sBeta[i] * gam * kk;
                }
                sAw[tid] = aw;
                sAg[tid] = ag;
            }
            __syncthreads();
            // ---- X = beta V - beta exp(g) (K S0);  QS = Qc S0
            {
                constexpr int G = SIMT_THREADS / DV;
                constexpr int NT = L / G;
                const int jv = tid % DV, ig = tid / DV;
                float ks[NT], qs[NT];
#pragma unroll
                for (int u = 0; u < NT; ++u) ks[u] = qs[u] = 0.f;
                for (int c = 0; c < DK; ++c) {
                    float s = sS[c * DV + jv];
#pragma unroll
                    for (int u = 0; u < NT; ++u) {
                        int i = ig + u * G;
                        ks[u] += sK[i * DK + c] * s;
                        qs[u] += sQt[i * DK + c] * s;
                    }
                }
#pragma unroll
                for (int u = 0; u < NT; ++u) {
                    int i = ig + u * G;
                    float b = sBeta[i];
                    sX[i * DV + jv] = b * sV[i * DV + jv] - b * tok_e[i] * ks[u];
                    sQS[i * DV + jv] = qs[u];
                }
            }
            __syncthreads();
            // ---- U = (I + Aw)^-1 X by forward substitution (column jv per thread)
            for (int jv = tid; jv < DV; jv += SIMT_THREADS) {
                for (int i = 0; i < L; ++i) {
                    float u = sX[i * DV + jv];
                    for (int l = 0; l < i; ++l) u -= sAw[i * L + l] * sU[l * DV + jv];
                    sU[i * DV + jv] = u;
                }
            }
            __syncthreads();
            // ---- O = exp(g) QS + tril(Ag) U
            for (int x = tid; x < Lc * DV; x += SIMT_THREADS) {
                int i = x / DV, jv = x % DV;
                float a = tok_e[i] * sQS[x];
                for (int l = 0; l <= i; ++l) a += sAg[i * L + l] * sU[l * DV + jv];
                io<TIn>::store(go + (size_t)(c0 + i) * DV + jv, a);
            }
            // ---- S <- exp(g_L) S + (K exp(g_L - g))^T U
            const float egL = expf(gL);
            for (int x = tid; x < DK * DV; x += SIMT_THREADS) {
                int c = x / DV, jv = x % DV;
                float a = egL * sS[x];
#pragma unroll
                for (int i = 0; i < L; ++i) a += sK[i * DK + c] * tok_d[i] * sU[i * DV + jv];
                sS[x] = a;
            }
        }
        // ---- C += K^T K, m += sum K
        for (int x = tid; x < DK * DK; x += SIMT_THREADS) {
            int c = x / DK, d = x % DK;
            float a = sC[x];
#pragma unroll
            for (int i = 0; i < L; ++i) a += sK[i * DK + c] * sK[i * DK + d];
            sC[x] = a;
        }
        if (tid < DK) {
            float a = sM[tid];
            for (int i = 0; i < L; ++i) a += sK[i * DK + tid];
            sM[tid] = a;
        }
        n += (double)Lc;
        __syncthreads();
    }

    if (p.S_out)
        for (int x = tid; x < DK * DV; x += SIMT_THREADS) p.S_out[(size_t)bh * DK * DV + x] = sS[x];
    if (p.C_out)
        for (int x = tid; x < DK * DK; x += SIMT_THREADS) p.C_out[(size_t)bh * DK * DK + x] = sC[x];
    if (p.m_out)
        for (int x = tid; x < DK; x += SIMT_THREADS) p.m_out[(size_t)bh * DK + x] = sM[x];
}

template <typename TIn, int DK, int DV, bool GDN>
static cudaError_t launch_one(const CcqParams &p, cudaStream_t st) {
    using SM = SimtSmem<DK, DV, GDN>;
    auto fn = simt_chunk_kernel<TIn, DK, DV, GDN>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SM::BYTES);
    if (e != cudaSuccess) return e;
    fn<<<p.B * p.H, SIMT_THREADS, SM::BYTES, st>>>(p);
    return cudaGetLastError();
}

template <typename TIn, bool GDN>
static cudaError_t launch_dims(const CcqParams &p, cudaStream_t st) {
    if (p.dk == 64 && p.dv == 64) return launch_one<TIn, 64, 64, GDN>(p, st);
    if (p.dk == 64 && p.dv == 128) return launch_one<TIn, 64, 128, GDN>(p, st);
    if (p.dk == 128 && p.dv == 64) return launch_one<TIn, 128, 64, GDN>(p, st);
    return launch_one<TIn, 128, 128, GDN>(p, st);
}

cudaError_t launch_simt(const CcqParams &p, bool gdn, bool bf16, cudaStream_t st) {
    if (p.B * p.H == 0) return cudaSuccess;
    if (bf16) return gdn ? launch_dims<__nv_bfloat16, true>(p, st)
                         : launch_dims<__nv_bfloat16, false>(p, st);
    return gdn ? launch_dims<float, true>(p, st) : launch_dims<float, false>(p, st);
}

}  // namespace ccq
