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
// cluster of NC CTAs per (b, h), each keeping its dk x W slice of S (W =
// dv / NC = 16) for the whole sequence.  Per chunk of L = 16 tokens (scalar
// cumulative log-decay g, Gam_il = exp(g_i - g_l)), the chunk form
//     Aw = strict_tril(beta_i Gam_il k_i . k_l),  Ag = tril(Gam_il qc_i . k_l)
//     U  = (I + Aw)^-1 (beta V - beta exp(g) (K S0))
//     O  = exp(g) (Qc S0) + Ag U
//     S <- exp(g_L) S0 + (K exp(g_L - g))^T U
// is evaluated for the CTA's columns.  The four 16 x 16 x 128 products (K K^T,
// Qc K^T, K S0, Qc S0) and the state update (128 x 16 x 16) run on the
// tensor cores through warp-level mma.sync (bf16 operands, fp32
// accumulation); the state slice itself stays in fp32 registers (one 16-row
// band per warp) for the whole sequence, and a bf16 copy in shared memory
// feeds the next chunk's products.  The unit-lower-triangular solve for U is a
// register-resident forward substitution, one lane per column.  Each chunk's
// inputs are loaded into registers while the previous chunk computes.
//
// qc and o share the output tensor: a cluster barrier per chunk (arrive once
// the chunk's qc is in shared memory, wait before the first o store)
// guarantees that every CTA has read it before any CTA overwrites it with o.
#include <cuda_bf16.h>

#include "common.cuh"
#include "sm103.cuh"

namespace ccq {
namespace gdnrule {

constexpr int NC = 8;          // CTAs per (b, h)
constexpr int L = 16;          // tokens per chunk
constexpr int DK = 128, DV = 128;
constexpr int W = DV / NC;     // columns of S per CTA (16)
constexpr int NTHREADS = 256;  // 8 warps: warp w owns rows [16w, 16w+16) of the S slice
// Shared rows are padded by 16 bytes: 256-byte rows would put the eight rows
// an mma fragment reads in the same banks.
constexpr int DKP = DK + 8;

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float bf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// D += A B for one m16n8k16 tile: A 16 x 16 (row-major fragment), B 16 x 8.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

struct Smem {
    __nv_bfloat16 K[L][DKP];     // chunk tiles (rows padded)
    __nv_bfloat16 Q[L][DKP];     // qc
    __nv_bfloat16 St[W][DKP];    // bf16 copy of the S slice, transposed ([column][row])
    __nv_bfloat16 Ut[W][L];      // bf16 U, transposed
    float V[L][W];
    // per-token scalars, by chunk parity: beta, g, exp(g), exp(-g), exp(g_L - g)
    float beta[2][L], G[2][L], E[2][L], EI[2][L], Dd[2][L];
    __align__(16) float AwT[L][L];                 // Aw transposed: [column][row]
    float Ag[L][L];
    float X[L][W], QS[L][W], U[L][W];
};

// One chunk's inputs as loaded by one thread: 16 bytes of a K row and of a qc
// row (row tid / 16, part tid % 16), one V element, and (tid < 16) log alpha
// and beta of one token.  Loads past the tail read the last valid token
// instead (always in bounds) and are zeroed only when stored, a chunk later:
// selecting on a loaded value would make the thread wait for the load.
struct Chunk {
    uint4 k, q;
    __nv_bfloat16 v, la, beta;
};

__global__ void __cluster_dims__(NC, 1, 1) __launch_bounds__(NTHREADS)
gdn_rule_kernel(const __grid_constant__ CcqParams p) {
    __shared__ __align__(128) Smem sm;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, t4 = lane & 3;  // mma fragment coordinates
    const uint32_t rank = sm103::cluster_ctarank();
    const int bh = blockIdx.x / NC;
    const int j0 = (int)rank * W;
    const int T = p.T;
    const int nch = (T + L - 1) / L;
    const __nv_bfloat16 *gk = static_cast<const __nv_bfloat16 *>(p.k) + (size_t)bh * T * DK;
    const __nv_bfloat16 *gv = static_cast<const __nv_bfloat16 *>(p.v) + (size_t)bh * T * DV;
    const __nv_bfloat16 *gla = static_cast<const __nv_bfloat16 *>(p.log_alpha) + (size_t)bh * T;
    const __nv_bfloat16 *gbeta = static_cast<const __nv_bfloat16 *>(p.beta) + (size_t)bh * T;
    __nv_bfloat16 *go = static_cast<__nv_bfloat16 *>(p.o) + (size_t)bh * T * DV;

    auto fetch = [&](int c) {
        const int last = T - 1 - c * L;  // last valid row of the chunk
        const int r = min(tid >> 4, last), part = tid & 15;
        const size_t row = (size_t)c * L + r;
        Chunk x;
        x.k = *reinterpret_cast<const uint4 *>(gk + row * DK + 8 * part);
        x.q = *reinterpret_cast<const uint4 *>(go + row * DV + 8 * part);
        const int i = min(tid / W, last), j = tid % W, t = min(lane & (L - 1), last);
        x.v = gv[(size_t)(c * L + i) * DV + j0 + j];
        x.la = gla[c * L + t];
        x.beta = gbeta[c * L + t];
        return x;
    };
    // warp 1 (which holds chunk c's log alphas) forms the cumulative
    // log-decay g, exp(+-g), exp(g_L - g) and beta into the chunk's parity slot
    // (|g| over a chunk stays far from the fp32 exponent range, so
    // Gam_il = exp(g_i) exp(-g_l) is formed by one product)
    auto scan = [&](const Chunk &x, int c) {
        const int lc = min(L, T - c * L), pb = c & 1;
        float g = (lane < L && lane < lc) ? __bfloat162float(x.la) : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, g, o);
            if (lane >= o) g += y;
        }
        const float gL = __shfl_sync(0xffffffffu, g, L - 1);
        if (lane < L) {
            sm.beta[pb][lane] = lane < lc ? __bfloat162float(x.beta) : 0.f;
            sm.G[pb][lane] = g;
            sm.E[pb][lane] = expf(g);
            sm.EI[pb][lane] = expf(-g);
            sm.Dd[pb][lane] = expf(gL - g);
        }
    };
    // stores a fetched chunk's tiles
    auto store = [&](const Chunk &x, int c) {
        const int lc = min(L, T - c * L);
        const int r = tid >> 4, part = tid & 15;
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(&sm.K[r][8 * part]) = r < lc ? x.k : z;
        *reinterpret_cast<uint4 *>(&sm.Q[r][8 * part]) = r < lc ? x.q : z;
        sm.V[tid / W][tid % W] = tid / W < lc ? __bfloat162float(x.v) : 0.f;
    };

    // ---- S slice: warp w holds rows [16w, 16w+16) x 16 columns as two m16n8
    // accumulator tiles; its bf16 transposed copy feeds K S0 and Qc S0
    float sacc[2][4];
    {
        const int r0 = 16 * warp;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = r0 + g4 + 8 * (e >> 1), j = 8 * nt + 2 * t4 + (e & 1);
                sacc[nt][e] = p.S0 ? p.S0[((size_t)bh * DK + r) * DV + j0 + j] : 0.f;
                sm.St[j][r] = __float2bfloat16_rn(sacc[nt][e]);
            }
    }
    if (nch > 0) {
        const Chunk x0 = fetch(0);
        store(x0, 0);
        if (warp == 1) scan(x0, 0);
    }
    __syncthreads();
    // this CTA holds chunk 0's qc; o may overwrite a chunk's qc once every CTA
    // of the cluster has said so (each wait sits just before the chunk's first
    // o store; an arrive follows the loads, so it is relaxed)
    if (nch > 0) sm103::cluster_arrive_relaxed();

    for (int c = 0; c < nch; ++c) {
        const int c0 = c * L, lc = min(L, T - c0);
        // next chunk's inputs: in flight while this chunk computes
        Chunk nxt{};
        if (c + 1 < nch) nxt = fetch(c + 1);

        const int pb = c & 1;  // parity slot of this chunk's per-token scalars
        const float gL = sm.G[pb][L - 1];

        // ---- four 16 x 8 tiles per product over k = 128: warp (prod, nt)
        {
            const int prod = warp >> 1, nt = warp & 1;  // 0 KK^T, 1 QK^T, 2 K S0, 3 Q S0
            const __nv_bfloat16(*A)[DKP] = (prod == 1 || prod == 3) ? sm.Q : sm.K;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < DK / 16; ++ks) {
                const int k0 = 16 * ks + 2 * t4;
                uint32_t a[4], bb[2];
                a[0] = *reinterpret_cast<const uint32_t *>(&A[g4][k0]);
                a[1] = *reinterpret_cast<const uint32_t *>(&A[g4 + 8][k0]);
                a[2] = *reinterpret_cast<const uint32_t *>(&A[g4][k0 + 8]);
                a[3] = *reinterpret_cast<const uint32_t *>(&A[g4 + 8][k0 + 8]);
                const int n = 8 * nt + g4;
                const __nv_bfloat16 *brow = prod < 2 ? &sm.K[n][0] : &sm.St[n][0];
                bb[0] = *reinterpret_cast<const uint32_t *>(brow + k0);
                bb[1] = *reinterpret_cast<const uint32_t *>(brow + k0 + 8);
                mma16816(d, a, bb);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = g4 + 8 * (e >> 1), n = 8 * nt + 2 * t4 + (e & 1);
                const bool row_ok = i < lc;
                const float gam = sm.E[pb][i] * sm.EI[pb][n];
                if (prod == 0) {
                    sm.AwT[n][i] = (row_ok && n < i) ? sm.beta[pb][i] * gam * d[e] : 0.f;
                } else if (prod == 1) {
                    sm.Ag[i][n] = (row_ok && n <= i) ? gam * d[e] : 0.f;
                } else if (prod == 2) {
                    sm.X[i][n] = row_ok ? sm.beta[pb][i] * (sm.V[i][n] - sm.E[pb][i] * d[e]) : 0.f;
                } else {
                    sm.QS[i][n] = d[e];
                }
            }
        }
        __syncthreads();

        // ---- U = (I + Aw)^-1 X: lane j of warp 0 owns column j; right-looking
        // elimination (once u_l is final, every later row subtracts its share:
        // independent updates, so the dependent depth is one FMA per row)
        if (warp == 0 && lane < W) {
            const int j = lane;
            float u[L];
#pragma unroll
            for (int i = 0; i < L; ++i) u[i] = sm.X[i][j];
#pragma unroll
            for (int l = 0; l < L - 1; ++l) {
                float a[L];  // column l of Aw (same address in every lane)
#pragma unroll
                for (int q = (l + 1) / 4; q < L / 4; ++q) {
                    const float4 f = reinterpret_cast<const float4 *>(&sm.AwT[l][0])[q];
                    a[4 * q] = f.x;
                    a[4 * q + 1] = f.y;
                    a[4 * q + 2] = f.z;
                    a[4 * q + 3] = f.w;
                }
#pragma unroll
                for (int i = l + 1; i < L; ++i) u[i] -= a[i] * u[l];
            }
#pragma unroll
            for (int i = 0; i < L; ++i) {
                sm.U[i][j] = u[i];
                sm.Ut[j][i] = __float2bfloat16_rn(u[i]);
            }
        }
        if (warp == 1 && c + 1 < nch) scan(nxt, c + 1);  // next chunk's scalars, meanwhile
        __syncthreads();

        // ---- O = exp(g) QS + Ag U (fp32, one (i, j) per thread)
        sm103::cluster_wait();  // every CTA holds this chunk's qc
        {
            const int i = tid / W, j = tid % W;
            if (i < lc) {
                float a = sm.E[pb][i] * sm.QS[i][j];
#pragma unroll
                for (int l = 0; l < L; ++l) a += sm.Ag[i][l] * sm.U[l][j];
                go[(size_t)(c0 + i) * DV + j0 + j] = __float2bfloat16_rn(a);
            }
        }
        // ---- S <- exp(g_L) S + (K exp(g_L - g))^T U: warp w, rows [16w, 16w+16)
        {
            const float egL = expf(gL);
            const int r0 = 16 * warp;
            uint32_t a[4];
            // A[m][k] = K[k][r0 + m] * d_k  (m: state row, k: token)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int m = g4 + 8 * (q & 1), k = 2 * t4 + 8 * (q >> 1);
                a[q] = pack_bf16(bf(&sm.K[k][r0 + m]) * sm.Dd[pb][k],
                                 bf(&sm.K[k + 1][r0 + m]) * sm.Dd[pb][k + 1]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t bb[2];
                const __nv_bfloat16 *ucol = &sm.Ut[8 * nt + g4][0];
                bb[0] = *reinterpret_cast<const uint32_t *>(ucol + 2 * t4);
                bb[1] = *reinterpret_cast<const uint32_t *>(ucol + 2 * t4 + 8);
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[nt][e] *= egL;
                mma16816(sacc[nt], a, bb);
            }
        }
        __syncthreads();  // this chunk no longer reads K, Q, V, St
        {
            const int r0 = 16 * warp;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = r0 + g4 + 8 * (e >> 1), j = 8 * nt + 2 * t4 + (e & 1);
                    sm.St[j][r] = __float2bfloat16_rn(sacc[nt][e]);
                }
        }
        if (c + 1 < nch) store(nxt, c + 1);
        __syncthreads();
        if (c + 1 < nch) sm103::cluster_arrive_relaxed();  // this CTA holds chunk c+1's qc
    }
    if (p.S_out) {
        const int r0 = 16 * warp;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = r0 + g4 + 8 * (e >> 1), j = 8 * nt + 2 * t4 + (e & 1);
                p.S_out[((size_t)bh * DK + r) * DV + j0 + j] = sacc[nt][e];
            }
    }
    sm103::cluster_sync();  // no CTA leaves while a peer may still be at a barrier
}

}  // namespace gdnrule

// Second pass (after launch_tc_qclean): dk = dv = 128, bf16.
cudaError_t launch_gdn_rule(const CcqParams &p, cudaStream_t st) {
    using namespace gdnrule;
    if (p.B * p.H == 0 || p.T == 0) return cudaSuccess;
    gdn_rule_kernel<<<p.B * p.H * NC, NTHREADS, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ccq
