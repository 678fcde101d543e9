// gla_bwd.cu -- gradients of the CCQ-GLA forward, fp32 on CUDA cores.
//
// Forward being differentiated (10100.com article, "method", item 1;
// gist.science summary of 2606.01294, section 2, "mechanism" and
// "integration"): per head and token
//   S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T,  C_t = C_{t-1} + k_t k_t^T,
//   m_t = m_{t-1} + k_t,  n_t = t0 + t + 1,  mu_t = m_t / n_t,
//   y_t = Sigma_t q_t = C_t q_t / n_t - mu_t (mu_t . q_t),
//   lambda_t = sigmoid(w . q_t + b)  (or given),  qc_t = q_t - lambda_t y_t,
//   o_t = S_t^T qc_t.
//
// Two sweeps over the tokens, one CTA per (b, h) in each:
//
// 1. Forward sweep.  Everything that depends on the forward state can be
//    formed going forward, because the upstream gradient g_t = dL/do_t is
//    known: gqc_t = S_t g_t, glambda_t = -y_t . gqc_t, gy_t = -lambda_t gqc_t,
//    and the query gradient
//      dq_t = gqc_t + Sigma_t gy_t + lambda_t (1 - lambda_t) glambda_t w.
//    C and S stay in registers: thread (x, part) owns row x of C and row x
//    of S, each over one slice of columns, the only elements it ever reads
//    or writes (C is symmetric, so C0 must be too: it is a sum of k k^T).
//    Per token it leaves in the workspace qc_t, gy_t, qc_t * gqc_t and the
//    two scalars (mu.q)/n and (mu.gy)/n that rebuild dL/dmu_t / n_t.
//
// 2. Reverse sweep.  The adjoints of the three sums run backwards:
//      GS_t = qc_t g_t^T + Diag(alpha_{t+1}) GS_{t+1}      (dL/dS_t)
//      GC_t = gy_t q_t^T / n_t + GC_{t+1}                  (dL/dC_t)
//      Gm_t = dL/dmu_t / n_t + Gm_{t+1}                    (dL/dm_t)
//    with dk_t = (GC_t + GC_t^T) k_t + Gm_t + GS_t v_t and dv_t = GS_t^T k_t.
//    GC enters only through GC + GC^T, so that symmetric sum is what is kept
//    (registers, row-owned); GS sits in shared memory with padded rows, read
//    by rows (GS v) and by columns (GS^T k).
//    The decay gradient uses d log A_t = qc_t * gqc_t - k_t * (GS_t v_t)
//    (A_t the running product of alpha; the final state adds
//    rowsum(dL/dS_T * S_T)), summed over t' >= t.
//
// Shapes: dk, dv in {64, 128}; any T (a ragged last chunk); 256 threads.
// Token vectors are staged TL tokens at a time with cp.async (16-byte
// copies, double-buffered) so each chunk's loads overlap the previous chunk.
#include <mutex>

#include "common.cuh"

namespace ccq {

namespace bwd {

constexpr int NT = 256;
constexpr int TL = 8;  // tokens per staged chunk

__device__ __forceinline__ void cp16(float *dst, const float *src) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all() {
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}
// n floats (n % 4 == 0; both ends 16-byte aligned), spread over the CTA
__device__ __forceinline__ void stage(float *dst, const float *src, int n) {
    for (int i = threadIdx.x * 4; i < n; i += NT * 4) cp16(dst + i, src + i);
}
__device__ __forceinline__ float4 ld4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}

struct Ws {
    float *qc, *gy, *t1, *sc, *rs;
    __device__ Ws(const BwdParams &p, int dk) {
        const size_t n = (size_t)p.BH * p.T;
        qc = p.ws;
        gy = qc + n * dk;
        t1 = gy + n * dk;
        sc = t1 + n * dk;
        rs = sc + n * 4;
    }
};

template <int DK, int DV>
__global__ void __launch_bounds__(NT, 1) fwd_sweep_kernel(const BwdParams p) {
    constexpr int NP = NT / DK, RC = DK / NP, RS = DV / NP, NW = DK / 32;
    constexpr int BUF = TL * (3 * DK + 2 * DV) + TL;  // q k la | v g | lambda
    extern __shared__ float4 smem_f4[];
    float *sm = reinterpret_cast<float *>(smem_f4);
    float *red1 = sm + 2 * BUF, *red2 = red1 + NT, *red3 = red2 + NT, *gyv = red3 + NT;
    float *wsum = gyv + DK;  // [4][8]: m.q, w.q, glambda, mu.gy per warp
    const int tid = threadIdx.x, x = tid % DK, part = tid / DK, lane = tid & 31, warp = tid >> 5;
    const int bh = blockIdx.x, h = bh % p.H, T = p.T;
    const size_t tok0 = (size_t)bh * T;
    const Ws ws(p, DK);
    const bool gate = p.lambda_in == nullptr;

    float Cr[RC], Sr[RS];  // C[x][part*RC + r],  S[x][part*RS + r]
#pragma unroll
    for (int r = 0; r < RC; ++r)
        Cr[r] = p.C0 ? p.C0[((size_t)bh * DK + x) * DK + part * RC + r] : 0.f;
#pragma unroll
    for (int r = 0; r < RS; ++r)
        Sr[r] = p.S0 ? p.S0[((size_t)bh * DK + x) * DV + part * RS + r] : 0.f;
    float m_x = (tid < DK && p.m0) ? p.m0[(size_t)bh * DK + x] : 0.f;
    const float wl = (gate && tid < DK) ? p.w_lambda[h * DK + x] : 0.f;
    const float bl = gate ? p.b_lambda[h] : 0.f;
    float dw = 0.f, db = 0.f;

    auto load = [&](int c) {
        float *b = sm + (c & 1) * BUF;
        const int tc = c * TL, n = min(TL, T - tc);
        const size_t r0 = tok0 + tc;
        stage(b, p.q + r0 * DK, n * DK);
        stage(b + TL * DK, p.k + r0 * DK, n * DK);
        stage(b + 2 * TL * DK, p.log_alpha + r0 * DK, n * DK);
        stage(b + 3 * TL * DK, p.v + r0 * DV, n * DV);
        stage(b + 3 * TL * DK + TL * DV, p.grad_o + r0 * DV, n * DV);
        if (!gate && tid < n) b[3 * TL * DK + 2 * TL * DV + tid] = p.lambda_in[r0 + tid];
        cp_commit();
    };

    const int nch = (T + TL - 1) / TL;
    if (nch > 0) load(0);
    for (int c = 0; c < nch; ++c) {
        cp_wait_all();
        __syncthreads();
        if (c + 1 < nch) load(c + 1);
        const float *b = sm + (c & 1) * BUF;
        const int tc = c * TL, n = min(TL, T - tc);
        for (int u = 0; u < n; ++u) {
            const long long t = tc + u;
            const float *qv = b + u * DK, *kv = b + TL * DK + u * DK;
            const float *lav = b + 2 * TL * DK + u * DK;
            const float *vv = b + 3 * TL * DK + u * DV, *gv = b + 3 * TL * DK + TL * DV + u * DV;
            const float qx = qv[x], kx = kv[x], ax = expf(lav[x]);
            // (1) write: C += k k^T (row x), S = Diag(alpha) S + k v^T (row x);
            //     partial C_t q and S_t g
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int r = 0; r < RC; r += 4) {
                const float4 k4 = ld4(kv + part * RC + r), q4 = ld4(qv + part * RC + r);
                Cr[r] = fmaf(k4.x, kx, Cr[r]);
                Cr[r + 1] = fmaf(k4.y, kx, Cr[r + 1]);
                Cr[r + 2] = fmaf(k4.z, kx, Cr[r + 2]);
                Cr[r + 3] = fmaf(k4.w, kx, Cr[r + 3]);
                a0 = fmaf(Cr[r], q4.x, a0);
                a1 = fmaf(Cr[r + 1], q4.y, a1);
                a2 = fmaf(Cr[r + 2], q4.z, a2);
                a3 = fmaf(Cr[r + 3], q4.w, a3);
            }
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
            for (int r = 0; r < RS; r += 4) {
                const float4 v4 = ld4(vv + part * RS + r), g4 = ld4(gv + part * RS + r);
                Sr[r] = fmaf(ax, Sr[r], kx * v4.x);
                Sr[r + 1] = fmaf(ax, Sr[r + 1], kx * v4.y);
                Sr[r + 2] = fmaf(ax, Sr[r + 2], kx * v4.z);
                Sr[r + 3] = fmaf(ax, Sr[r + 3], kx * v4.w);
                s0 = fmaf(Sr[r], g4.x, s0);
                s1 = fmaf(Sr[r + 1], g4.y, s1);
                s2 = fmaf(Sr[r + 2], g4.z, s2);
                s3 = fmaf(Sr[r + 3], g4.w, s3);
            }
            red1[part * DK + x] = (a0 + a1) + (a2 + a3);
            red2[part * DK + x] = (s0 + s1) + (s2 + s3);
            if (tid < DK) {
                m_x += kx;
                const float mq = warp_sum(m_x * qx), z = warp_sum(wl * qx);
                if (lane == 0) {
                    wsum[warp] = mq;
                    wsum[8 + warp] = z;
                }
            }
            __syncthreads();
            // (2) the read and the local gradients, one thread per channel x
            float gqc = 0.f, qc = 0.f, gy = 0.f, lam = 0.f, rn = 0.f, mu = 0.f, mqn = 0.f;
            if (tid < DK) {
                float mq = 0.f, z = 0.f, cq = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    mq += wsum[w];
                    z += wsum[8 + w];
                }
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    cq += red1[j * DK + x];
                    gqc += red2[j * DK + x];
                }
                rn = 1.0f / (float)(p.t0 + t + 1);
                mu = m_x * rn;
                mqn = mq * rn;  // mu . q
                const float y = cq * rn - mu * mqn;
                lam = gate ? 1.0f / (1.0f + expf(-(z + bl))) : b[3 * TL * DK + 2 * TL * DV + u];
                qc = qx - lam * y;
                gy = -lam * gqc;
                gyv[x] = gy;
                const float gl = warp_sum(-y * gqc), mg = warp_sum(mu * gy);
                if (lane == 0) {
                    wsum[16 + warp] = gl;
                    wsum[24 + warp] = mg;
                }
            }
            __syncthreads();
            // (3) partial C_t gy
            a0 = a1 = a2 = a3 = 0.f;
#pragma unroll
            for (int r = 0; r < RC; r += 4) {
                const float4 y4 = ld4(gyv + part * RC + r);
                a0 = fmaf(Cr[r], y4.x, a0);
                a1 = fmaf(Cr[r + 1], y4.y, a1);
                a2 = fmaf(Cr[r + 2], y4.z, a2);
                a3 = fmaf(Cr[r + 3], y4.w, a3);
            }
            red3[part * DK + x] = (a0 + a1) + (a2 + a3);
            __syncthreads();
            // (4) dq_t and what the reverse sweep needs
            if (tid < DK) {
                float gl = 0.f, mg = 0.f, cgy = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    gl += wsum[16 + w];
                    mg += wsum[24 + w];
                }
#pragma unroll
                for (int j = 0; j < NP; ++j) cgy += red3[j * DK + x];
                const float gz = gate ? gl * lam * (1.0f - lam) : 0.f;
                const size_t o = (tok0 + t) * DK + x;
                p.grad_q[o] = gqc + (cgy * rn - mu * mg) + gz * wl;
                ws.qc[o] = qc;
                ws.gy[o] = gy;
                ws.t1[o] = qc * gqc;
                if (x == 0)
                    *reinterpret_cast<float4 *>(ws.sc + (tok0 + t) * 4) =
                        make_float4(mqn * rn, mg * rn, 0.f, 0.f);
                dw = fmaf(gz, qx, dw);
                db += gz;
            }
        }
    }
    // rowsum(dL/dS_T * S_T): the final state's share of the decay gradient
    float rs = 0.f;
    if (p.grad_S) {
#pragma unroll
        for (int r = 0; r < RS; ++r)
            rs = fmaf(p.grad_S[((size_t)bh * DK + x) * DV + part * RS + r], Sr[r], rs);
    }
    red1[part * DK + x] = rs;
    __syncthreads();
    if (tid < DK) {
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < NP; ++j) s += red1[j * DK + x];
        ws.rs[(size_t)bh * DK + x] = s;
        if (p.grad_w) p.grad_w[(size_t)bh * DK + x] = dw;
        if (p.grad_b && x == 0) p.grad_b[bh] = db;
    }
}

template <int DK, int DV>
__global__ void __launch_bounds__(NT, 1) rev_sweep_kernel(const BwdParams p) {
    constexpr int NP = NT / DK, RC = DK / NP, RS = DV / NP;
    constexpr int NPV = NT / DV, RV = DK / NPV;
    constexpr int BUF = TL * (6 * DK + 2 * DV + 4);  // q k la qc gy t1 | v g | scalars
    constexpr int GSP = DV + 1;                        // padded row of GS
    extern __shared__ float4 smem_f4[];
    float *sm = reinterpret_cast<float *>(smem_f4);
    float *GS = sm + 2 * BUF;       // [DK][GSP]
    float *red1 = GS + DK * GSP;    // [2][NT]  rows of GS v, by token parity
    float *red2 = red1 + 2 * NT;    // [2][NT]  rows of (GC + GC^T) k
    float *red3 = red2 + 2 * NT;    // [NT]     columns of GS^T k
    const int tid = threadIdx.x, x = tid % DK, part = tid / DK;
    const int y = tid % DV, vpart = tid / DV;
    const int bh = blockIdx.x, T = p.T;
    const size_t tok0 = (size_t)bh * T;
    const Ws ws(p, DK);

    for (int e = tid; e < DK * DV; e += NT)
        GS[(e / DV) * GSP + e % DV] = p.grad_S ? p.grad_S[(size_t)bh * DK * DV + e] : 0.f;
    float G[RC];  // (GC + GC^T)[x][part*RC + r]
#pragma unroll
    for (int r = 0; r < RC; ++r) {
        const int j = part * RC + r;
        G[r] = p.grad_C ? p.grad_C[((size_t)bh * DK + x) * DK + j] +
                              p.grad_C[((size_t)bh * DK + j) * DK + x]
                        : 0.f;
    }
    float Gm = (tid < DK && p.grad_m) ? p.grad_m[(size_t)bh * DK + x] : 0.f;
    float acc = tid < DK ? ws.rs[(size_t)bh * DK + x] : 0.f;
    float an = 1.0f;  // alpha of the token after the current one
    __syncthreads();

    auto load = [&](int c) {
        float *b = sm + (c & 1) * BUF;
        const int tc = c * TL, n = min(TL, T - tc);
        const size_t r0 = tok0 + tc;
        stage(b, p.q + r0 * DK, n * DK);
        stage(b + TL * DK, p.k + r0 * DK, n * DK);
        stage(b + 2 * TL * DK, p.log_alpha + r0 * DK, n * DK);
        stage(b + 3 * TL * DK, ws.qc + r0 * DK, n * DK);
        stage(b + 4 * TL * DK, ws.gy + r0 * DK, n * DK);
        stage(b + 5 * TL * DK, ws.t1 + r0 * DK, n * DK);
        stage(b + 6 * TL * DK, p.v + r0 * DV, n * DV);
        stage(b + 6 * TL * DK + TL * DV, p.grad_o + r0 * DV, n * DV);
        stage(b + 6 * TL * DK + 2 * TL * DV, ws.sc + r0 * 4, n * 4);
        cp_commit();
    };

    const int nch = (T + TL - 1) / TL;
    if (nch > 0) load(nch - 1);
    for (int c = nch - 1; c >= 0; --c) {
        cp_wait_all();
        __syncthreads();
        if (c > 0) load(c - 1);
        const float *b = sm + (c & 1) * BUF;
        const int tc = c * TL, n = min(TL, T - tc);
        for (int u = n - 1; u >= 0; --u) {
            const long long t = tc + u;
            const int par = (int)(t & 1);
            const float *qv = b + u * DK, *kv = b + TL * DK + u * DK;
            const float *lav = b + 2 * TL * DK + u * DK, *qcv = b + 3 * TL * DK + u * DK;
            const float *gyv = b + 4 * TL * DK + u * DK, *t1v = b + 5 * TL * DK + u * DK;
            const float *vv = b + 6 * TL * DK + u * DV, *gv = b + 6 * TL * DK + TL * DV + u * DV;
            const float *scv = b + 6 * TL * DK + 2 * TL * DV + u * 4;
            const float qx = qv[x], kx = kv[x], qcx = qcv[x], gyx = gyv[x];
            const float rn = 1.0f / (float)(p.t0 + t + 1);
            // (1) GS = Diag(alpha_{t+1}) GS + qc g^T (row x), row sums GS v;
            //     G += (gy q^T + q gy^T) / n (row x), row sums G k
            float *g = GS + x * GSP + part * RS;
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
            for (int r = 0; r < RS; r += 4) {
                const float4 g4 = ld4(gv + part * RS + r), v4 = ld4(vv + part * RS + r);
                const float e0 = fmaf(an, g[r], qcx * g4.x), e1 = fmaf(an, g[r + 1], qcx * g4.y);
                const float e2 = fmaf(an, g[r + 2], qcx * g4.z), e3 = fmaf(an, g[r + 3], qcx * g4.w);
                g[r] = e0;
                g[r + 1] = e1;
                g[r + 2] = e2;
                g[r + 3] = e3;
                s0 = fmaf(e0, v4.x, s0);
                s1 = fmaf(e1, v4.y, s1);
                s2 = fmaf(e2, v4.z, s2);
                s3 = fmaf(e3, v4.w, s3);
            }
            const float gyn = gyx * rn, qn = qx * rn;
            float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
#pragma unroll
            for (int r = 0; r < RC; r += 4) {
                const float4 q4 = ld4(qv + part * RC + r), y4 = ld4(gyv + part * RC + r);
                const float4 k4 = ld4(kv + part * RC + r);
                G[r] = fmaf(gyn, q4.x, fmaf(qn, y4.x, G[r]));
                G[r + 1] = fmaf(gyn, q4.y, fmaf(qn, y4.y, G[r + 1]));
                G[r + 2] = fmaf(gyn, q4.z, fmaf(qn, y4.z, G[r + 2]));
                G[r + 3] = fmaf(gyn, q4.w, fmaf(qn, y4.w, G[r + 3]));
                c0 = fmaf(G[r], k4.x, c0);
                c1 = fmaf(G[r + 1], k4.y, c1);
                c2 = fmaf(G[r + 2], k4.z, c2);
                c3 = fmaf(G[r + 3], k4.w, c3);
            }
            red1[par * NT + part * DK + x] = (s0 + s1) + (s2 + s3);
            red2[par * NT + part * DK + x] = (c0 + c1) + (c2 + c3);
            an = expf(lav[x]);
            __syncthreads();
            // (2) column sums GS^T k (column y)
            float v0 = 0.f, v1 = 0.f;
#pragma unroll 8
            for (int r = 0; r < RV; r += 2) {
                const int cc = vpart * RV + r;
                v0 = fmaf(GS[cc * GSP + y], kv[cc], v0);
                v1 = fmaf(GS[(cc + 1) * GSP + y], kv[cc + 1], v1);
            }
            red3[vpart * DV + y] = v0 + v1;
            __syncthreads();
            // (3) dk_t, the decay gradient, dv_t
            if (tid < DK) {
                float gsv = 0.f, gk = 0.f;
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    gsv += red1[par * NT + j * DK + x];
                    gk += red2[par * NT + j * DK + x];
                }
                Gm -= gyx * scv[0] + qx * scv[1];
                const size_t o = (tok0 + t) * DK + x;
                p.grad_k[o] = gk + Gm + gsv;
                acc += t1v[x] - kx * gsv;
                p.grad_la[o] = acc;
            }
            if (tid < DV) {
                float s = 0.f;
#pragma unroll
                for (int j = 0; j < NPV; ++j) s += red3[j * DV + y];
                p.grad_v[(tok0 + t) * DV + y] = s;
            }
        }
    }
    // gradients of the carried state (each thread writes what it owns)
    if (p.grad_S0) {
#pragma unroll
        for (int r = 0; r < RS; ++r)
            p.grad_S0[((size_t)bh * DK + x) * DV + part * RS + r] = an * GS[x * GSP + part * RS + r];
    }
    if (p.grad_C0) {
#pragma unroll
        for (int r = 0; r < RC; ++r)
            p.grad_C0[((size_t)bh * DK + x) * DK + part * RC + r] = 0.5f * G[r];
    }
    if (p.grad_m0 && tid < DK) p.grad_m0[(size_t)bh * DK + x] = Gm;
}

template <int DK, int DV>
size_t fwd_smem() {
    return sizeof(float) * (2 * (TL * (3 * DK + 2 * DV) + TL) + 3 * NT + DK + 32);
}
template <int DK, int DV>
size_t rev_smem() {
    return sizeof(float) * (2 * TL * (6 * DK + 2 * DV + 4) + DK * (DV + 1) + 5 * NT);
}

template <int DK, int DV>
cudaError_t launch_shape(const BwdParams &p, cudaStream_t st) {
    const size_t fb = fwd_smem<DK, DV>(), rb = rev_smem<DK, DV>();
    cudaError_t e = cudaFuncSetAttribute(fwd_sweep_kernel<DK, DV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fb);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(rev_sweep_kernel<DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)rb);
    if (e != cudaSuccess) return e;
    fwd_sweep_kernel<DK, DV><<<p.BH, NT, fb, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    rev_sweep_kernel<DK, DV><<<p.BH, NT, rb, st>>>(p);
    return cudaGetLastError();
}

}  // namespace bwd

size_t gla_bwd_workspace_floats(long long BH, long long T, int dk) {
    return (size_t)(BH * T * (3LL * dk + 4) + BH * dk);
}

cudaError_t launch_gla_bwd(const BwdParams &p, int dk, int dv, cudaStream_t st) {
    using namespace bwd;
    if (p.BH == 0) return cudaSuccess;
    if (dk == 64 && dv == 64) return launch_shape<64, 64>(p, st);
    if (dk == 64 && dv == 128) return launch_shape<64, 128>(p, st);
    if (dk == 128 && dv == 64) return launch_shape<128, 64>(p, st);
    return launch_shape<128, 128>(p, st);
}

}  // namespace ccq

// ---- ccq_gla_bwd_noalloc: the same two kernels on a fixed scratch array --
//
// For callers that must not allocate device memory on the call path (a
// runtime that hands all device memory to its own allocator up front, or
// latency-bound code that cannot take the implicit device synchronisation of
// cudaMalloc and cudaFree): the workspace is this file-scope array, sized by
// CCQ_GLA_BWD_NOALLOC_SCRATCH_BYTES.  Nothing in it needs to start at zero:
// the forward sweep writes every word the reverse sweep reads.  Every call on
// a device shares it, so calls whose kernels overlap on the GPU race.
static __device__ __align__(256) float ccq_bwd_scratch[CCQ_GLA_BWD_NOALLOC_SCRATCH_BYTES /
                                                        sizeof(float)];

namespace {
std::mutex scratch_mu;
void *scratch_ptr[64] = {};

// Device address of ccq_bwd_scratch on the current device, looked up on the
// first call on that device and kept.
void *static_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(scratch_mu);
    if (!scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, ccq_bwd_scratch) != cudaSuccess) return nullptr;
        scratch_ptr[dev] = ptr;
    }
    return scratch_ptr[dev];
}
}  // namespace

extern "C" ccq_status ccq_gla_bwd_noalloc(
    const float *q, const float *k, const float *v, const float *log_alpha,
    const float *w_lambda, const float *b_lambda, const float *lambda_in, const float *S0,
    const float *C0, const float *m0, int64_t t0, const float *grad_o, const float *grad_S,
    const float *grad_C, const float *grad_m, float *grad_q, float *grad_k, float *grad_v,
    float *grad_log_alpha, float *grad_w_lambda, float *grad_b_lambda, float *grad_S0,
    float *grad_C0, float *grad_m0, int B, int H, int T, int dk, int dv, unsigned flags,
    ccq_stream_t stream) {
    const size_t need = ccq_gla_bwd_workspace_bytes(B, H, T, dk, dv);
    if (need > (size_t)CCQ_GLA_BWD_NOALLOC_SCRATCH_BYTES) return CCQ_ERR_TOO_LARGE;
    void *ws = nullptr;
    if (B > 0 && H > 0) {  // no CUDA call for an empty batch or a rejected size
        ws = static_scratch();
        if (!ws) return CCQ_ERR_CUDA;
    }
    return ccq_gla_bwd(q, k, v, log_alpha, w_lambda, b_lambda, lambda_in, S0, C0, m0, t0, grad_o,
                       grad_S, grad_C, grad_m, grad_q, grad_k, grad_v, grad_log_alpha,
                       grad_w_lambda, grad_b_lambda, grad_S0, grad_C0, grad_m0, ws,
                       (size_t)CCQ_GLA_BWD_NOALLOC_SCRATCH_BYTES, B, H, T, dk, dv, flags, stream);
}
