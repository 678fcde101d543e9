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
// Two sweeps over the tokens, one CTA per (b, h) in each, chunks of TL = 8
// tokens with one warp per token of a chunk:
//
// 1. Forward sweep.  Everything that depends on the forward state can be
//    formed going forward, because the upstream gradient g_t = dL/do_t is
//    known: gqc_t = S_t g_t, glambda_t = -y_t . gqc_t, gy_t = -lambda_t gqc_t,
//    and the query gradient
//      dq_t = gqc_t + Sigma_t gy_t + lambda_t (1 - lambda_t) glambda_t w.
//    C and S stay in registers: thread (x, part) owns row x of C and row x
//    of S, each over one slice of columns, the only elements it ever reads
//    or writes (C is symmetric, so C0 must be too: it is a sum of k k^T).
//    Per chunk: (A) every thread applies the chunk's writes token by token
//    to its rows and leaves the partial products C_u q_u and S_u g_u;
//    (B) warp u finishes token u's read and local gradients; (C) the
//    products C_end gy_u with the chunk's last C, corrected in (D) by
//    - sum_{u'>u} k_u' (k_u' . gy_u) to C_u gy_u.  Four block barriers per
//    chunk.  Per token it leaves in the workspace qc_t, gy_t, qc_t * gqc_t
//    and the two scalars (mu.q)/n and (mu.gy)/n that rebuild dL/dmu_t / n_t.
//
// 2. Reverse sweep.  The adjoints of the three sums run backwards:
//      GS_t = qc_t g_t^T + Diag(alpha_{t+1}) GS_{t+1}      (dL/dS_t)
//      GC_t = gy_t q_t^T / n_t + GC_{t+1}                  (dL/dC_t)
//      Gm_t = dL/dmu_t / n_t + Gm_{t+1}                    (dL/dm_t)
//    with dk_t = (GC_t + GC_t^T) k_t + Gm_t + GS_t v_t and dv_t = GS_t^T k_t.
//    GC enters only through GC + GC^T, so that symmetric sum is what is kept
//    (registers, row-owned, updated token by token).  GS sits in shared
//    memory with padded rows and moves a chunk at a time: inside a chunk,
//    with X the adjoint entering it and P_u the decay product from token u
//    to the chunk's end,
//      GS_u = P_u X + sum_{u' >= u} (P_u / P_u') qc_u' g_u'^T,
//    so GS_u v_u and GS_u^T k_u are one pass over the rows and one over the
//    columns of X against all eight tokens, plus 8 x 8 in-chunk terms.
//    The decay gradient uses d log A_t = qc_t * gqc_t - k_t * (GS_t v_t)
//    (A_t the running product of alpha; the final state adds
//    rowsum(dL/dS_T * S_T)), summed over t' >= t: no sweep ever needs
//    S_{t-1}, and no state is rebuilt by dividing out a decay.  Five block
//    barriers per chunk.
//
// Shapes: dk, dv in {64, 128}; any T (a ragged last chunk); 256 threads.
// Token vectors are staged a chunk at a time with cp.async (16-byte
// copies, double-buffered) so each chunk's loads overlap the previous chunk.
#include <mutex>

#include "common.cuh"

namespace ccq {

namespace bwd {

// CTA size and chunk length of the two sweeps: 512 threads (16 warps, so
// each SM has warps to switch to while one waits on shared memory); the
// forward sweep takes 16-token chunks (one warp per token), the reverse
// sweep 8-token chunks (its chunk buffers and partial products are larger).
constexpr int NT_F = 512, TL_F = 16;
constexpr int NT_R = 512, TL_R = 8;

__device__ __forceinline__ void cp16(float *dst, const float *src) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all() {
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}
// n floats (n % 4 == 0; both ends 16-byte aligned), spread over the CTA
template <int NT>
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

template <int DK, int DV, int NT = NT_F, int TL = TL_F>
__global__ void __launch_bounds__(NT, 1) fwd_sweep_kernel(const BwdParams p) {
    constexpr int NP = NT / DK, RC = DK / NP, RS = DV / NP, XL = DK / 32;
    constexpr int BUF = TL * (3 * DK + 2 * DV) + TL;  // q k la | v g | lambda
    static_assert(NT / 32 == TL, "one warp per token of a chunk");
    extern __shared__ float4 smem_f4[];
    float *sm = reinterpret_cast<float *>(smem_f4);
    float *red1 = sm + 2 * BUF;     // [TL][NT]  C_u q_u partials, by (x, part)
    float *red2 = red1 + TL * NT;   // [TL][NT]  S_u g_u partials
    float *red3 = red2 + TL * NT;   // [TL][NT]  C_end gy_u partials
    float *mb = red3 + TL * NT;     // [TL][DK]  m after token u
    float *gyb = mb + TL * DK;      // [TL][DK]  gy_u
    float *dmat = gyb + TL * DK;    // [TL][TL]  k_u' . gy_u (u' > u)
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
    float m_x = (part == 0 && p.m0) ? p.m0[(size_t)bh * DK + x] : 0.f;
    // per-lane values of the warp-per-token phases: channel x = lane + 32 i
    float wl[XL], dw[XL];
#pragma unroll
    for (int i = 0; i < XL; ++i) {
        wl[i] = gate ? p.w_lambda[h * DK + lane + 32 * i] : 0.f;
        dw[i] = 0.f;
    }
    const float bl = gate ? p.b_lambda[h] : 0.f;
    float db = 0.f;

    auto load = [&](int c) {
        float *b = sm + (c & 1) * BUF;
        const int tc = c * TL, n = min(TL, T - tc);
        const size_t r0 = tok0 + tc;
        stage<NT>(b, p.q + r0 * DK, n * DK);
        stage<NT>(b + TL * DK, p.k + r0 * DK, n * DK);
        stage<NT>(b + 2 * TL * DK, p.log_alpha + r0 * DK, n * DK);
        stage<NT>(b + 3 * TL * DK, p.v + r0 * DV, n * DV);
        stage<NT>(b + 3 * TL * DK + TL * DV, p.grad_o + r0 * DV, n * DV);
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
        const float *Q = b, *K = b + TL * DK, *LA = b + 2 * TL * DK;
        const float *V = b + 3 * TL * DK, *G = V + TL * DV, *LAM = G + TL * DV;
        const int tc = c * TL, n = min(TL, T - tc);

        // (A) the write, token by token, in registers: C += k k^T and
        //     S = Diag(alpha) S + k v^T on the owned rows, with the partial
        //     products C_u q_u and S_u g_u of every token
        for (int u = 0; u < n; ++u) {
            const float *qv = Q + u * DK, *kv = K + u * DK, *vv = V + u * DV, *gv = G + u * DV;
            const float kx = kv[x], ax = expf(LA[u * DK + x]);
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
            red1[u * NT + part * DK + x] = (a0 + a1) + (a2 + a3);
            red2[u * NT + part * DK + x] = (s0 + s1) + (s2 + s3);
            if (part == 0) {
                m_x += kx;
                mb[u * DK + x] = m_x;
            }
        }
        __syncthreads();

        // (B) warp u: the read and the local gradients of token u
        const int u = warp;
        const long long t = tc + u;
        float gqc[XL], qc[XL], gy[XL], mu[XL];
        float rn = 0.f, mqn = 0.f, lam = 0.f, gl = 0.f, mg = 0.f;
        if (u < n) {
            const float *qv = Q + u * DK;
            float cq[XL], mq = 0.f, z = 0.f;
#pragma unroll
            for (int i = 0; i < XL; ++i) {
                const int xi = lane + 32 * i;
                cq[i] = 0.f;
                gqc[i] = 0.f;
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    cq[i] += red1[u * NT + j * DK + xi];
                    gqc[i] += red2[u * NT + j * DK + xi];
                }
                mq = fmaf(mb[u * DK + xi], qv[xi], mq);
                z = fmaf(wl[i], qv[xi], z);
            }
            mq = warp_sum(mq);
            z = warp_sum(z);
            rn = 1.0f / (float)(p.t0 + t + 1);
            mqn = mq * rn;  // mu . q
            lam = gate ? 1.0f / (1.0f + expf(-(z + bl))) : LAM[u];
            float glp = 0.f, mgp = 0.f;
#pragma unroll
            for (int i = 0; i < XL; ++i) {
                const int xi = lane + 32 * i;
                mu[i] = mb[u * DK + xi] * rn;
                const float y = cq[i] * rn - mu[i] * mqn;
                qc[i] = qv[xi] - lam * y;
                gy[i] = -lam * gqc[i];
                gyb[u * DK + xi] = gy[i];
                glp = fmaf(-y, gqc[i], glp);
                mgp = fmaf(mu[i], gy[i], mgp);
            }
            gl = warp_sum(glp);
            mg = warp_sum(mgp);
            // k_u' . gy_u for the later tokens of the chunk: C_u = C_end - sum_{u'>u} k k^T
            for (int up = u + 1; up < n; ++up) {
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < XL; ++i) s = fmaf(K[up * DK + lane + 32 * i], gy[i], s);
                s = warp_sum(s);
                if (lane == 0) dmat[up * TL + u] = s;
            }
        }
        __syncthreads();

        // (C) C_end gy_u for every token, on the owned rows
        for (int v_ = 0; v_ < n; ++v_) {
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int r = 0; r < RC; r += 4) {
                const float4 y4 = ld4(gyb + v_ * DK + part * RC + r);
                a0 = fmaf(Cr[r], y4.x, a0);
                a1 = fmaf(Cr[r + 1], y4.y, a1);
                a2 = fmaf(Cr[r + 2], y4.z, a2);
                a3 = fmaf(Cr[r + 3], y4.w, a3);
            }
            red3[v_ * NT + part * DK + x] = (a0 + a1) + (a2 + a3);
        }
        __syncthreads();

        // (D) warp u: dq_u and what the reverse sweep needs
        if (u < n) {
            const float gz = gate ? gl * lam * (1.0f - lam) : 0.f;
            const float *qv = Q + u * DK;
#pragma unroll
            for (int i = 0; i < XL; ++i) {
                const int xi = lane + 32 * i;
                float cgy = 0.f;
#pragma unroll
                for (int j = 0; j < NP; ++j) cgy += red3[u * NT + j * DK + xi];
                for (int up = u + 1; up < n; ++up) cgy -= K[up * DK + xi] * dmat[up * TL + u];
                const size_t o = (tok0 + t) * DK + xi;
                p.grad_q[o] = gqc[i] + (cgy * rn - mu[i] * mg) + gz * wl[i];
                ws.qc[o] = qc[i];
                ws.gy[o] = gy[i];
                ws.t1[o] = qc[i] * gqc[i];
                dw[i] = fmaf(gz, qv[xi], dw[i]);
            }
            if (lane == 0) {
                *reinterpret_cast<float4 *>(ws.sc + (tok0 + t) * 4) =
                    make_float4(mqn * rn, mg * rn, 0.f, 0.f);
                db += gz;
            }
        }
    }
    // rowsum(dL/dS_T * S_T): the final state's share of the decay gradient;
    // the gate gradients summed over the warps
    float rs = 0.f;
    if (p.grad_S) {
#pragma unroll
        for (int r = 0; r < RS; ++r)
            rs = fmaf(p.grad_S[((size_t)bh * DK + x) * DV + part * RS + r], Sr[r], rs);
    }
    __syncthreads();
    red1[part * DK + x] = rs;
#pragma unroll
    for (int i = 0; i < XL; ++i) red2[warp * DK + lane + 32 * i] = dw[i];
    if (lane == 0) red2[TL * DK + warp] = db;
    __syncthreads();
    if (tid < DK) {
        float s = 0.f, w_ = 0.f;
#pragma unroll
        for (int j = 0; j < NP; ++j) s += red1[j * DK + x];
#pragma unroll
        for (int j = 0; j < TL; ++j) w_ += red2[j * DK + x];
        ws.rs[(size_t)bh * DK + x] = s;
        if (p.grad_w) p.grad_w[(size_t)bh * DK + x] = w_;
        if (p.grad_b && x == 0) {
            float b_ = 0.f;
            for (int j = 0; j < TL; ++j) b_ += red2[TL * DK + j];
            p.grad_b[bh] = b_;
        }
    }
}

template <int DK, int DV, int NT = NT_R, int TL = TL_R>
__global__ void __launch_bounds__(NT, 1) rev_sweep_kernel(const BwdParams p) {
    constexpr int NP = NT / DK, RC = DK / NP, RS = DV / NP, XL = DK / 32, YL = DV / 32;
    constexpr int NPV = NT / DV, RV = DK / NPV;
    constexpr int BUF = TL * (6 * DK + 2 * DV + 4);  // q k la qc gy t1 | v g | scalars
    constexpr int GSP = DV + 1;                        // padded row of GS
    static_assert(NT / 32 >= TL && TL == 8, "one warp per token of a chunk");
    extern __shared__ float4 smem_f4[];
    float *sm = reinterpret_cast<float *>(smem_f4);
    float *GS = sm + 2 * BUF;          // [DK][GSP]  dL/dS after the chunk's last token + 1
    float *red_row = GS + DK * GSP;    // [TL][NT]   X v_u partials, by (x, part)
    float *red_gk = red_row + TL * NT; // [TL][NT]   (GC + GC^T)_u k_u partials
    float *red_col = red_gk + TL * NT; // [TL][NT]   X^T (P_u k_u) partials, by (y, vpart)
    float *Lc = red_col + TL * NT;     // [TL][DK]   log P_u
    float *kPt = Lc + TL * DK;         // [DK][TL]   P_u k_u, transposed
    float *vt = kPt + DK * TL;         // [DV][TL]   v_u, transposed
    float *gt = vt + DV * TL;          // [DV][TL]   g_u, transposed
    float *gsvb = gt + DV * TL;        // [TL][DK]   GS_u v_u
    float *Wv = gsvb + TL * DK;        // [TL][TL]   g_u' . v_u
    float *Wk = Wv + TL * TL;          // [TL][TL]   sum_x P_u/P_u' qc_u' k_u
    float *carry = Wk + TL * TL;       // [2][3][DK] acc, Gm, log alpha of the next token
    const int tid = threadIdx.x, x = tid % DK, part = tid / DK, lane = tid & 31, warp = tid >> 5;
    const int y = tid % DV, vpart = tid / DV;
    const int bh = blockIdx.x, T = p.T;
    const size_t tok0 = (size_t)bh * T;
    const Ws ws(p, DK);

    for (int e = tid; e < DK * DV; e += NT)
        GS[(e / DV) * GSP + e % DV] = p.grad_S ? p.grad_S[(size_t)bh * DK * DV + e] : 0.f;
    float Gr[RC];  // (GC + GC^T)[x][part*RC + r]
#pragma unroll
    for (int r = 0; r < RC; ++r) {
        const int j = part * RC + r;
        Gr[r] = p.grad_C ? p.grad_C[((size_t)bh * DK + x) * DK + j] +
                               p.grad_C[((size_t)bh * DK + j) * DK + x]
                         : 0.f;
    }
    if (tid < DK) {
        carry[0 * DK + x] = ws.rs[(size_t)bh * DK + x];
        carry[1 * DK + x] = p.grad_m ? p.grad_m[(size_t)bh * DK + x] : 0.f;
        carry[2 * DK + x] = 0.f;
    }
    __syncthreads();

    auto load = [&](int c) {
        float *b = sm + (c & 1) * BUF;
        const int tc = c * TL, n = min(TL, T - tc);
        const size_t r0 = tok0 + tc;
        stage<NT>(b, p.q + r0 * DK, n * DK);
        stage<NT>(b + TL * DK, p.k + r0 * DK, n * DK);
        stage<NT>(b + 2 * TL * DK, p.log_alpha + r0 * DK, n * DK);
        stage<NT>(b + 3 * TL * DK, ws.qc + r0 * DK, n * DK);
        stage<NT>(b + 4 * TL * DK, ws.gy + r0 * DK, n * DK);
        stage<NT>(b + 5 * TL * DK, ws.t1 + r0 * DK, n * DK);
        stage<NT>(b + 6 * TL * DK, p.v + r0 * DV, n * DV);
        stage<NT>(b + 6 * TL * DK + TL * DV, p.grad_o + r0 * DV, n * DV);
        stage<NT>(b + 6 * TL * DK + 2 * TL * DV, ws.sc + r0 * 4, n * 4);
        cp_commit();
    };

    const int nch = (T + TL - 1) / TL;
    if (nch > 0) load(nch - 1);
    int it = 0;
    for (int c = nch - 1; c >= 0; --c, ++it) {
        cp_wait_all();
        __syncthreads();
        if (c > 0) load(c - 1);
        const float *b = sm + (c & 1) * BUF;
        const float *Q = b, *K = b + TL * DK, *LA = b + 2 * TL * DK, *QC = b + 3 * TL * DK;
        const float *GY = b + 4 * TL * DK, *T1 = b + 5 * TL * DK, *V = b + 6 * TL * DK;
        const float *G = V + TL * DV, *SC = G + TL * DV;
        const float *cin = carry + (it & 1) * 3 * DK;
        float *cout = carry + ((it + 1) & 1) * 3 * DK;
        const int tc = c * TL, n = min(TL, T - tc);

        // (prep) log P_u = sum of log alpha over the tokens after u up to the
        // first token of the next chunk; P_u k_u, v and g transposed
        if (tid < DK) {
            float s = cin[2 * DK + x];
            for (int u = TL - 1; u >= 0; --u) {
                if (u < n) {
                    Lc[u * DK + x] = s;
                    kPt[x * TL + u] = expf(s) * K[u * DK + x];
                    s += LA[u * DK + x];
                } else {
                    kPt[x * TL + u] = 0.f;
                }
            }
        } else if (tid < DK + DV) {
            const int d = tid - DK;
#pragma unroll
            for (int u = 0; u < TL; ++u) {
                vt[d * TL + u] = u < n ? V[u * DV + d] : 0.f;
                gt[d * TL + u] = u < n ? G[u * DV + d] : 0.f;
            }
        }
        __syncthreads();

        // (1a) rows of the entry state against every v_u
        {
            float acc[TL];
#pragma unroll
            for (int u = 0; u < TL; ++u) acc[u] = 0.f;
            const float *row = GS + x * GSP + part * RS;
#pragma unroll 4
            for (int r = 0; r < RS; ++r) {
                const float xv = row[r];
                const float4 a = ld4(vt + (part * RS + r) * TL), c4 = ld4(vt + (part * RS + r) * TL + 4);
                acc[0] = fmaf(xv, a.x, acc[0]);
                acc[1] = fmaf(xv, a.y, acc[1]);
                acc[2] = fmaf(xv, a.z, acc[2]);
                acc[3] = fmaf(xv, a.w, acc[3]);
                acc[4] = fmaf(xv, c4.x, acc[4]);
                acc[5] = fmaf(xv, c4.y, acc[5]);
                acc[6] = fmaf(xv, c4.z, acc[6]);
                acc[7] = fmaf(xv, c4.w, acc[7]);
            }
#pragma unroll
            for (int u = 0; u < TL; ++u) red_row[u * NT + part * DK + x] = acc[u];
        }
        // (1b) columns of the entry state against every P_u k_u
        {
            float acc[TL];
#pragma unroll
            for (int u = 0; u < TL; ++u) acc[u] = 0.f;
#pragma unroll 4
            for (int r = 0; r < RV; ++r) {
                const int xr = vpart * RV + r;
                const float xv = GS[xr * GSP + y];
                const float4 a = ld4(kPt + xr * TL), c4 = ld4(kPt + xr * TL + 4);
                acc[0] = fmaf(xv, a.x, acc[0]);
                acc[1] = fmaf(xv, a.y, acc[1]);
                acc[2] = fmaf(xv, a.z, acc[2]);
                acc[3] = fmaf(xv, a.w, acc[3]);
                acc[4] = fmaf(xv, c4.x, acc[4]);
                acc[5] = fmaf(xv, c4.y, acc[5]);
                acc[6] = fmaf(xv, c4.z, acc[6]);
                acc[7] = fmaf(xv, c4.w, acc[7]);
            }
#pragma unroll
            for (int u = 0; u < TL; ++u) red_col[u * NT + vpart * DV + y] = acc[u];
        }
        // (1c) the symmetric C adjoint, token by token backwards, on the owned rows
        for (int u = n - 1; u >= 0; --u) {
            const float rn = 1.0f / (float)(p.t0 + tc + u + 1);
            const float gyn = GY[u * DK + x] * rn, qn = Q[u * DK + x] * rn;
            const float *qv = Q + u * DK, *yv = GY + u * DK, *kv = K + u * DK;
            float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
#pragma unroll
            for (int r = 0; r < RC; r += 4) {
                const float4 q4 = ld4(qv + part * RC + r), y4 = ld4(yv + part * RC + r);
                const float4 k4 = ld4(kv + part * RC + r);
                Gr[r] = fmaf(gyn, q4.x, fmaf(qn, y4.x, Gr[r]));
                Gr[r + 1] = fmaf(gyn, q4.y, fmaf(qn, y4.y, Gr[r + 1]));
                Gr[r + 2] = fmaf(gyn, q4.z, fmaf(qn, y4.z, Gr[r + 2]));
                Gr[r + 3] = fmaf(gyn, q4.w, fmaf(qn, y4.w, Gr[r + 3]));
                c0 = fmaf(Gr[r], k4.x, c0);
                c1 = fmaf(Gr[r + 1], k4.y, c1);
                c2 = fmaf(Gr[r + 2], k4.z, c2);
                c3 = fmaf(Gr[r + 3], k4.w, c3);
            }
            red_gk[u * NT + part * DK + x] = (c0 + c1) + (c2 + c3);
        }
        // (1d) warp u: the in-chunk pairs u' >= u
        const int u = warp;
        if (u < n) {
#pragma unroll
            for (int up = 0; up < TL; ++up) {
                if (up < u || up >= n) continue;  // warp-uniform
                float sv = 0.f, sk = 0.f;
#pragma unroll
                for (int i = 0; i < YL; ++i)
                    sv = fmaf(G[up * DV + lane + 32 * i], V[u * DV + lane + 32 * i], sv);
#pragma unroll
                for (int i = 0; i < XL; ++i) {
                    const int xi = lane + 32 * i;
                    const float rq = expf(Lc[u * DK + xi] - Lc[up * DK + xi]) * QC[up * DK + xi];
                    sk = fmaf(rq, K[u * DK + xi], sk);
                }
                sv = warp_sum(sv);
                sk = warp_sum(sk);
                if (lane == 0) {
                    Wv[up * TL + u] = sv;
                    Wk[up * TL + u] = sk;
                }
            }
        }
        __syncthreads();

        // (2e) the state adjoint moves to the chunk's first token (owned rows)
        {
            float coef[TL];
            const float l0 = n > 0 ? Lc[x] : 0.f;
#pragma unroll
            for (int up = 0; up < TL; ++up)
                coef[up] = up < n ? expf(l0 - Lc[up * DK + x]) * QC[up * DK + x] : 0.f;
            const float e0 = expf(l0);
            float *row = GS + x * GSP + part * RS;
#pragma unroll 4
            for (int r = 0; r < RS; ++r) {
                const float4 a = ld4(gt + (part * RS + r) * TL), c4 = ld4(gt + (part * RS + r) * TL + 4);
                float g = e0 * row[r];
                g = fmaf(coef[0], a.x, g);
                g = fmaf(coef[1], a.y, g);
                g = fmaf(coef[2], a.z, g);
                g = fmaf(coef[3], a.w, g);
                g = fmaf(coef[4], c4.x, g);
                g = fmaf(coef[5], c4.y, g);
                g = fmaf(coef[6], c4.z, g);
                g = fmaf(coef[7], c4.w, g);
                row[r] = g;
            }
        }
        // (2f) warp u: dk_u, dv_u and GS_u v_u
        if (u < n) {
            const long long t = tc + u;
#pragma unroll
            for (int i = 0; i < XL; ++i) {
                const int xi = lane + 32 * i;
                float row = 0.f, gk = 0.f;
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    row += red_row[u * NT + j * DK + xi];
                    gk += red_gk[u * NT + j * DK + xi];
                }
                float gsv = expf(Lc[u * DK + xi]) * row;
                float gm = cin[DK + xi];
#pragma unroll
                for (int up = 0; up < TL; ++up) {
                    if (up < u || up >= n) continue;
                    const float rq = expf(Lc[u * DK + xi] - Lc[up * DK + xi]) * QC[up * DK + xi];
                    gsv = fmaf(rq, Wv[up * TL + u], gsv);
                    gm -= GY[up * DK + xi] * SC[up * 4] + Q[up * DK + xi] * SC[up * 4 + 1];
                }
                gsvb[u * DK + xi] = gsv;
                p.grad_k[(tok0 + t) * DK + xi] = gk + gm + gsv;
                if (u == 0) cout[DK + xi] = gm;
            }
#pragma unroll
            for (int i = 0; i < YL; ++i) {
                const int yi = lane + 32 * i;
                float s = 0.f;
#pragma unroll
                for (int j = 0; j < NPV; ++j) s += red_col[u * NT + j * DV + yi];
                for (int up = u; up < n; ++up) s = fmaf(G[up * DV + yi], Wk[up * TL + u], s);
                p.grad_v[(tok0 + t) * DV + yi] = s;
            }
        }
        __syncthreads();

        // (3) warp u: the decay gradient, a suffix sum over the tokens
        if (u < n) {
            const long long t = tc + u;
#pragma unroll
            for (int i = 0; i < XL; ++i) {
                const int xi = lane + 32 * i;
                float a = cin[xi];
                for (int up = u; up < n; ++up)
                    a += T1[up * DK + xi] - K[up * DK + xi] * gsvb[up * DK + xi];
                p.grad_la[(tok0 + t) * DK + xi] = a;
                if (u == 0) {
                    cout[xi] = a;
                    cout[2 * DK + xi] = LA[xi];
                }
            }
        }
    }
    __syncthreads();
    // gradients of the carried state (each thread writes what it owns)
    const float *cfin = carry + (it & 1) * 3 * DK;
    if (p.grad_S0) {
        const float a0 = expf(cfin[2 * DK + x]);
#pragma unroll
        for (int r = 0; r < RS; ++r)
            p.grad_S0[((size_t)bh * DK + x) * DV + part * RS + r] = a0 * GS[x * GSP + part * RS + r];
    }
    if (p.grad_C0) {
#pragma unroll
        for (int r = 0; r < RC; ++r)
            p.grad_C0[((size_t)bh * DK + x) * DK + part * RC + r] = 0.5f * Gr[r];
    }
    if (p.grad_m0 && tid < DK) p.grad_m0[(size_t)bh * DK + x] = cfin[DK + x];
}

template <int DK, int DV, int NT = NT_F, int TL = TL_F>
size_t fwd_smem() {
    return sizeof(float) * (2 * (TL * (3 * DK + 2 * DV) + TL) + 3 * TL * NT + 2 * TL * DK + TL * TL);
}
template <int DK, int DV, int NT = NT_R, int TL = TL_R>
size_t rev_smem() {
    return sizeof(float) * (2 * TL * (6 * DK + 2 * DV + 4) + DK * (DV + 1) + 3 * TL * NT +
                            TL * DK + DK * TL + 2 * DV * TL + TL * DK + 2 * TL * TL + 6 * DK);
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
    fwd_sweep_kernel<DK, DV><<<p.BH, NT_F, fb, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    rev_sweep_kernel<DK, DV><<<p.BH, NT_R, rb, st>>>(p);
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
