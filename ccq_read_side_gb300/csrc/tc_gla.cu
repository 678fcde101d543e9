// tc_gla.cu -- tcgen05 tensor-core CCQ-GLA forward (bf16 in, fp32 state),
// d_k = d_v = 128, chunks of L = 64 tokens.
//
// One thread-block cluster of two CTAs per (b, h).  The sequence is walked
// chunk by chunk; the two CTAs split each chunk's work by what it depends on:
//
//   CTA 0 ("covariance side") owns the undecayed key statistics: C (d_k x d_k,
//   fp32, in tensor memory), m (fp32, shared memory) and the token count.
//   Per chunk it forms the CCQ read of the gist.science summary of 2606.01294
//   (section 2, "mechanism": q_clean = q - lambda Sigma_t q, Sigma_t the key
//   covariance including the current token), written over the chunk:
//       A    = Q K^T                          (tcgen05, M=64 N=64 K=128)
//       s_i  = m0.q_i + sum_{j<=i} A_ij,   Ah_ij = [j<=i] (A_ij - s_i/t_i)
//       P^T  = C0 Q^T + K^T Ah^T              (tcgen05, M=128 N=64, K=128 / 64)
//       qc_i = q_i - (lambda_i / t_i) (P_i - (s_i/t_i) m0)    = q_i - lambda_i Sigma q_i
//       C   += K^T K                          (tcgen05 into the TMEM accumulator)
//   and scales the cleaned query by the chunk's per-channel decay,
//   Qt = qc * exp(-E), E_ic = sum of log alpha over the chunk's tokens after i
//   (the GLA write Diag(alpha_t) of the pages' backbone), and ships Qt^T
//   (16 KB) to CTA 1 through distributed shared memory.
//
//   CTA 1 ("GLA side") owns S (d_k x d_v, fp32, in tensor memory).  With
//   Kh = K * exp(E) (so Qt Kh^T carries exp(B_i - B_j), B the inclusive
//   cumulative log-decay) and Sb = Diag(exp R) S0 (R = the chunk's total
//   log-decay):
//       Ag   = [j<=i] Qt Kh^T                 (tcgen05, M=64 N=64 K=128)
//       O^T  = Sb^T Qt^T + V^T Ag^T           (tcgen05, M=128 N=64, K=128 / 64)
//       S    = Sb + Kh^T V                    (tcgen05 into the TMEM accumulator)
//   which is o_t = S_t^T q_clean with S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T.
//
// Warp roles per CTA: warps 0-3 run the element-wise steps (one thread per
// TMEM lane), warp 4 issues TMA loads, warp 5 issues tcgen05 MMAs.  Every
// wait is a bounded mbarrier poll; a wait that gives up records
// CCQ_ERR_TIMEOUT and the CTA winds down.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "sm103.cuh"

namespace ccq {
using namespace sm103;

namespace tcgla {

constexpr int L = 64;        // tokens per chunk
constexpr int D = 128;       // d_k = d_v
constexpr int NTHREADS = 192;
constexpr uint32_t TILE = L * D * 2;  // one [64 x 128] bf16 tile = two 64x64 TMA boxes
constexpr uint32_t BOX = L * 64 * 2;  // 8 KB

// Shared-memory tiles (byte offsets from a 1024-aligned base).  All bf16
// tiles use the 128-byte swizzle; see sw128_off / sw128_chunk.
struct CovLayout {  // CTA 0
    static constexpr uint32_t Q = 0;              // 2 stages x [64 tok][128]
    static constexpr uint32_t K = Q + 2 * TILE;   // 2 stages
    static constexpr uint32_t LA = K + 2 * TILE;  // 2 stages (log alpha)
    static constexpr uint32_t C0 = LA + 2 * TILE; // bf16 C0, K-major [128 rows][128]
    static constexpr uint32_t AH = C0 + 32768;    // bf16 Ah [64 q][64 k]
    static constexpr uint32_t QT = AH + 8192;     // bf16 Qt^T [128 ch][64 tok] (send buffer)
    static constexpr uint32_t END = QT + 16384;
};
struct GlaLayout {  // CTA 1
    static constexpr uint32_t K = 0;               // 2 stages
    static constexpr uint32_t LA = K + 2 * TILE;   // 2 stages
    static constexpr uint32_t V = LA + 2 * TILE;   // 2 stages
    static constexpr uint32_t KH = V + 2 * TILE;   // bf16 Kh^T [128 ch][64 tok]
    static constexpr uint32_t SB = KH + 16384;     // bf16 Sb [128 dk rows][128 dv], MN-major
    static constexpr uint32_t AG = SB + 32768;     // bf16 Ag [64 q][64 k]
    static constexpr uint32_t QTR = AG + 8192;     // 2 x Qt^T receive slots
    static constexpr uint32_t O = QTR + 32768;     // bf16 O tile [64 tok][128] (two boxes)
    static constexpr uint32_t END = O + 16384;
};
constexpr uint32_t TILES_END = GlaLayout::END > CovLayout::END ? GlaLayout::END : CovLayout::END;

struct Aux {
    uint64_t full[2], empty[2];                    // TMA stages
    uint64_t b_aqk, b_p, b_c, b_c0, b_ahat;        // CTA 0
    uint64_t qt_empty[2];                          // CTA 0: receive slot freed by CTA 1
    uint64_t qt_full[2];                           // CTA 1: Qt^T arrived
    uint64_t b_ops, b_stage1, b_ag, b_o;           // CTA 1
    uint32_t tmem_base;
    int abort;
    float m[D];                                    // CTA 0: running key sum
    float w[D];                                    // CTA 0: gate weights of this head
    float tokA[L], tokS[L];                        // CTA 0: lambda_i/t_i, s_i/t_i
};
constexpr size_t SMEM_BYTES = 1024 + TILES_END + sizeof(Aux);

// TMEM columns (512 allocated)
constexpr uint32_t C_COL = 0, AQK_COL = 128, P_COL = 256;   // CTA 0
constexpr uint32_t S_COL = 0, AG_COL = 128, O_COL = 256;    // CTA 1
constexpr uint32_t TMEM_COLS = 512;

struct Args {
    CUtensorMap mq, mk, mv, mla, mo;
    CcqParams p;
};

__device__ __forceinline__ float bf16_at(const uint8_t *tile, int r, int c, int rows) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + sw128_off(r, c, rows)));
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ void store8(uint8_t *dst, const float (&v)[8]) {
    *reinterpret_cast<uint4 *>(dst) =
        make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
}
__device__ __forceinline__ void unpack8(uint4 u, float (&v)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        v[2 * e] = __uint_as_float(w[e] << 16);
        v[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
}
// Named barrier 1 over the 128 element-wise threads (warps 0-3) that also ORs a failure
// flag, so every thread leaves the chunk loop together.
__device__ __forceinline__ bool epi_sync_any(bool fail) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n"
        " bar.red.or.pred po, 1, 128, pi;\n selp.u32 %0, 1, 0, po;\n}"
        : "=r"(r)
        : "r"((uint32_t)fail)
        : "memory");
    return r != 0;
}

// Instruction descriptors used below (bf16 x bf16 -> fp32).
constexpr uint32_t ID_M64N64_KK = idesc_bf16(64, 64, 0, 0);
constexpr uint32_t ID_M64N64_MM = idesc_bf16(64, 64, 1, 1);
constexpr uint32_t ID_M128N64_KK = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_M128N64_MK = idesc_bf16(128, 64, 1, 0);
constexpr uint32_t ID_M128N64_MM = idesc_bf16(128, 64, 1, 1);
constexpr uint32_t ID_M128N128_MM = idesc_bf16(128, 128, 1, 1);
constexpr uint32_t ID_M128N128_KM = idesc_bf16(128, 128, 0, 1);

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
tc_gla_kernel(const __grid_constant__ Args args) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Aux &aux = *reinterpret_cast<Aux *>(smem + TILES_END);
    const CcqParams &p = args.p;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int bh = blockIdx.x >> 1, h = bh % p.H;
    const int T = p.T;
    const int nch = (T + L - 1) / L;
    const uint32_t lane_base = (uint32_t)(warp & 3) * 32u;
    volatile int *abort = &aux.abort;

    // ------------------------------------------------------------ set-up
    if (tid == 0) {
        aux.abort = 0;
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&aux.full[s]), 1);
            mbar_init(smem_u32(&aux.empty[s]), 2);
            mbar_init(smem_u32(&aux.qt_empty[s]), 1);
            mbar_init(smem_u32(&aux.qt_full[s]), 1);
        }
        mbar_init(smem_u32(&aux.b_aqk), 1);
        mbar_init(smem_u32(&aux.b_p), 1);
        mbar_init(smem_u32(&aux.b_c), 1);
        mbar_init(smem_u32(&aux.b_c0), 1);
        mbar_init(smem_u32(&aux.b_ahat), 1);
        mbar_init(smem_u32(&aux.b_ops), 1);
        mbar_init(smem_u32(&aux.b_stage1), 1);
        mbar_init(smem_u32(&aux.b_ag), 1);
        mbar_init(smem_u32(&aux.b_o), 1);
        fence_mbar_init();
    }
    if (rank == 0 && tid < D) {
        aux.m[tid] = p.m0 ? p.m0[(size_t)bh * D + tid] : 0.f;
        aux.w[tid] = p.lambda_in ? 0.f : p.w_lambda[(size_t)h * D + tid];
    }
    if (warp == 4 && lane == 0) {
        prefetch_tensormap(&args.mk);
        prefetch_tensormap(&args.mla);
        prefetch_tensormap(rank == 0 ? &args.mq : &args.mv);
        if (rank == 1) prefetch_tensormap(&args.mo);
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(&aux.tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync();  // barriers of both CTAs initialised before any peer traffic
    tc_fence_after();
    const uint32_t tmem = aux.tmem_base;
    const float b_lam = p.lambda_in ? 0.f : p.b_lambda[h];

    if (rank == 0) {
        // ============================================================ CTA 0
        if (warp == 4) {
            if (lane == 0) {  // ---- TMA producer: Q, K, log alpha
                for (int n = 0; n < nch; ++n) {
                    const int s = n & 1;
                    if (n >= 2 && !mbar_wait(smem_u32(&aux.empty[s]), ((n >> 1) - 1) & 1, abort))
                        break;
                    const uint32_t fb = smem_u32(&aux.full[s]);
                    mbar_expect_tx(fb, 3 * TILE);
                    for (int b = 0; b < 2; ++b) {
                        tma_load_3d(smem_u32(smem + CovLayout::Q + s * TILE + b * BOX), &args.mq,
                                    fb, b * 64, n * L, bh);
                        tma_load_3d(smem_u32(smem + CovLayout::K + s * TILE + b * BOX), &args.mk,
                                    fb, b * 64, n * L, bh);
                        tma_load_3d(smem_u32(smem + CovLayout::LA + s * TILE + b * BOX),
                                    &args.mla, fb, b * 64, n * L, bh);
                    }
                }
            }
            __syncwarp();
        } else if (warp == 5) {
            if (lane == 0) {  // ---- MMA issuer
                for (int n = 0; n < nch; ++n) {
                    const int s = n & 1;
                    if (!mbar_wait(smem_u32(&aux.full[s]), (n >> 1) & 1, abort)) break;
                    tc_fence_after();
                    const uint32_t sQ = smem_u32(smem + CovLayout::Q + s * TILE);
                    const uint32_t sK = smem_u32(smem + CovLayout::K + s * TILE);
                    // A = Q K^T
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        uint32_t off = (ks >> 2) * BOX + (ks & 3) * 32;
                        mma_bf16(tmem + AQK_COL, sw128_desc(sQ + off, 0, 1024),
                                 sw128_desc(sK + off, 0, 1024), ID_M64N64_KK, ks > 0);
                    }
                    mma_commit(smem_u32(&aux.b_aqk));
                    if (!mbar_wait(smem_u32(&aux.b_c0), n & 1, abort)) break;
                    tc_fence_after();
                    // P^T = C0 Q^T
                    const uint32_t sC0 = smem_u32(smem + CovLayout::C0);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        mma_bf16(tmem + P_COL,
                                 sw128_desc(sC0 + (ks >> 2) * 16384 + (ks & 3) * 32, 0, 1024),
                                 sw128_desc(sQ + (ks >> 2) * BOX + (ks & 3) * 32, 0, 1024),
                                 ID_M128N64_KK, ks > 0);
                    }
                    // C += K^T K
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        uint64_t dk = sw128_desc(sK + ks * 2048, BOX, 1024);
                        mma_bf16(tmem + C_COL, dk, dk, ID_M128N128_MM, 1);
                    }
                    mma_commit(smem_u32(&aux.b_c));
                    if (!mbar_wait(smem_u32(&aux.b_ahat), n & 1, abort)) break;
                    tc_fence_after();
                    // P^T += K^T Ah^T
                    const uint32_t sAH = smem_u32(smem + CovLayout::AH);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        mma_bf16(tmem + P_COL, sw128_desc(sK + ks * 2048, BOX, 1024),
                                 sw128_desc(sAH + ks * 32, 0, 1024), ID_M128N64_MK, 1);
                    }
                    mma_commit(smem_u32(&aux.b_p));
                    mma_commit(smem_u32(&aux.empty[s]));
                }
            }
            __syncwarp();
        } else {
            // ---- element-wise threads: thread c <-> TMEM lane c <-> channel c
            const int c = tid;
            bool fail = false;
            for (int n = 0; n < nch && !fail; ++n) {
                const int s = n & 1;
                const int c0t = n * L;
                const int Lc = min(L, T - c0t);
                const uint8_t *sQs = smem + CovLayout::Q + s * TILE;
                const uint8_t *sKs = smem + CovLayout::K + s * TILE;
                const uint8_t *sLAs = smem + CovLayout::LA + s * TILE;

                // ---- C0 operand (bf16) for this chunk; C accumulator initialised at n = 0
                bool ok = true;
                if (n > 0) {
                    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&aux.b_c), (n - 1) & 1, abort));
                    tc_fence_after();
                }
                if (ok) {
#pragma unroll
                    for (int cb = 0; cb < 4; ++cb) {
                        uint32_t r[32];
                        const uint32_t ta = tmem + (lane_base << 16) + C_COL + cb * 32;
                        if (n == 0) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                r[j] = __float_as_uint(
                                    p.C0 ? p.C0[((size_t)bh * D + c) * D + cb * 32 + j] : 0.f);
                            tmem_st32(ta, r);
                        } else {
                            tmem_ld32(ta, r);
                            tmem_ld_wait();
                        }
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            float v[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(r[8 * g + e]);
                            store8(smem + CovLayout::C0 + sw128_chunk(c, cb * 32 + 8 * g, 128), v);
                        }
                    }
                    if (n == 0) tmem_st_wait();
                }
                tc_fence_before();
                fence_async_smem();
                if (epi_sync_any(!ok)) { fail = true; break; }
                if (tid == 0) mbar_arrive(smem_u32(&aux.b_c0));

                // ---- gate, s_i, Ah (one thread per query row: lanes 0-15 of each warp)
                ok = __all_sync(0xffffffffu,
                                mbar_wait(smem_u32(&aux.full[s]), (n >> 1) & 1, abort) &&
                                    mbar_wait(smem_u32(&aux.b_aqk), n & 1, abort));
                tc_fence_after();
                if (ok) {
                    uint32_t a0[32], a1[32];
                    tmem_ld32(tmem + (lane_base << 16) + AQK_COL, a0);
                    tmem_ld32(tmem + (lane_base << 16) + AQK_COL + 32, a1);
                    tmem_ld_wait();
                    if (lane < 16) {
                        const int i = (warp & 3) * 16 + lane;
                        float mq = 0.f, wq = 0.f;
#pragma unroll 4
                        for (int g = 0; g < 16; ++g) {
                            float qv[8];
                            unpack8(*reinterpret_cast<const uint4 *>(sQs + sw128_chunk(i, 8 * g, 64)),
                                    qv);
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                mq += aux.m[8 * g + e] * qv[e];
                                wq += aux.w[8 * g + e] * qv[e];
                            }
                        }
                        float rs = 0.f;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            if (j <= i) rs += __uint_as_float(a0[j]);
                            if (j + 32 <= i) rs += __uint_as_float(a1[j]);
                        }
                        const bool valid = i < Lc;
                        const float t = (float)(p.t0 + (long long)(c0t + i + 1));
                        const float sdt = (mq + rs) / t;
                        float lam = 0.f;
                        if (valid) {
                            size_t ti = (size_t)bh * T + c0t + i;
                            lam = p.lambda_in ? p.lambda_in[ti] : sigmoidf_(wq + b_lam);
                            if (p.lambda_out) p.lambda_out[ti] = lam;
                        }
                        aux.tokA[i] = valid ? lam / t : 0.f;
                        aux.tokS[i] = valid ? sdt : 0.f;
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            float v[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int j = 8 * g + e;
                                const float a = __uint_as_float(j < 32 ? a0[j & 31] : a1[j & 31]);
                                v[e] = (valid && j <= i) ? a - sdt : 0.f;
                            }
                            store8(smem + CovLayout::AH + sw128_chunk(i, 8 * g, 64), v);
                        }
                    }
                }
                tc_fence_before();
                fence_async_smem();
                if (epi_sync_any(!ok)) { fail = true; break; }
                if (tid == 0) mbar_arrive(smem_u32(&aux.b_ahat));

                // ---- cleaned, decay-scaled query Qt^T (thread c = channel c)
                ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&aux.b_p), n & 1, abort));
                tc_fence_after();
                if (ok) {
                    uint32_t p0[32], p1[32];
                    tmem_ld32(tmem + (lane_base << 16) + P_COL, p0);
                    tmem_ld32(tmem + (lane_base << 16) + P_COL + 32, p1);
                    tmem_ld_wait();
                    const float mc = aux.m[c];
                    float E = 0.f, ksum = 0.f;
#pragma unroll
                    for (int g = 7; g >= 0; --g) {
                        float v[8];
#pragma unroll
                        for (int e = 7; e >= 0; --e) {
                            const int i = 8 * g + e;
                            const float la = bf16_at(sLAs, i, c, 64);
                            const float qv = bf16_at(sQs, i, c, 64);
                            const float P = __uint_as_float(i < 32 ? p0[i & 31] : p1[i & 31]);
                            const float qc = qv - aux.tokA[i] * (P - aux.tokS[i] * mc);
                            v[e] = qc * __expf(-E);
                            E += la;
                            ksum += bf16_at(sKs, i, c, 64);
                        }
                        store8(smem + CovLayout::QT + sw128_chunk(c, 8 * g, 128), v);
                    }
                    if (E < -80.f) record_status(p.status, CCQ_ERR_RANGE);
                    aux.m[c] = mc + ksum;
                }
                fence_async_smem();
                if (epi_sync_any(!ok)) { fail = true; break; }
                if (tid == 0) {
                    mbar_arrive(smem_u32(&aux.empty[s]));
                    const int slot = n & 1;
                    bool sent = true;
                    if (n >= 2)
                        sent = mbar_wait(smem_u32(&aux.qt_empty[slot]), ((n >> 1) - 1) & 1, abort,
                                         true);
                    if (sent) {
                        const uint32_t rfull = mapa(smem_u32(&aux.qt_full[slot]), 1);
                        const uint32_t rdst =
                            mapa(smem_u32(smem + GlaLayout::QTR + slot * 16384), 1);
                        mbar_expect_tx_cluster(rfull, 16384);
                        bulk_copy_to_peer(rdst, smem_u32(smem + CovLayout::QT), 16384, rfull);
                        bulk_commit();
                        bulk_wait_read0();
                    } else {
                        *abort = 1;
                    }
                }
            }
            // ---- final state: C (TMEM) and m
            if (!fail && nch > 0) {
                bool ok = __all_sync(0xffffffffu,
                                     mbar_wait(smem_u32(&aux.b_c), (nch - 1) & 1, abort));
                tc_fence_after();
                if (ok && p.C_out) {
#pragma unroll
                    for (int cb = 0; cb < 4; ++cb) {
                        uint32_t r[32];
                        tmem_ld32(tmem + (lane_base << 16) + C_COL + cb * 32, r);
                        tmem_ld_wait();
                        float4 *dst = reinterpret_cast<float4 *>(
                            p.C_out + ((size_t)bh * D + c) * D + cb * 32);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                 __uint_as_float(r[4 * j + 2]),
                                                 __uint_as_float(r[4 * j + 3]));
                    }
                }
                epi_sync_any(false);
                if (ok && p.m_out) p.m_out[(size_t)bh * D + c] = aux.m[c];
            }
        }
    } else {
        // ============================================================ CTA 1
        if (warp == 4) {
            if (lane == 0) {  // ---- TMA producer: K, log alpha, V
                for (int n = 0; n < nch; ++n) {
                    const int s = n & 1;
                    if (n >= 2 && !mbar_wait(smem_u32(&aux.empty[s]), ((n >> 1) - 1) & 1, abort))
                        break;
                    const uint32_t fb = smem_u32(&aux.full[s]);
                    mbar_expect_tx(fb, 3 * TILE);
                    for (int b = 0; b < 2; ++b) {
                        tma_load_3d(smem_u32(smem + GlaLayout::K + s * TILE + b * BOX), &args.mk,
                                    fb, b * 64, n * L, bh);
                        tma_load_3d(smem_u32(smem + GlaLayout::LA + s * TILE + b * BOX),
                                    &args.mla, fb, b * 64, n * L, bh);
                        tma_load_3d(smem_u32(smem + GlaLayout::V + s * TILE + b * BOX), &args.mv,
                                    fb, b * 64, n * L, bh);
                    }
                }
            }
            __syncwarp();
        } else if (warp == 5) {
            if (lane == 0) {  // ---- MMA issuer
                for (int n = 0; n < nch; ++n) {
                    const int s = n & 1, slot = n & 1;
                    if (!mbar_wait(smem_u32(&aux.full[s]), (n >> 1) & 1, abort)) break;
                    if (!mbar_wait(smem_u32(&aux.b_ops), n & 1, abort)) break;
                    if (!mbar_wait(smem_u32(&aux.qt_full[slot]), (n >> 1) & 1, abort, true)) break;
                    tc_fence_after();
                    const uint32_t sQT = smem_u32(smem + GlaLayout::QTR + slot * 16384);
                    const uint32_t sKH = smem_u32(smem + GlaLayout::KH);
                    const uint32_t sSB = smem_u32(smem + GlaLayout::SB);
                    const uint32_t sV = smem_u32(smem + GlaLayout::V + s * TILE);
                    const uint32_t sAG = smem_u32(smem + GlaLayout::AG);
                    // Ag = Qt Kh^T   (both operands stored channel-major)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16(tmem + AG_COL, sw128_desc(sQT + ks * 2048, 16384, 1024),
                                 sw128_desc(sKH + ks * 2048, 16384, 1024), ID_M64N64_MM, ks > 0);
                    // O^T = Sb^T Qt^T
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16(tmem + O_COL, sw128_desc(sSB + ks * 2048, 16384, 1024),
                                 sw128_desc(sQT + ks * 2048, 16384, 1024), ID_M128N64_MM, ks > 0);
                    mma_commit(smem_u32(&aux.b_stage1));
                    // S += Kh^T V
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(tmem + S_COL, sw128_desc(sKH + ks * 32, 0, 1024),
                                 sw128_desc(sV + ks * 2048, BOX, 1024), ID_M128N128_KM, 1);
                    if (!mbar_wait(smem_u32(&aux.b_ag), n & 1, abort)) break;
                    tc_fence_after();
                    // O^T += V^T Ag^T
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(tmem + O_COL, sw128_desc(sV + ks * 2048, BOX, 1024),
                                 sw128_desc(sAG + ks * 32, 0, 1024), ID_M128N64_MK, 1);
                    mma_commit(smem_u32(&aux.b_o));
                    mma_commit(smem_u32(&aux.empty[s]));
                }
            }
            __syncwarp();
        } else {
            // ---- element-wise threads: thread c <-> TMEM lane c
            const int c = tid;
            bool fail = false;
            for (int n = 0; n < nch && !fail; ++n) {
                const int s = n & 1;
                const int c0t = n * L;
                const uint8_t *sKs = smem + GlaLayout::K + s * TILE;
                const uint8_t *sLAs = smem + GlaLayout::LA + s * TILE;

                // ---- Kh^T = (K * exp(E))^T and gamma = exp(R); Sb = gamma * S
                bool ok = mbar_wait(smem_u32(&aux.full[s]), (n >> 1) & 1, abort);
                if (n > 0) ok = ok && mbar_wait(smem_u32(&aux.b_o), (n - 1) & 1, abort);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
                if (ok) {
                    float E = 0.f;
#pragma unroll
                    for (int g = 7; g >= 0; --g) {
                        float v[8];
#pragma unroll
                        for (int e = 7; e >= 0; --e) {
                            const int i = 8 * g + e;
                            v[e] = bf16_at(sKs, i, c, 64) * __expf(E);
                            E += bf16_at(sLAs, i, c, 64);
                        }
                        store8(smem + GlaLayout::KH + sw128_chunk(c, 8 * g, 128), v);
                    }
                    if (E < -80.f) record_status(p.status, CCQ_ERR_RANGE);
                    const float gam = __expf(E);
#pragma unroll
                    for (int cb = 0; cb < 4; ++cb) {
                        uint32_t r[32];
                        const uint32_t ta = tmem + (lane_base << 16) + S_COL + cb * 32;
                        if (n == 0) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                r[j] = __float_as_uint(
                                    p.S0 ? p.S0[((size_t)bh * D + c) * D + cb * 32 + j] : 0.f);
                        } else {
                            tmem_ld32(ta, r);
                            tmem_ld_wait();
                        }
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(gam * __uint_as_float(r[j]));
                        tmem_st32(ta, r);
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            float v[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(r[8 * g + e]);
                            store8(smem + GlaLayout::SB + sw128_chunk(c, cb * 32 + 8 * g, 128), v);
                        }
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                fence_async_smem();
                if (epi_sync_any(!ok)) { fail = true; break; }
                if (tid == 0) {
                    mbar_arrive(smem_u32(&aux.b_ops));
                    mbar_arrive(smem_u32(&aux.empty[s]));
                }

                // ---- causal mask of Ag (one thread per query row)
                ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&aux.b_stage1), n & 1, abort));
                tc_fence_after();
                if (ok) {
                    uint32_t a0[32], a1[32];
                    tmem_ld32(tmem + (lane_base << 16) + AG_COL, a0);
                    tmem_ld32(tmem + (lane_base << 16) + AG_COL + 32, a1);
                    tmem_ld_wait();
                    if (lane < 16) {
                        const int i = (warp & 3) * 16 + lane;
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            float v[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int j = 8 * g + e;
                                const float a = __uint_as_float(j < 32 ? a0[j & 31] : a1[j & 31]);
                                v[e] = j <= i ? a : 0.f;
                            }
                            store8(smem + GlaLayout::AG + sw128_chunk(i, 8 * g, 64), v);
                        }
                    }
                }
                tc_fence_before();
                fence_async_smem();
                if (epi_sync_any(!ok)) { fail = true; break; }
                if (tid == 0) {
                    mbar_arrive(smem_u32(&aux.b_ag));
                    mbar_arrive_cluster(mapa(smem_u32(&aux.qt_empty[n & 1]), 0));
                }

                // ---- output tile: O^T lane = d_v channel, columns = tokens
                ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&aux.b_o), n & 1, abort));
                tc_fence_after();
                if (ok) {
                    uint32_t o0[32], o1[32];
                    tmem_ld32(tmem + (lane_base << 16) + O_COL, o0);
                    tmem_ld32(tmem + (lane_base << 16) + O_COL + 32, o1);
                    tmem_ld_wait();
                    uint8_t *sO = smem + GlaLayout::O;
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const float x = __uint_as_float(i < 32 ? o0[i & 31] : o1[i & 31]);
                        *reinterpret_cast<__nv_bfloat16 *>(sO + sw128_off(i, c, 64)) =
                            __float2bfloat16_rn(x);
                    }
                }
                fence_async_smem();
                if (epi_sync_any(!ok)) { fail = true; break; }
                if (tid == 0) {
                    const uint32_t sO = smem_u32(smem + GlaLayout::O);
                    tma_store_3d(&args.mo, sO, 0, c0t, bh);
                    tma_store_3d(&args.mo, sO + BOX, 64, c0t, bh);
                    bulk_commit();
                    bulk_wait_read0();
                }
            }
            // ---- final state S (TMEM)
            if (!fail && nch > 0 && p.S_out) {
                bool ok = __all_sync(0xffffffffu,
                                     mbar_wait(smem_u32(&aux.b_o), (nch - 1) & 1, abort));
                tc_fence_after();
                if (ok) {
#pragma unroll
                    for (int cb = 0; cb < 4; ++cb) {
                        uint32_t r[32];
                        tmem_ld32(tmem + (lane_base << 16) + S_COL + cb * 32, r);
                        tmem_ld_wait();
                        float4 *dst = reinterpret_cast<float4 *>(
                            p.S_out + ((size_t)bh * D + c) * D + cb * 32);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                 __uint_as_float(r[4 * j + 2]),
                                                 __uint_as_float(r[4 * j + 3]));
                    }
                }
            }
            if (tid == 0) bulk_wait0();
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && aux.abort) record_status(p.status, CCQ_ERR_TIMEOUT);
    cluster_sync();  // no peer traffic may target a CTA that has exited
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 3-D view [B*H][T][128] of a bf16 tensor, box [1][64][64], 128-byte swizzle.
static bool make_map(CUtensorMap *m, const void *base, int T, int BH) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)T * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)L, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace tcgla

bool tc_gla_supported(const CcqParams &p) {
    auto al = [](const void *x) { return ((uintptr_t)x & 15u) == 0; };
    return p.dk == tcgla::D && p.dv == tcgla::D && p.T > 0 && p.B * p.H > 0 &&
           !(p.flags & CCQ_FLAG_L2NORM_QK) && al(p.q) && al(p.k) && al(p.v) &&
           al(p.log_alpha) && al(p.o) && (long long)p.B * p.H * 2 < 0x7fffffffLL;
}

cudaError_t launch_tc_gla(const CcqParams &p, cudaStream_t st) {
    using namespace tcgla;
    Args a;
    a.p = p;
    const int BH = p.B * p.H;
    if (!make_map(&a.mq, p.q, p.T, BH) || !make_map(&a.mk, p.k, p.T, BH) ||
        !make_map(&a.mv, p.v, p.T, BH) || !make_map(&a.mla, p.log_alpha, p.T, BH) ||
        !make_map(&a.mo, p.o, p.T, BH))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(tc_gla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    tc_gla_kernel<<<2 * BH, NTHREADS, SMEM_BYTES, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ccq
