// phase2_tc.cu -- Phase 2 of OSDN on the sm_103a tensor cores (tcgen05 +
// TMEM + TMA): the chunkwise delta-rule pass with the stored keys replaced by
// the preconditioned keys Ktilde in the chunk Gram matrix and in the
// intra-chunk scores (gist.science summary of arXiv 2605.13473, section 2.1).
//
// Recurrence (per sequence):  S_t = a_t S_{t-1} + b_t (v_t - a_t S_{t-1} k_t) kt_t^T,
//                             o_t = S_t q_t        (a = alpha, b = beta, kt = ktilde)
// Per chunk of C = 64 tokens, with g the inclusive within-chunk product of
// alpha (g = 1 without decay), G_ij = g_i / g_j and S the state entering the
// chunk:
//   L  = tril(diag(b) (G . K Kt^T), -1),   X = (I + L)^-1
//   U  = X diag(b) V - X diag(b g) K S^T           (the chunk's scaled residuals)
//   O  = diag(g) Q S^T + tril(G . Q Kt^T) U
//   S' = g_C S + U^T diag(g_C / g) Kt
//
// Work split: one CTA per (sequence, 64-row slice of S); 256 threads.  The
// state slice lives in fp32 registers of the epilogue threads and in a bf16
// copy in shared memory that feeds the MMAs; nothing of it leaves the SM
// between chunks.  Products on the tensor cores, all bf16 x bf16 -> fp32 in
// TMEM (M = rows of the accumulator):
//   [K;Q] Kt^T   M=128 N=64   Gram (rows 0-63) and scores (rows 64-127)
//   S Q^T        M=64  N=64   the inter-chunk part of O (transposed)
//   K^T Xh^T     M=K   N=64   Kw^T, Xh = X diag(b g)
//   V^T Xb^T     M=64  N=64   initialises U^T, Xb = X diag(b)
//   -S Kw^T      M=64  N=64   accumulates U^T = (XbV - Kw S^T)^T
//   Uh^T Kt      M=64  N=K    state increment, Uh = diag(g_C/g) U
//   U^T A^T      M=64  N=64   the intra-chunk part of O, A = tril(G . Q Kt^T)
// The unit lower-triangular inverse X is formed in fp32 by 16x16 blocks.
// Input tiles (Q, K, Kt, V) arrive by TMA with 128-byte swizzle, double
// buffered so the next chunk streams in while this one computes.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "osdn_device.cuh"
#include "ptx.cuh"

namespace osdn {
namespace tc {

constexpr int C = 64;          // tokens per chunk
constexpr int BV = 64;         // rows of S per CTA
constexpr int kThreads = 256;
constexpr int kLP = 65;        // fp32 pitch of the solver tiles
constexpr uint32_t kWaitLimit = 1u << 22;

// TMEM columns of the accumulators
constexpr uint32_t kColG = 0, kColKw = 64, kColU = 128, kColO1 = 192, kColO2 = 256, kColDS = 320;
constexpr uint32_t kTmemCols = 512;

template <int K>
struct Smem {
    // input stage (double buffered)
    static constexpr int kKQ = 128 * K * 2;   // [K;Q] rows, K/64 blocks of 128 rows x 128 B
    static constexpr int kKt = C * K * 2;     // Ktilde
    static constexpr int kV = C * BV * 2;     // value slice
    static constexpr int kStage = kKQ + kKt + kV;
    // per-chunk operand tiles
    static constexpr int oStage0 = 0;
    static constexpr int oStage1 = kStage;
    static constexpr int oXh = 2 * kStage;
    static constexpr int oXb = oXh + C * C * 2;
    static constexpr int oA = oXb + C * C * 2;
    static constexpr int oKw = oA + C * C * 2;        // K rows x 128 B
    static constexpr int oS = oKw + K * 128;          // BV rows, K/64 blocks of 8 KB
    static constexpr int oU = oS + BV * K * 2;
    static constexpr int oUh = oU + BV * C * 2;
    static constexpr int oL = oUh + BV * C * 2;       // fp32 64 x 65
    static constexpr int oX = oL + C * kLP * 4;
    static constexpr int kBytes = oX + C * kLP * 4;
    static constexpr int kAlloc = kBytes + 1024;      // slack for 1024-byte alignment
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Store n (multiple of 8) consecutive bf16 values of row r, columns
// [c0, c0+n) inside one 64-column block, into a 128B-swizzled K-major tile
// whose blocks hold `rows` rows.
__device__ __forceinline__ void st_row_sw128(uint8_t *tile, int rows, int r, int c0,
                                             const float *vals, int n) {
    uint8_t *rowp = tile + (c0 >> 6) * rows * 128 + r * 128;
    const int cb = (c0 & 63) >> 3;
#pragma unroll 4
    for (int i = 0; i < n; i += 8) {
        uint4 pk;
        pk.x = pack_bf16x2(vals[i + 0], vals[i + 1]);
        pk.y = pack_bf16x2(vals[i + 2], vals[i + 3]);
        pk.z = pack_bf16x2(vals[i + 4], vals[i + 5]);
        pk.w = pack_bf16x2(vals[i + 6], vals[i + 7]);
        const int chunk = (cb + (i >> 3)) ^ (r & 7);
        *reinterpret_cast<uint4 *>(rowp + chunk * 16) = pk;
    }
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    float a[16], b[16];
    ptx::tmem_ld16(taddr, a);
    ptx::tmem_ld16(taddr + 16, b);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[i] = a[i];
        v[16 + i] = b[i];
    }
}

// K-major operand, 128B swizzle: k-slice ks (16 elements) of a tile whose
// 64-column blocks hold `rows` rows.
__device__ __forceinline__ uint64_t desc_k(uint32_t base, int rows, int ks) {
    return ptx::sdesc(base + (ks >> 2) * rows * 128 + (ks & 3) * 32, 16, 1024, 2);
}
// MN-major operand, 128B swizzle: k-slice ks (16 rows of the stored tile);
// consecutive 64-element MN blocks are `block_bytes` apart.
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, int block_bytes, int ks) {
    return ptx::sdesc(base + ks * 2048, block_bytes, 1024, 2);
}

struct Params {
    int T, V, nchunks;
    const float *beta, *alpha, *S0;
    __nv_bfloat16 *o;
    float *ST;
    int *status;
};

template <int K, bool GATED>
__global__ void __launch_bounds__(kThreads, 1)
delta_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_v,
                Params p) {
    using SM = Smem<K>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_full[2], bar_mma;
    __shared__ uint32_t tmem_base_sh;
    __shared__ float sBeta[C], sLg[C];
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, half = warp >> 2;      // TMEM lane quarter, column half
    const int seq = blockIdx.y, v0 = blockIdx.x * BV;
    const int T = p.T;

    uint8_t *sXh = smem + SM::oXh, *sXb = smem + SM::oXb, *sA = smem + SM::oA;
    uint8_t *sKw = smem + SM::oKw, *sS = smem + SM::oS, *sU = smem + SM::oU;
    uint8_t *sUh = GATED ? smem + SM::oUh : sU;
    float *sL = reinterpret_cast<float *>(smem + SM::oL);
    float *sX = reinterpret_cast<float *>(smem + SM::oX);

    if (tid == 0) {
        ptx::mbar_init(&bar_full[0], 1);
        ptx::mbar_init(&bar_full[1], 1);
        ptx::mbar_init(&bar_mma, 1);
        ptx::fence_mbar_init();
        s_abort = 0;
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_kt);
        ptx::prefetch_tmap(&tm_v);
    }
    if (warp == 0) {
        ptx::tmem_alloc(&tmem_base_sh, kTmemCols);
        ptx::tmem_relinquish();
    }

    // state slice: thread (q4, half, lane < 16) owns row v = 16 q4 + lane,
    // key columns [half K/2, (half+1) K/2)
    constexpr int KH = K / 2;
    const bool srow = lane < 16;
    const int vrow = 16 * q4 + lane;
    float S[KH];
#pragma unroll
    for (int j = 0; j < KH; ++j)
        S[j] = (srow && p.S0) ? p.S0[((size_t)seq * p.V + v0 + vrow) * K + half * KH + j] : 0.0f;
    if (srow) {
#pragma unroll
        for (int j = 0; j < KH; j += 32) st_row_sw128(sS, BV, vrow, half * KH + j, S + j, 32);
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;

    auto stage_ptr = [&](int b) { return smem + (b ? SM::oStage1 : SM::oStage0); };
    auto issue_loads = [&](int chunk, int b) {
        uint8_t *st = stage_ptr(b);
        uint8_t *kq = st, *kt = st + SM::kKQ, *vv = st + SM::kKQ + SM::kKt;
        const int t0 = chunk * C;
        ptx::mbar_arrive_expect_tx(&bar_full[b], SM::kStage);
#pragma unroll
        for (int cb = 0; cb < K / 64; ++cb) {
            ptx::tma_load_3d(kq + cb * 16384, &tm_k, &bar_full[b], cb * 64, t0, seq);
            ptx::tma_load_3d(kq + cb * 16384 + 8192, &tm_q, &bar_full[b], cb * 64, t0, seq);
            ptx::tma_load_3d(kt + cb * 8192, &tm_kt, &bar_full[b], cb * 64, t0, seq);
        }
        ptx::tma_load_3d(vv, &tm_v, &bar_full[b], v0, t0, seq);
    };
    int issued = 0, consumed = -1;  // chunk indices of the loads issued / waited for
    if (tid == 0) issue_loads(0, 0);

    uint32_t mma_phase = 0;
    bool ok = true;
    auto wait_mma = [&]() {
        if (!ptx::mbar_wait(&bar_mma, mma_phase, kWaitLimit)) {
            report_status(p.status, OSDN_ERR_TIMEOUT);
            s_abort = 1;
        }
        mma_phase ^= 1u;
        ptx::tc_fence_after();
    };

    for (int chunk = 0; chunk < p.nchunks && ok; ++chunk) {
        const int b = chunk & 1;
        const int t0 = chunk * C;
        uint8_t *st = stage_ptr(b);
        uint8_t *sKQ = st, *sKt = st + SM::kKQ, *sV = st + SM::kKQ + SM::kKt;
        const uint32_t aKQ = ptx::smem_u32(sKQ), aKt = ptx::smem_u32(sKt), aV = ptx::smem_u32(sV);

        // ---- 1. inputs of this chunk; prefetch the next chunk -------------------
        if (!ptx::mbar_wait(&bar_full[b], (chunk >> 1) & 1, kWaitLimit)) {
            report_status(p.status, OSDN_ERR_TIMEOUT);
            s_abort = 1;
        }
        consumed = chunk;
        if (tid == 0 && chunk + 1 < p.nchunks) {
            issue_loads(chunk + 1, b ^ 1);
            issued = chunk + 1;
        }

        // ---- 2. Gram + scores, and S Q^T (state of the previous chunk) ---------
        if (tid == 0) {
            ptx::tc_fence_after();
            const uint32_t id_g = ptx::idesc_bf16(128, 64, 0, 0);
            const uint32_t id_o = ptx::idesc_bf16(64, 64, 0, 0);
            const uint32_t aS = ptx::smem_u32(sS);
#pragma unroll
            for (int ks = 0; ks < K / 16; ++ks)
                ptx::umma_bf16(tmem + kColG, desc_k(aKQ, 128, ks), desc_k(aKt, 64, ks), id_g, ks > 0);
#pragma unroll
            for (int ks = 0; ks < K / 16; ++ks)
                ptx::umma_bf16(tmem + kColO1, desc_k(aS, BV, ks), desc_k(aKQ + 8192, 128, ks), id_o,
                               ks > 0);
            ptx::umma_commit(&bar_mma);
        }
        // gates of this chunk: beta (0 past the end) and the inclusive cumulative
        // log of alpha (alpha = 1 past the end)
        if (warp == 7) {
            float bb[2], lg[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = t0 + 2 * lane + e;
                const bool valid = t < T;
                bb[e] = valid ? p.beta[(size_t)seq * T + t] : 0.0f;
                lg[e] = (GATED && valid) ? logf(p.alpha[(size_t)seq * T + t]) : 0.0f;
            }
            float s = lg[0] + lg[1];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(kFullMask, s, off);
                if (lane >= off) s += y;
            }
            const float excl = s - (lg[0] + lg[1]);
            sBeta[2 * lane] = bb[0];
            sBeta[2 * lane + 1] = bb[1];
            sLg[2 * lane] = excl + lg[0];
            sLg[2 * lane + 1] = excl + lg[0] + lg[1];
        }
        __syncthreads();
        wait_mma();

        // ---- 3. L (fp32, for the solve) and the masked scores A (bf16) ---------
        {
            float g[32];
            tmem_ld32(tmem + lane_off + kColG + 32 * half, g);
            const int row = 32 * q4 + lane;
            if (row < C) {
                const int i = row;
                const float bi = sBeta[i];
                const float lgi = sLg[i];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = 32 * half + jj;
                    float val = 0.0f;
                    if (j < i) val = bi * (GATED ? __expf(lgi - sLg[j]) : 1.0f) * g[jj];
                    sL[i * kLP + j] = val;
                }
            } else {
                const int t = row - C;
                const float lgt = sLg[t];
                float a[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int s = 32 * half + jj;
                    a[jj] = (s <= t) ? (GATED ? __expf(lgt - sLg[s]) : 1.0f) * g[jj] : 0.0f;
                }
                st_row_sw128(sA, C, t, 32 * half, a, 32);
            }
        }
        ptx::tc_fence_before();
        __syncthreads();

        // ---- 4. X = (I + L)^-1 by 16x16 blocks (fp32) ---------------------------
        if (tid < 64) {  // diagonal blocks: thread (a, c) forms column c of block a
            const int a = tid >> 4, c = tid & 15;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float s = (i == c) ? 1.0f : 0.0f;
#pragma unroll
                for (int k = 0; k < i; ++k) s = fmaf(-sL[(16 * a + i) * kLP + 16 * a + k], x[k], s);
                x[i] = s;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) sX[(16 * a + i) * kLP + 16 * a + c] = x[i];
        }
        __syncthreads();
#pragma unroll 1
        for (int d = 1; d < 4; ++d) {
            const int items = (4 - d) * 256;
            // P_ab = sum_{b <= cc < a} L_a,cc X_cc,b, kept in the (unused) upper block (b, a) of L
            for (int it = tid; it < items; it += kThreads) {
                const int b = it >> 8, a = b + d, r = (it >> 4) & 15, c = it & 15;
                float s = 0.0f;
                for (int cc = b; cc < a; ++cc)
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        s = fmaf(sL[(16 * a + r) * kLP + 16 * cc + k], sX[(16 * cc + k) * kLP + 16 * b + c], s);
                sL[(16 * b + r) * kLP + 16 * a + c] = s;
            }
            __syncthreads();
            // X_ab = -X_aa P_ab
            for (int it = tid; it < items; it += kThreads) {
                const int b = it >> 8, a = b + d, r = (it >> 4) & 15, c = it & 15;
                float s = 0.0f;
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    s = fmaf(sX[(16 * a + r) * kLP + 16 * a + k], sL[(16 * b + k) * kLP + 16 * a + c], s);
                sX[(16 * a + r) * kLP + 16 * b + c] = -s;
            }
            __syncthreads();
        }
        // Xh = X diag(beta g), Xb = X diag(beta): B operands, row t, column s
        {
            const int t = tid >> 2, s0 = 16 * (tid & 3);
            float xh[16], xb[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int s = s0 + e;
                const float x = (s <= t) ? sX[t * kLP + s] : 0.0f;
                xb[e] = x * sBeta[s];
                xh[e] = GATED ? xb[e] * __expf(sLg[s]) : xb[e];
            }
            st_row_sw128(sXb, C, t, s0, xb, 16);
            if (GATED) st_row_sw128(sXh, C, t, s0, xh, 16);
        }
        ptx::fence_proxy_async_smem();
        __syncthreads();

        // ---- 5. Kw^T = K^T Xh^T and U^T <- V^T Xb^T ---------------------------
        if (tid == 0) {
            ptx::tc_fence_after();
            const uint32_t aXh = ptx::smem_u32(GATED ? sXh : sXb), aXb = ptx::smem_u32(sXb);
            const uint32_t id_kw = ptx::idesc_bf16(K, 64, 1, 0);
            const uint32_t id_v = ptx::idesc_bf16(64, 64, 1, 0);
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks)
                ptx::umma_bf16(tmem + kColKw, desc_mn(aKQ, 16384, ks), desc_k(aXh, C, ks), id_kw, ks > 0);
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks)
                ptx::umma_bf16(tmem + kColU, desc_mn(aV, 8192, ks), desc_k(aXb, C, ks), id_v, ks > 0);
            ptx::umma_commit(&bar_mma);
        }
        __syncwarp();
        wait_mma();

        // ---- 6. Kw^T to shared memory (bf16, MN-major B operand) --------------
        {
            float kw[32];
            tmem_ld32(tmem + lane_off + kColKw + 32 * half, kw);
            const int krow = (K == 128) ? 32 * q4 + lane : 16 * q4 + lane;
            if (K == 128 || lane < 16) st_row_sw128(sKw, K, krow, 32 * half, kw, 32);
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();

        // ---- 7. U^T += -S Kw^T ---------------------------------------------------
        if (tid == 0) {
            ptx::tc_fence_after();
            const uint32_t aS = ptx::smem_u32(sS), aKw = ptx::smem_u32(sKw);
            const uint32_t id_u = ptx::idesc_bf16(64, 64, 0, 1, 1);
#pragma unroll
            for (int ks = 0; ks < K / 16; ++ks)
                ptx::umma_bf16(tmem + kColU, desc_k(aS, BV, ks), desc_mn(aKw, 8192, ks), id_u, 1);
            ptx::umma_commit(&bar_mma);
        }
        __syncwarp();
        wait_mma();

        // ---- 8. U^T (and Uh^T = U^T diag(g_C / g)) to shared memory -----------
        {
            float u[32];
            tmem_ld32(tmem + lane_off + kColU + 32 * half, u);
            if (srow) {
                st_row_sw128(sU, BV, vrow, 32 * half, u, 32);
                if (GATED) {
                    const float lgC = sLg[C - 1];
#pragma unroll
                    for (int e = 0; e < 32; ++e) u[e] *= __expf(lgC - sLg[32 * half + e]);
                    st_row_sw128(sUh, BV, vrow, 32 * half, u, 32);
                }
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();

        // ---- 9. dS = Uh^T Kt and O2 = U^T A^T ----------------------------------
        if (tid == 0) {
            ptx::tc_fence_after();
            const uint32_t aU = ptx::smem_u32(sU), aUh = ptx::smem_u32(sUh), aA = ptx::smem_u32(sA);
            const uint32_t id_ds = ptx::idesc_bf16(64, K, 0, 1);
            const uint32_t id_o2 = ptx::idesc_bf16(64, 64, 0, 0);
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks)
                ptx::umma_bf16(tmem + kColDS, desc_k(aUh, BV, ks), desc_mn(aKt, 8192, ks), id_ds, ks > 0);
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks)
                ptx::umma_bf16(tmem + kColO2, desc_k(aU, BV, ks), desc_k(aA, C, ks), id_o2, ks > 0);
            ptx::umma_commit(&bar_mma);
        }
        __syncwarp();
        wait_mma();

        // ---- 10. state carry and output -----------------------------------------
        {
            const float gC = GATED ? __expf(sLg[C - 1]) : 1.0f;
#pragma unroll
            for (int j = 0; j < KH; j += 32) {
                float ds[32];
                tmem_ld32(tmem + lane_off + kColDS + half * KH + j, ds);
#pragma unroll
                for (int e = 0; e < 32; ++e) S[j + e] = fmaf(gC, S[j + e], ds[e]);
                if (srow) st_row_sw128(sS, BV, vrow, half * KH + j, S + j, 32);
            }
            float o1[32], o2[32];
            tmem_ld32(tmem + lane_off + kColO1 + 32 * half, o1);
            tmem_ld32(tmem + lane_off + kColO2 + 32 * half, o2);
            // stage O (t rows, v columns, bf16) in the free L tile
            __nv_bfloat16 *sO = reinterpret_cast<__nv_bfloat16 *>(sL);
            if (srow) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int t = 32 * half + e;
                    const float gt = GATED ? __expf(sLg[t]) : 1.0f;
                    sO[t * BV + vrow] = __float2bfloat16_rn(fmaf(gt, o1[e], o2[e]));
                }
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ok = !__syncthreads_or(s_abort);
        {
            const __nv_bfloat16 *sO = reinterpret_cast<const __nv_bfloat16 *>(sL);
            // 64 rows x 128 bytes: 8 threads per row, 16 bytes each
            const int r = tid >> 3, part = tid & 7;
#pragma unroll
            for (int rr = 0; rr < C; rr += kThreads / 8) {
                const int t = t0 + r + rr;
                if (t < T)
                    *reinterpret_cast<uint4 *>(p.o + ((size_t)seq * T + t) * p.V + v0 + part * 8) =
                        *reinterpret_cast<const uint4 *>(sO + (r + rr) * BV + part * 8);
            }
        }
        __syncthreads();
    }

    // ---- final state ------------------------------------------------------------
    if (p.ST && srow && ok) {
        float *dst = p.ST + ((size_t)seq * p.V + v0 + vrow) * K + half * KH;
#pragma unroll
        for (int j = 0; j < KH; j += 4) *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    // Bulk copies still in flight (only after an abort) must land before exit.
    if (tid == 0 && !ok && issued > consumed)
        ptx::mbar_wait(&bar_full[issued & 1], (issued >> 1) & 1, kWaitLimit);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ----------------------------------------------------------------------- host
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static bool get_encoder() {
    if (g_encode) return true;
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}

// [BH][T][width] bf16, boxes of 64 columns x 64 tokens, 128-byte swizzle;
// tokens past T read as zero.
static bool make_map(CUtensorMap *m, const void *ptr, int BH, int T, int width) {
    cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * (cuuint64_t)T};
    cuuint32_t box[3] = {64, (cuuint32_t)C, 1}, es[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <int K, bool GATED>
static cudaError_t launch(int BH, int T, int V, const void *q, const void *k, const void *kt,
                          const void *v, const float *beta, const float *alpha, const float *S0,
                          void *o, float *ST, int *status, cudaStream_t stream) {
    CUtensorMap mq, mk, mkt, mv;
    if (!make_map(&mq, q, BH, T, K) || !make_map(&mk, k, BH, T, K) ||
        !make_map(&mkt, kt, BH, T, K) || !make_map(&mv, v, BH, T, V))
        return cudaErrorInvalidValue;
    constexpr int smem = Smem<K>::kAlloc;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(delta_tc_kernel<K, GATED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    Params p;
    p.T = T;
    p.V = V;
    p.nchunks = (T + C - 1) / C;
    p.beta = beta;
    p.alpha = alpha;
    p.S0 = S0;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.ST = ST;
    p.status = status;
    dim3 grid(V / BV, BH);
    delta_tc_kernel<K, GATED><<<grid, kThreads, smem, stream>>>(mq, mk, mkt, mv, p);
    return cudaGetLastError();
}

}  // namespace tc

cudaError_t delta_tc_launch(int BH, int T, int K, int V, const void *q, const void *k,
                            const void *kt, const void *v, const float *beta, const float *alpha,
                            const float *S0, void *o, float *ST, int *status, cudaStream_t stream) {
    if (!tc::get_encoder()) return cudaErrorNotSupported;
    if (K == 128) {
        if (alpha) return tc::launch<128, true>(BH, T, V, q, k, kt, v, beta, alpha, S0, o, ST, status, stream);
        return tc::launch<128, false>(BH, T, V, q, k, kt, v, beta, alpha, S0, o, ST, status, stream);
    }
    if (alpha) return tc::launch<64, true>(BH, T, V, q, k, kt, v, beta, alpha, S0, o, ST, status, stream);
    return tc::launch<64, false>(BH, T, V, q, k, kt, v, beta, alpha, S0, o, ST, status, stream);
}

}  // namespace osdn
