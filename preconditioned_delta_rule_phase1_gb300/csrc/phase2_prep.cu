// phase2_prep.cu -- chunk preparation of Phase 2 on the sm_103a tensor cores:
// everything in the chunkwise delta-rule pass that does not depend on the
// state S, for all chunks of all sequences in parallel (gist.science summary
// of arXiv 2605.13473, section 2.1: Phase 2 is the delta-rule chunk pass with
// the preconditioned keys Kt in the Gram matrix and in the scores).
//
// Per chunk of C = 64 tokens, with g the inclusive within-chunk product of
// alpha (g = 1 without decay), G_ij = g_i / g_j:
//   L   = tril(diag(b) (G . K Kt^T), -1)      A  = tril(G . Q Kt^T)
//   X   = (I + L)^-1                          Xb = X diag(b)
//   Kwn = -Xb diag(g) K                       Ae = A Xb
//   Qe  = diag(g) Q + A Kwn
// so that, for the state S entering the chunk, the chunk's residuals and
// outputs are the single stacked product
//   [U; O] = [Xb; Ae] V + [Kwn; Qe] S^T
// and the state leaves as S' = g_C S + U^T diag(g_C / g) Kt.  The kernel
// writes Kwn, Qe, Xb, Ae (bf16) and the gate factors g_C / g and g_C (fp32)
// to the workspace, chunk-padded (rows past T are zero).
//
// One CTA per (chunk, sequence), 288 threads: warps 0-7 compute (epilogues
// out of TMEM and the triangular solve), warp 8 issues the TMA loads and the
// tcgen05 MMAs.  58 KB of shared memory and 128 TMEM columns, so three CTAs
// share an SM and hide each other's latency.
#include "tc_common.cuh"

namespace osdn {
namespace tc {

namespace {

constexpr int kLP = 68;              // fp32 pitch of the solver tile
constexpr int kPrepThreads = 256;    // compute warps 0-7
constexpr int kPrepBlock = 288;      // + the control warp
constexpr uint32_t kPrepCols = 128;  // TMEM columns

struct PrepParams {
    int T;
    const float *beta, *alpha;
    __nv_bfloat16 *kwn, *qe, *xb, *ae;
    float *gk, *gc;
    int *status;
};

// Shared memory: [K;Q] stacked in 128-row blocks of 64 columns (K rows 0-63,
// Q rows 64-127); Kt in 64-row blocks, whose space takes the fp32 solver tile
// L once the Gram product has read Kt, and after the solve Xb and Xb diag(g)
// (bf16); then the masked scores A (bf16).
template <int K>
struct PrepLay {
    static constexpr int kLBytes = C * kLP * 4;
    static constexpr int kKtBytes = C * K * 2;
    static constexpr int kRegion = ((kKtBytes > kLBytes ? kKtBytes : kLBytes) + 1023) / 1024 * 1024;
    static constexpr int oKQ = 0;
    static constexpr int oKt = 128 * K * 2;
    static constexpr int oXb = oKt;
    static constexpr int oXg = oKt + C * C * 2;
    static constexpr int oA = oKt + kRegion;
    static constexpr int kBytes = oA + C * C * 2;
    static constexpr int kAlloc = kBytes + 1024;
};

// --------------------------------------------------------------- mma.sync
__device__ __forceinline__ uint32_t tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// acc (16x8 tile) += A[16 x k] * B[k x 8], fp32 row-major tiles of pitch kLP.
__device__ __forceinline__ void warp_mm(float (&acc)[4], const float *A, const float *B, int k,
                                        int lane) {
    const int g = lane >> 2, tq = lane & 3;
    for (int k0 = 0; k0 < k; k0 += 8) {
        uint32_t a[4];
        a[0] = tf32(A[g * kLP + k0 + tq]);
        a[1] = tf32(A[(g + 8) * kLP + k0 + tq]);
        a[2] = tf32(A[g * kLP + k0 + tq + 4]);
        a[3] = tf32(A[(g + 8) * kLP + k0 + tq + 4]);
        mma_tf32(acc, a, tf32(B[(k0 + tq) * kLP + g]), tf32(B[(k0 + tq + 4) * kLP + g]));
    }
}
__device__ __forceinline__ void warp_store(float *D, const float (&acc)[4], float scale, int lane) {
    const int g = lane >> 2, tq = lane & 3;
    D[g * kLP + 2 * tq] = scale * acc[0];
    D[g * kLP + 2 * tq + 1] = scale * acc[1];
    D[(g + 8) * kLP + 2 * tq] = scale * acc[2];
    D[(g + 8) * kLP + 2 * tq + 1] = scale * acc[3];
}

// X = (I + L)^-1 in place in sL (strictly lower L in, unit lower X out, the
// diagonal written as 1; the upper quadrant rows 0-31 x cols 32-63 is
// scratch).  Recursive doubling: the four 16x16 diagonal blocks by forward
// substitution in fp32 (one thread per column), then X21 = -X22 L21 X11 on
// 16x16 and 32x32 blocks with mma.sync (tf32 inputs, fp32 accumulation).
// Called by the 256 compute threads.
__device__ void solve_unit_lower(float *sL, int pt) {
    const int pw = pt >> 5, lane = pt & 31;
    if (pt < 64) {  // 16x16 diagonal blocks: thread (blk, c) forms column c
        const int blk = pt >> 4, c = pt & 15;
        float *b = sL + 16 * blk * kLP + 16 * blk;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            // x_i = delta_ic - sum_{k<i} L_ik x_k, summed as a tree of 4 partials
            float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < i; ++k) part[k & 3] = fmaf(b[i * kLP + k], x[k], part[k & 3]);
            x[i] = ((i == c) ? 1.0f : 0.0f) - ((part[0] + part[1]) + (part[2] + part[3]));
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 16; ++i) b[i * kLP + c] = x[i];
    }
    ptx::named_bar(1, kPrepThreads);
    // X_10 = -D_1 L_10 D_0 and X_32 = -D_3 L_32 D_2 on 16x16 blocks (warps 0 and 1)
    if (pw < 2) {
        const int a = 2 * pw + 1;
        float *Lab = sL + 16 * a * kLP + 16 * (a - 1);
        float *Db = sL + 16 * (a - 1) * kLP + 16 * (a - 1);
        float *Da = sL + 16 * a * kLP + 16 * a;
        float *P = sL + 16 * pw * kLP + 32 + 16 * pw;   // upper quadrant: scratch
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float acc[4] = {0, 0, 0, 0};
            warp_mm(acc, Lab, Db + 8 * nt, 16, lane);
            warp_store(P + 8 * nt, acc, 1.0f, lane);
        }
        __syncwarp();
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float acc[4] = {0, 0, 0, 0};
            warp_mm(acc, Da, P + 8 * nt, 16, lane);
            warp_store(Lab + 8 * nt, acc, -1.0f, lane);
        }
    }
    ptx::named_bar(1, kPrepThreads);
    // X21 = -X22 (L21 X11) on the 32x32 halves; warp (mt, nt) owns a 16x8 tile
    {
        const int mt = pw >> 2, nt = pw & 3;
        float acc[4] = {0, 0, 0, 0};
        warp_mm(acc, sL + (32 + 16 * mt) * kLP, sL + 8 * nt, 32, lane);
        warp_store(sL + 16 * mt * kLP + 32 + 8 * nt, acc, 1.0f, lane);   // P in the upper quadrant
    }
    ptx::named_bar(1, kPrepThreads);
    {
        const int mt = pw >> 2, nt = pw & 3;
        float acc[4] = {0, 0, 0, 0};
        warp_mm(acc, sL + (32 + 16 * mt) * kLP + 32, sL + 32 + 8 * nt, 32, lane);
        warp_store(sL + (32 + 16 * mt) * kLP + 8 * nt, acc, -1.0f, lane);
    }
    ptx::named_bar(1, kPrepThreads);
}

template <int K, bool GATED>
__global__ void __launch_bounds__(kPrepBlock, 3)
chunk_prep_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_kt, PrepParams p) {
    using LY = PrepLay<K>;
    constexpr int NH = K / 2;   // columns of a K-wide M=64 accumulator per thread
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    __shared__ uint64_t bar_full, bar_g, bar_x2, bar_ae, bar_x3, bar_kw, bar_x4, bar_qe;
    __shared__ uint32_t tmem_base_sh;
    __shared__ float sBeta[C], sLg[C];
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j = blockIdx.x, seq = blockIdx.y, nch = gridDim.x;
    const int T = p.T, t0 = j * C, Tp = nch * C;
    const int nvalid = min(C, T - t0);
    uint8_t *sKQ = smem + LY::oKQ, *sKt = smem + LY::oKt, *sA = smem + LY::oA;
    uint8_t *sXb = smem + LY::oXb, *sXg = GATED ? smem + LY::oXg : sXb;
    float *sL = reinterpret_cast<float *>(smem + LY::oKt);
    int *st = p.status;
    const size_t row0 = (size_t)seq * Tp + t0;   // first padded row of this chunk

    if (tid == kPrepThreads) {
        uint64_t *all[] = {&bar_full, &bar_g, &bar_x2, &bar_ae, &bar_x3, &bar_kw, &bar_x4, &bar_qe};
        for (uint64_t *b : all) ptx::mbar_init(b, 1);
        ptx::fence_mbar_init();
        s_abort = 0;
    }
    if (warp == 8) {
        ptx::tmem_alloc(&tmem_base_sh, kPrepCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 8) {
        // ============================================ TMA + MMA (one thread)
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(&bar_full, 3 * C * K * 2);
#pragma unroll
            for (int cb = 0; cb < K / 64; ++cb) {
                ptx::tma_load_3d(sKQ + cb * 16384, &tm_k, &bar_full, cb * 64, t0, seq);
                ptx::tma_load_3d(sKQ + cb * 16384 + 8192, &tm_q, &bar_full, cb * 64, t0, seq);
                ptx::tma_load_3d(sKt + cb * 8192, &tm_kt, &bar_full, cb * 64, t0, seq);
            }
            uint64_t *last = &bar_full;   // completes once everything issued so far has
            const uint32_t aKQ = ptx::smem_u32(sKQ), aKt = ptx::smem_u32(sKt);
            const uint32_t aA = ptx::smem_u32(sA), aXb = ptx::smem_u32(sXb), aXg = ptx::smem_u32(sXg);
            bool ok = wait_bar(&bar_full, 0, &s_abort, st);
            if (ok) {  // [K;Q] Kt^T (M=128): Gram rows 0-63, scores rows 64-127
                ptx::tc_fence_after();
                const uint32_t id = ptx::idesc_bf16(128, 64, 0, 0);
                const uint64_t da = dk0(aKQ), db = dk0(aKt);
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks)
                    ptx::umma_bf16(tmem, da + koff(128, ks), db + koff(C, ks), id, ks > 0);
                ptx::umma_commit(&bar_g);
                last = &bar_g;
            }
            ok = ok && wait_bar(&bar_x2, 0, &s_abort, st);
            if (ok) {  // Ae = A Xb
                ptx::tc_fence_after();
                const uint32_t id = ptx::idesc_bf16(64, 64, 0, 1);
                const uint64_t da = dk0(aA), db = dmn0(aXb, 8192);
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    ptx::umma_bf16(tmem, da + koff(C, ks), db + mnoff(ks), id, ks > 0);
                ptx::umma_commit(&bar_ae);
                last = &bar_ae;
            }
            ok = ok && wait_bar(&bar_x3, 0, &s_abort, st);
            if (ok) {  // Kw = Xb diag(g) K  (K read as an MN-major operand)
                ptx::tc_fence_after();
                const uint32_t id = ptx::idesc_bf16(64, K, 0, 1);
                const uint64_t da = dk0(aXg), db = dmn0(aKQ, 16384);
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    ptx::umma_bf16(tmem, da + koff(C, ks), db + mnoff(ks), id, ks > 0);
                ptx::umma_commit(&bar_kw);
                last = &bar_kw;
            }
            ok = ok && wait_bar(&bar_x4, 0, &s_abort, st);
            if (ok) {  // A Kwn  (Kwn written over the K rows)
                ptx::tc_fence_after();
                const uint32_t id = ptx::idesc_bf16(64, K, 0, 1);
                const uint64_t da = dk0(aA), db = dmn0(aKQ, 16384);
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    ptx::umma_bf16(tmem, da + koff(C, ks), db + mnoff(ks), id, ks > 0);
                ptx::umma_commit(&bar_qe);
                last = &bar_qe;
            }
            // the copies and products this CTA started land before it exits
            drain_bar(&bar_full, 0);
            drain_bar(last, 0);
        }
        __syncwarp();
    } else {
        // ============================================ compute warps 0-7
        const int pt = tid, q4 = warp & 3, half = warp >> 2;
        const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
        if (warp == 0) {
            // beta (0 past T) and the inclusive cumulative log alpha, two tokens a lane
            float bb[2], lg[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int i = 2 * lane + e;
                const bool valid = i < nvalid;
                bb[e] = valid ? p.beta[(size_t)seq * T + t0 + i] : 0.0f;
                lg[e] = (GATED && valid) ? logf(p.alpha[(size_t)seq * T + t0 + i]) : 0.0f;
            }
            float sc = lg[0] + lg[1];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(kFullMask, sc, off);
                if (lane >= off) sc += y;
            }
            const float excl = sc - (lg[0] + lg[1]);
            sBeta[2 * lane] = bb[0];
            sBeta[2 * lane + 1] = bb[1];
            sLg[2 * lane] = excl + lg[0];
            sLg[2 * lane + 1] = excl + lg[0] + lg[1];
        }
        ptx::named_bar(1, kPrepThreads);
        if (GATED && pt < C) {
            // tokens past T add nothing to the log, so sLg[C-1] is the chunk's total
            const float lgC = sLg[C - 1];
            p.gk[row0 + pt] = (pt < nvalid) ? __expf(lgC - sLg[pt]) : 0.0f;
            if (pt == 0) p.gc[(size_t)seq * nch + j] = __expf(lgC);
        }

        // ---- Gram / scores: L (fp32) over Kt's space, A (bf16) for the MMAs
        bool ok = vote_all(wait_bar(&bar_g, 0, &s_abort, st), 1, kPrepThreads);
        if (ok) {
            ptx::tc_fence_after();
            float g[32];
            tmem_ld32(tmem + lane_off + 32 * half, g);
            const int grow = 32 * q4 + lane;
            if (grow < C) {  // L = tril(diag(beta) (G . K Kt^T), -1)
                const int i = grow;
                const float bi = sBeta[i], lgi = sLg[i];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int col = 32 * half + jj;
                    float val = 0.0f;
                    if (col < i) val = bi * (GATED ? __expf(lgi - sLg[col]) : 1.0f) * g[jj];
                    sL[i * kLP + col] = val;
                }
            } else {  // A = tril(G . Q Kt^T)
                const int t = grow - C;
                const float lgt = sLg[t];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int col = 32 * half + jj;
                    g[jj] = (col <= t) ? (GATED ? __expf(lgt - sLg[col]) : 1.0f) * g[jj] : 0.0f;
                }
                st_row_sw128(sA, C, t, 32 * half, g, 32);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_bar(1, kPrepThreads);
            solve_unit_lower(sL, pt);
            // ---- Xb = X diag(beta) (global and shared), Xb diag(g) (shared)
            const int t = pt >> 2, s0 = 16 * (pt & 3);
            float xb[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int s = s0 + e;
                xb[e] = (s <= t) ? sL[t * kLP + s] * sBeta[s] : 0.0f;
            }
            ptx::named_bar(1, kPrepThreads);   // L fully read before Xb overwrites it
            st_global_bf16(p.xb + (row0 + t) * C + s0, xb, 16);
            st_row_sw128(sXb, C, t, s0, xb, 16);
            if (GATED) {
#pragma unroll
                for (int e = 0; e < 16; ++e) xb[e] *= __expf(sLg[s0 + e]);
                st_row_sw128(sXg, C, t, s0, xb, 16);
            }
            ptx::fence_proxy_async_smem();
            ptx::named_bar(1, kPrepThreads);
            if (pt == 0) ptx::mbar_arrive(&bar_x2);
        }
        // M=64 accumulators: row 16*q4 + lane (lanes 0-15 of each quarter)
        const int mrow = 16 * q4 + lane;
        const bool act = lane < 16;
        // ---- Ae out of TMEM
        if (ok) ok = vote_all(wait_bar(&bar_ae, 0, &s_abort, st), 1, kPrepThreads);
        if (ok) {
            ptx::tc_fence_after();
            float a[32];
            tmem_ld32(tmem + lane_off + 32 * half, a);
            if (act) st_global_bf16(p.ae + (row0 + mrow) * C + 32 * half, a, 32);
            ptx::tc_fence_before();
            ptx::named_bar(1, kPrepThreads);
            if (pt == 0) ptx::mbar_arrive(&bar_x3);
        }
        // ---- Kwn = -Kw: to the workspace and over the K rows (B operand of A Kwn)
        if (ok) ok = vote_all(wait_bar(&bar_kw, 0, &s_abort, st), 1, kPrepThreads);
        if (ok) {
            ptx::tc_fence_after();
#pragma unroll
            for (int c = 0; c < NH; c += 16) {
                float w[16];
                ptx::tmem_ld16(tmem + lane_off + half * NH + c, w);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) w[e] = -w[e];
                if (act) {
                    st_global_bf16(p.kwn + (row0 + mrow) * K + half * NH + c, w, 16);
                    st_row_sw128(sKQ, 128, mrow, half * NH + c, w, 16);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_bar(1, kPrepThreads);
            if (pt == 0) ptx::mbar_arrive(&bar_x4);
        }
        // ---- Qe = diag(g) Q + A Kwn
        if (ok) ok = vote_all(wait_bar(&bar_qe, 0, &s_abort, st), 1, kPrepThreads);
        if (ok) {
            ptx::tc_fence_after();
            const float gt = GATED ? __expf(sLg[mrow]) : 1.0f;
#pragma unroll
            for (int c = 0; c < NH; c += 16) {
                float d[16], qv[16];
                ptx::tmem_ld16(tmem + lane_off + half * NH + c, d);
                ptx::tmem_wait_ld();
                if (act) {
                    ld_row_sw128(sKQ, 128, C + mrow, half * NH + c, qv, 16);
#pragma unroll
                    for (int e = 0; e < 16; ++e) d[e] = fmaf(gt, qv[e], d[e]);
                    st_global_bf16(p.qe + (row0 + mrow) * K + half * NH + c, d, 16);
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 8) ptx::tmem_dealloc(tmem, kPrepCols);
}

template <int K, bool GATED>
cudaError_t prep_launch_t(int BH, int T, const void *q, const void *k, const void *kt,
                          const float *beta, const float *alpha, __nv_bfloat16 *kwn,
                          __nv_bfloat16 *qe, __nv_bfloat16 *xb, __nv_bfloat16 *ae, float *gk,
                          float *gc, int *status, cudaStream_t stream) {
    CUtensorMap mk, mq, mkt;
    if (!make_map(&mk, k, BH, T, K) || !make_map(&mq, q, BH, T, K) || !make_map(&mkt, kt, BH, T, K))
        return cudaErrorInvalidValue;
    constexpr int smem = PrepLay<K>::kAlloc;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel<K, GATED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    PrepParams p;
    p.T = T;
    p.beta = beta;
    p.alpha = alpha;
    p.kwn = kwn;
    p.qe = qe;
    p.xb = xb;
    p.ae = ae;
    p.gk = gk;
    p.gc = gc;
    p.status = status;
    dim3 grid((T + C - 1) / C, BH);
    chunk_prep_kernel<K, GATED><<<grid, kPrepBlock, smem, stream>>>(mk, mq, mkt, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t chunk_prep_launch(int BH, int T, int K, const void *q, const void *k, const void *kt,
                              const float *beta, const float *alpha, __nv_bfloat16 *kwn,
                              __nv_bfloat16 *qe, __nv_bfloat16 *xb, __nv_bfloat16 *ae, float *gk,
                              float *gc, int *status, cudaStream_t stream) {
    if (K == 128) {
        if (alpha)
            return prep_launch_t<128, true>(BH, T, q, k, kt, beta, alpha, kwn, qe, xb, ae, gk, gc, status, stream);
        return prep_launch_t<128, false>(BH, T, q, k, kt, beta, alpha, kwn, qe, xb, ae, gk, gc, status, stream);
    }
    if (alpha)
        return prep_launch_t<64, true>(BH, T, q, k, kt, beta, alpha, kwn, qe, xb, ae, gk, gc, status, stream);
    return prep_launch_t<64, false>(BH, T, q, k, kt, beta, alpha, kwn, qe, xb, ae, gk, gc, status, stream);
}

}  // namespace tc
}  // namespace osdn
