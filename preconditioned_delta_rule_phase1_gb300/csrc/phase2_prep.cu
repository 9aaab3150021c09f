// phase2_prep.cu -- chunk preparation of Phase 2 on the sm_103a tensor cores:
// everything in the chunkwise delta-rule pass that does not depend on the
// state S, for all chunks of all sequences in parallel (gist.science summary
// of arXiv 2605.13473, section 2.1: Phase 2 is the delta-rule chunk pass with
// the preconditioned keys Kt in the Gram matrix and in the scores).
//
// Per chunk of C = 64 tokens, with g the inclusive within-chunk product of
// alpha (g = 1 without decay), G_ij = g_i / g_j and D = diag(g_C / g):
//   L  = tril(diag(b) (G . K Kt^T), -1)       A  = tril(G . Q Kt^T)
//   X  = (I + L)^-1,  Xb = X diag(b)          Kw = Xb diag(g) K
//   W  = (D Kt)^T Xb          (K x C)         M  = -(D Kt)^T Kw     (K x K)
//   Ae = A Xb                 (C x C)         Qe = diag(g) Q - A Kw (C x K)
// so that, for the state S entering the chunk (U = Xb V - Kw S^T its scaled
// residuals), the chunk's outputs and the state it leaves are
//   O    = Ae V + Qe S^T
//   S'^T = g_C S^T + W V + M S^T
// -- one product with the state per chunk instead of two dependent ones.
// The kernel writes W, M, Qe, Ae (bf16) and g_C (fp32) to the workspace;
// rows past T are zero.
//
// One CTA per (chunk, sequence), 288 threads: warps 0-7 compute (epilogues
// out of TMEM and the triangular solve), warp 8 issues the TMA loads and the
// tcgen05 MMAs.  The outputs are staged in shared memory in the tensor maps'
// box layout, in tiles the kernel no longer needs, and leave by TMA stores.
// 90 KB of shared memory and 256 TMEM columns: two CTAs share an SM and hide
// each other's latency.  The load warp also prefetches into L2 the K, Q and
// Kt tiles of the CTA one wave (two CTAs per SM) later in launch order, so
// that its loads find them there.
//
// Fused forward pass (template flag FUSED): Kt is not read but rebuilt from
// the preconditioner scan's checkpoints -- d_c, the preconditioner entering
// the chunk, and e_t of every token (d_{t+1} = r_t d_t + e_t w_t, w = k . k):
//   Kt = (rho d_c^T + P W) . K,   P_tu = pi_ut e_u (u < t),   W_u = w_u,
// with rho_t = prod_{v<t} r_v and pi_ut = prod_{u<v<t} r_v inside the chunk.
// P W runs on the tensor cores with P and W each split into a bf16 high
// part and a bf16 remainder (three products: hi.hi + hi.lo + lo.hi), so the
// rebuilt preconditioner carries about 2^-16 relative error instead of the
// 2^-9 of one bf16 product.  The four tiles use space that is dead at that
// point: W over L, its remainder over Xb / Xb diag(g), P over A, its
// remainder over Kt.
//
// Decay per key channel (template flag PCH; S_t = S_{t-1} Diag(alpha_t) +
// ..., alpha_t a K-vector): with Gam_t the within-chunk inclusive product of
// alpha_t (per channel), the Gram and the scores become
//   (Gam_t . k_t) . (kt_s / Gam_s)   and   (Gam_t . q_t) . (kt_s / Gam_s),
// the decay can no longer be factored out of the dot products, and 1/Gam
// would overflow under strong decay.  So each 16-token block b of rows takes
// a reference point m = 16 b - 1 (the token before the block): rows are
// scaled by Gam_t / Gam_m <= 1 and the columns of a copy of Kt by Gam_m /
// Gam_s (<= 1 before the block, at most the product of 16 decays' inverses
// inside it; 0 past it), and four M=128 products, one per reference, fill
// the 256 TMEM columns; row t reads its block's.  Two copies of Kt at a time
// live in the dead L and Xb tiles.  Then K rows are rescaled to Gam . K (for
// Kw), Kt to (Gam_C / Gam_s) . kt (for W and M), Q to Gam . Q inside the Qe
// epilogue, and the chunk's Gam_C goes to the workspace per channel.  The
// decay must lie in [2^-6, 2^6] (every factor then stays inside the fp32 and
// bf16 range); anything else is recorded as OSDN_ERR_DEVICE.  A decay alpha that is not positive and finite (its
// log enters the algebra), or a beta that is not finite, is recorded in the
// status word as OSDN_ERR_DEVICE.
#include "tc_common.cuh"

namespace osdn {
namespace tc {

namespace {

constexpr int kLP = 68;              // fp32 pitch of the solver tile
constexpr int kPrepThreads = 256;    // compute warps 0-7
constexpr int kPrepBlock = 288;      // + the control warp
constexpr uint32_t kPrepCols = 256;  // TMEM columns
constexpr float kMinDecay = 0.015625f, kMaxDecay = 64.0f;   // per-channel decay range (2^-6, 2^6)

// Byte offset of element (r, c) in a 128B-swizzled tile whose 64-column
// blocks hold `rows` rows of 128 bytes (the layout st_row_sw128 writes).
__device__ __forceinline__ int sw_off(int rows, int r, int c) {
    return (c >> 6) * rows * 128 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + ((c & 7) << 1);
}

struct PrepParams {
    int BH, T, nch, c0;   // sequences, sequence length, its chunks, first chunk of this launch
    int ahead;            // CTAs resident at once: the CTA that many later gets its inputs into L2
    const float *beta, *alpha;
    const float *r;       // fused: retention r_t [BH][T], or NULL (r = 1)
    const float *ecoef;   // fused: e_t [BH][T]
    const float *dchk;    // fused: d entering each chunk [BH][nch][K]
    const float *alpha_k; // per-channel decay [BH][T][K] (PCH)
    float *gc;            // g_C per chunk [BH][nch], or per channel [BH][nch][K] (PCH)
    int *status;
};

// Shared memory: [K;Q] stacked in 128-row blocks of 64 columns (K rows 0-63,
// later overwritten by Kw; Q rows 64-127), Kt in 64-row blocks (scaled to
// D Kt in place once the Gram product has read it), the fp32 solver tile L,
// then the bf16 tiles A, Xb and Xb diag(g).
template <int K>
struct PrepLay {
    static constexpr int oKQ = 0;
    static constexpr int oKt = 128 * K * 2;
    static constexpr int oL = oKt + C * K * 2;
    static constexpr int oA = oL + ((C * kLP * 4 + 1023) / 1024) * 1024;
    static constexpr int oXb = oA + C * C * 2;
    static constexpr int oXg = oXb + C * C * 2;
    static constexpr int kBytes = oXg + C * C * 2;
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

template <int K, bool GATED, bool FUSED, bool PCH>
__global__ void __launch_bounds__(kPrepBlock, 2)
chunk_prep_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_w,
                  const __grid_constant__ CUtensorMap tm_m, const __grid_constant__ CUtensorMap tm_qe,
                  const __grid_constant__ CUtensorMap tm_ae, PrepParams p) {
    using LY = PrepLay<K>;
    constexpr int NH = K / 2;   // columns of a K-wide accumulator per thread
    // TMEM columns: Gram; then Kw | W | Ae; then M' | Qe'
    constexpr uint32_t cKw = 0, cW = 128, cAe = 192, cM = 0, cQe = 128;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    __shared__ uint64_t bar_full, bar_g, bar_x2, bar_p1, bar_x3, bar_p2;
    __shared__ uint64_t bar_f0, bar_f1, bar_kt;   // fused: W, P staged; P W done; Kt built
    // per-channel decay: Kt copies 0 and 1 staged, their products done, copies 2, 3 staged
    __shared__ uint64_t bar_c01, bar_r0, bar_r1, bar_c2, bar_c3;
    // per-channel decay: log Gam at the four reference points (0 for block 0)
    // and at the chunk's end, and the per-group partial sums of log alpha
    __shared__ float sLref[PCH ? 4 : 1][PCH ? K : 1], sLamC[PCH ? K : 1];
    __shared__ float sGref[PCH ? 4 : 1][PCH ? K : 1];   // exp(sLref): Gam at the references
    __shared__ float sGrp[PCH ? 512 / K : 1][PCH ? K : 1];
    __shared__ uint32_t tmem_base_sh;
    __shared__ float sBeta[C], sLg[C], sD[C];
    // fused: e_t, r_t, and sPre[b][t] = prod_{16 b <= v < t} r_v (1 for t <= 16 b):
    // sPre[0] is rho, sPre[b] for b > 0 the r products from column block b on
    __shared__ float sE[FUSED ? C : 1], sR[FUSED ? C : 1], sPre[FUSED ? 4 : 1][FUSED ? C : 1];
    __shared__ __align__(16) float sD0[FUSED ? K : 1];
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (grid_seq() >= (size_t)p.BH) return;
    const int j = p.c0 + blockIdx.x, seq = (int)grid_seq(), nch = p.nch;
    const int T = p.T, t0 = j * C;
    const int nvalid = min(C, T - t0);
    uint8_t *sKQ = smem + LY::oKQ, *sKt = smem + LY::oKt, *sA = smem + LY::oA;
    uint8_t *sXb = smem + LY::oXb, *sXg = GATED ? smem + LY::oXg : sXb;
    float *sL = reinterpret_cast<float *>(smem + LY::oL);
    int *st = p.status;
    const int krow0 = j * K;   // this chunk's rows of W and M within the sequence
    // staging of the outputs: W over L; Ae over Xb; M (64x64 boxes) over Kt
    // and the Kw rows of [K;Q]; Qe in place of Q
    uint8_t *sW = smem + LY::oL;
    auto mbox = [&](int rb, int cb) {
        const int i = rb * (K / 64) + cb;
        return i < 2 ? sKt + i * 8192 : sKQ + (i - 2) * 16384;
    };

    if (tid == kPrepThreads) {
        uint64_t *all[] = {&bar_full, &bar_g, &bar_x2, &bar_p1, &bar_x3, &bar_p2,
                           &bar_f0, &bar_f1, &bar_kt, &bar_c01, &bar_r0, &bar_r1, &bar_c2, &bar_c3};
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
            ptx::mbar_arrive_expect_tx(&bar_full, (FUSED ? 2 : 3) * C * K * 2);
#pragma unroll
            for (int cb = 0; cb < K / 64; ++cb) {
                ptx::tma_load_3d(sKQ + cb * 16384, &tm_k, &bar_full, cb * 64, t0, seq);
                ptx::tma_load_3d(sKQ + cb * 16384 + 8192, &tm_q, &bar_full, cb * 64, t0, seq);
                if (!FUSED) ptx::tma_load_3d(sKt + cb * 8192, &tm_kt, &bar_full, cb * 64, t0, seq);
            }
            {   // the inputs of the CTA about one wave later, into L2
                const size_t gx = gridDim.x, gy = gridDim.y;
                const size_t me = blockIdx.x + gx * (blockIdx.y + gy * (size_t)blockIdx.z);
                const size_t later = me + (size_t)p.ahead;
                if (later < gx * gy * gridDim.z) {
                    const size_t yz = later / gx;
                    const int c2 = p.c0 + (int)(later % gx);
                    const int seq2 = (int)(yz % gy + gy * (yz / gy));
                    if (seq2 < p.BH) {
#pragma unroll
                        for (int cb = 0; cb < K / 64; ++cb) {
                            ptx::tma_prefetch_3d(&tm_k, cb * 64, c2 * C, seq2);
                            ptx::tma_prefetch_3d(&tm_q, cb * 64, c2 * C, seq2);
                            if (!FUSED) ptx::tma_prefetch_3d(&tm_kt, cb * 64, c2 * C, seq2);
                        }
                    }
                }
            }
            uint64_t *last = &bar_full;   // completes once everything issued so far has
            const uint32_t aKQ = ptx::smem_u32(sKQ), aKt = ptx::smem_u32(sKt);
            const uint32_t aA = ptx::smem_u32(sA), aXb = ptx::smem_u32(sXb), aXg = ptx::smem_u32(sXg);
            bool ok = wait_poll(&bar_full, 0, &s_abort, st);
            if (FUSED) {
                ok = ok && wait_poll(&bar_f0, 0, &s_abort, st);
                if (ok) {  // P W = Ph Wh + Ph Wl + Pl Wh (M=64, N=K), MN-major W tiles
                    ptx::tc_fence_after();
                    const uint32_t idk = ptx::idesc_bf16(64, K, 0, 1);
                    const uint64_t dPh = dk0(aA), dPl = dk0(aKt);
                    const uint64_t dWh = dmn0(ptx::smem_u32(smem + LY::oL), 8192);
                    const uint64_t dWl = dmn0(aXb, 8192);
#pragma unroll
                    for (int ks = 0; ks < C / 16; ++ks) {
                        ptx::umma_bf16(tmem, dPh + koff(C, ks), dWh + mnoff(ks), idk, ks > 0);
                        ptx::umma_bf16(tmem, dPh + koff(C, ks), dWl + mnoff(ks), idk, 1);
                        ptx::umma_bf16(tmem, dPl + koff(C, ks), dWh + mnoff(ks), idk, 1);
                    }
                    ptx::umma_commit(&bar_f1);
                    last = &bar_f1;
                }
                ok = ok && wait_poll(&bar_kt, 0, &s_abort, st);
            }
            if (ok && PCH) {  // one [K;Q] Kt_b^T product per reference point b (columns 64 b..)
                const uint32_t id = ptx::idesc_bf16(128, 64, 0, 0);
                const uint64_t da = dk0(aKQ);
                const uint64_t dbuf[2] = {dk0(ptx::smem_u32(smem + LY::oL)), dk0(aXb)};
                uint64_t *staged[4] = {&bar_c01, &bar_c01, &bar_c2, &bar_c3};
                uint64_t *done[4] = {&bar_r0, &bar_r1, &bar_g, &bar_g};
                for (int b = 0; b < 4 && ok; ++b) {
                    if (b != 1) ok = wait_poll(staged[b], 0, &s_abort, st);
                    if (!ok) break;
                    ptx::tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < K / 16; ++ks)
                        ptx::umma_bf16(tmem + 64 * b, da + koff(128, ks), dbuf[b & 1] + koff(C, ks), id,
                                       ks > 0);
                    if (b != 2) {
                        ptx::umma_commit(done[b]);
                        last = done[b];
                    }
                }
            } else if (ok) {  // [K;Q] Kt^T (M=128): Gram rows 0-63, scores rows 64-127
                ptx::tc_fence_after();
                const uint32_t id = ptx::idesc_bf16(128, 64, 0, 0);
                const uint64_t da = dk0(aKQ), db = dk0(aKt);
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks)
                    ptx::umma_bf16(tmem, da + koff(128, ks), db + koff(C, ks), id, ks > 0);
                ptx::umma_commit(&bar_g);
                last = &bar_g;
            }
            ok = ok && wait_poll(&bar_x2, 0, &s_abort, st);
            if (ok) {  // Kw = Xb diag(g) K;  W = (D Kt)^T Xb;  Ae = A Xb
                ptx::tc_fence_after();
                const uint32_t idk = ptx::idesc_bf16(64, K, 0, 1);
                const uint32_t idw = ptx::idesc_bf16(K, 64, 1, 1);
                const uint32_t ida = ptx::idesc_bf16(64, 64, 0, 1);
                const uint64_t dXg = dk0(aXg), dK = dmn0(aKQ, 16384), dKt = dmn0(aKt, 8192);
                const uint64_t dXb = dmn0(aXb, 8192), dA = dk0(aA);
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    ptx::umma_bf16(tmem + cKw, dXg + koff(C, ks), dK + mnoff(ks), idk, ks > 0);
                    ptx::umma_bf16(tmem + cW, dKt + mnoff(ks), dXb + mnoff(ks), idw, ks > 0);
                    ptx::umma_bf16(tmem + cAe, dA + koff(C, ks), dXb + mnoff(ks), ida, ks > 0);
                }
                ptx::umma_commit(&bar_p1);
                last = &bar_p1;
            }
            ok = ok && wait_poll(&bar_x3, 0, &s_abort, st);
            if (ok) {  // M' = (D Kt)^T Kw;  Qe' = A Kw  (Kw written over the K rows)
                ptx::tc_fence_after();
                const uint32_t idm = ptx::idesc_bf16(K, K, 1, 1);
                const uint32_t idq = ptx::idesc_bf16(64, K, 0, 1);
                const uint64_t dKt = dmn0(aKt, 8192), dKw = dmn0(aKQ, 16384), dA = dk0(aA);
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    ptx::umma_bf16(tmem + cM, dKt + mnoff(ks), dKw + mnoff(ks), idm, ks > 0);
                    ptx::umma_bf16(tmem + cQe, dA + koff(C, ks), dKw + mnoff(ks), idq, ks > 0);
                }
                ptx::umma_commit(&bar_p2);
                last = &bar_p2;
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
            bool bad = false;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int i = 2 * lane + e;
                const bool valid = i < nvalid;
                bb[e] = valid ? p.beta[(size_t)seq * T + t0 + i] : 0.0f;
                const float a = (GATED && valid) ? p.alpha[(size_t)seq * T + t0 + i] : 1.0f;
                // the chunk algebra takes log alpha: a decay must be positive and finite
                bad |= !isfinite(bb[e]) || !(a > 0.0f) || !isfinite(a);
                lg[e] = (GATED && valid) ? logf(a) : 0.0f;
            }
            if (bad) report_status(p.status, OSDN_ERR_DEVICE);
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
        if (FUSED && warp == 1) {
            // e_t and r_t, two tokens a lane (e = 0 and r = 1 past T), and the
            // exclusive products of r from token 0, 16, 32 and 48 on, by
            // product scans (no division: r may be 0)
            float ee[2], rr[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int i = 2 * lane + e;
                const bool valid = i < nvalid;
                ee[e] = valid ? p.ecoef[(size_t)seq * T + t0 + i] : 0.0f;
                rr[e] = (valid && p.r) ? p.r[(size_t)seq * T + t0 + i] : 1.0f;
            }
            sE[2 * lane] = ee[0];
            sE[2 * lane + 1] = ee[1];
            sR[2 * lane] = rr[0];
            sR[2 * lane + 1] = rr[1];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const float r0 = 2 * lane >= 16 * b ? rr[0] : 1.0f;
                const float r1 = 2 * lane + 1 >= 16 * b ? rr[1] : 1.0f;
                float pr = r0 * r1;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(kFullMask, pr, off);
                    if (lane >= off) pr *= y;
                }
                float excl = __shfl_up_sync(kFullMask, pr, 1);
                if (lane == 0) excl = 1.0f;
                sPre[b][2 * lane] = excl;
                sPre[b][2 * lane + 1] = excl * r0;
            }
        }
        if (FUSED && pt >= 64 && pt < 64 + K)   // the preconditioner entering the chunk
            sD0[pt - 64] = p.dchk[((size_t)seq * nch + j) * K + (pt - 64)];
        ptx::named_bar(1, kPrepThreads);
        if (GATED && pt < C) {
            // tokens past T add nothing to the log, so sLg[C-1] is the chunk's total
            const float lgC = sLg[C - 1];
            sD[pt] = (pt < nvalid) ? __expf(lgC - sLg[pt]) : 0.0f;
            if (pt == 0) p.gc[(size_t)seq * nch + j] = __expf(lgC);
        }

        bool fok = true;
        if (PCH) {
            // ---- log Gam per channel: thread (column pair fp, token group grp)
            // sums log alpha over its tokens for columns 2 fp and 2 fp + 1
            constexpr int CP = K / 2, QT = kPrepThreads / CP, TPT = C / QT;
            const int fp = pt % CP, grp = pt / CP, f0 = 2 * fp;
            float lam[TPT][2];
            {
                float run0 = 0.0f, run1 = 0.0f;
                bool bad = false;
#pragma unroll
                for (int i = 0; i < TPT; ++i) {
                    const int t = grp * TPT + i;
                    float2 a = make_float2(1.0f, 1.0f);
                    if (t < nvalid)
                        a = *reinterpret_cast<const float2 *>(p.alpha_k + ((size_t)seq * T + t0 + t) * K + f0);
                    if (!(a.x >= kMinDecay && a.x <= kMaxDecay)) { bad = true; a.x = 1.0f; }   // NaN fails too
                    if (!(a.y >= kMinDecay && a.y <= kMaxDecay)) { bad = true; a.y = 1.0f; }
                    run0 += __logf(a.x);
                    run1 += __logf(a.y);
                    lam[i][0] = run0;
                    lam[i][1] = run1;
                }
                if (bad) report_status(p.status, OSDN_ERR_DEVICE);
                sGrp[grp][f0] = run0;
                sGrp[grp][f0 + 1] = run1;
            }
            ptx::named_bar(1, kPrepThreads);
            {
                float off0 = 0.0f, off1 = 0.0f;
                for (int g2 = 0; g2 < grp; ++g2) {
                    off0 += sGrp[g2][f0];
                    off1 += sGrp[g2][f0 + 1];
                }
#pragma unroll
                for (int i = 0; i < TPT; ++i) {
                    lam[i][0] += off0;
                    lam[i][1] += off1;
                    const int t = grp * TPT + i;
                    if ((t & 15) == 15 && t < C - 1) {
                        sLref[(t >> 4) + 1][f0] = lam[i][0];
                        sLref[(t >> 4) + 1][f0 + 1] = lam[i][1];
                    }
                    if (t == C - 1) {   // tokens past T add nothing: this is the chunk's Gam_C
                        sLamC[f0] = lam[i][0];
                        sLamC[f0 + 1] = lam[i][1];
                        *reinterpret_cast<float2 *>(p.gc + ((size_t)seq * nch + j) * K + f0) =
                            make_float2(expf(lam[i][0]), expf(lam[i][1]));
                    }
                }
                if (grp == 0) {
                    sLref[0][f0] = 0.0f;
                    sLref[0][f0 + 1] = 0.0f;
                }
            }
            ptx::named_bar(1, kPrepThreads);
            // bf16 pairs in the swizzled tiles (columns f0, f0 + 1 share a 4-byte word)
            auto ld2 = [](const uint8_t *tile, int off) {
                return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(tile + off));
            };
            auto st2 = [](uint8_t *tile, int off, float x, float y) {
                *reinterpret_cast<__nv_bfloat162 *>(tile + off) = __floats2bfloat162_rn(x, y);
            };
            uint8_t *bufs[2] = {smem + LY::oL, sXb};
            // This thread's tokens lie in one 16-token block bs (m = 16 bs - 1 its
            // reference, e = 16 bs + 15 its last token).  With E_s = Gam_e / Gam_s
            // (<= 1; one exp a token), every factor is E_s times a per-column
            // constant: the row factor Gam_s / Gam_m = (Gam_e / Gam_m) / E_s, the
            // copy b >= bs factor Gam_m(b) / Gam_s = (Gam_m(b) / Gam_e) E_s, and
            // Gam_C / Gam_s = (Gam_C / Gam_e) E_s.
            const int bs = (grp * TPT) / 16;
            const float le0 = bs < 3 ? sLref[bs + 1][f0] : sLamC[f0];
            const float le1 = bs < 3 ? sLref[bs + 1][f0 + 1] : sLamC[f0 + 1];
            const float2 cblk = make_float2(__expf(le0 - sLref[bs][f0]), __expf(le1 - sLref[bs][f0 + 1]));
            const float2 cdk = make_float2(__expf(sLamC[f0] - le0), __expf(sLamC[f0 + 1] - le1));
            float2 cb[4];
#pragma unroll
            for (int b = 0; b < 4; ++b)
                cb[b] = b >= bs ? make_float2(__expf(sLref[b][f0] - le0), __expf(sLref[b][f0 + 1] - le1))
                                : make_float2(0.0f, 0.0f);
            for (int x = pt; x < 4 * K; x += kPrepThreads) sGref[x / K][x % K] = __expf(sLref[x / K][x % K]);
            float2 E[TPT];
#pragma unroll
            for (int i = 0; i < TPT; ++i) E[i] = make_float2(__expf(le0 - lam[i][0]), __expf(le1 - lam[i][1]));
            // ---- once the tiles have landed: [K;Q] rows relative to their block's
            // reference, and the first two reference copies of Kt
            fok = vote_all(wait_poll(&bar_full, 0, &s_abort, st), 1, kPrepThreads);
            if (fok) {
                const float2 c0v = cb[0], c1v = cb[1];
#pragma unroll
                for (int i = 0; i < TPT; ++i) {
                    const int t = grp * TPT + i;
                    const float fx = __fdividef(cblk.x, E[i].x), fy = __fdividef(cblk.y, E[i].y);
                    const int ok_ = sw_off(128, t, f0), oq = sw_off(128, C + t, f0), ot = sw_off(C, t, f0);
                    const float2 kv = ld2(sKQ, ok_), qv = ld2(sKQ, oq), raw = ld2(sKt, ot);
                    st2(sKQ, ok_, kv.x * fx, kv.y * fy);
                    st2(sKQ, oq, qv.x * fx, qv.y * fy);
                    st2(bufs[0], ot, raw.x * c0v.x * E[i].x, raw.y * c0v.y * E[i].y);
                    st2(bufs[1], ot, raw.x * c1v.x * E[i].x, raw.y * c1v.y * E[i].y);
                }
                ptx::fence_proxy_async_smem();
                ptx::named_bar(1, kPrepThreads);
                if (pt == 0) ptx::mbar_arrive(&bar_c01);
            }
            fok = fok && vote_all(wait_poll(&bar_r0, 0, &s_abort, st), 1, kPrepThreads);
            if (fok) {   // reference 0's product has read its buffer
#pragma unroll
                for (int i = 0; i < TPT; ++i) {
                    const int ot = sw_off(C, grp * TPT + i, f0);
                    const float2 raw = ld2(sKt, ot);
                    st2(bufs[0], ot, raw.x * cb[2].x * E[i].x, raw.y * cb[2].y * E[i].y);
                }
                ptx::fence_proxy_async_smem();
                ptx::named_bar(1, kPrepThreads);
                if (pt == 0) ptx::mbar_arrive(&bar_c2);
            }
            fok = fok && vote_all(wait_poll(&bar_r1, 0, &s_abort, st), 1, kPrepThreads);
            if (fok) {
                // copy 3, and Kt itself to (Gam_C / Gam_s) . kt for W and M
#pragma unroll
                for (int i = 0; i < TPT; ++i) {
                    const int ot = sw_off(C, grp * TPT + i, f0);
                    const float2 raw = ld2(sKt, ot);
                    st2(bufs[1], ot, raw.x * cb[3].x * E[i].x, raw.y * cb[3].y * E[i].y);
                    st2(sKt, ot, raw.x * cdk.x * E[i].x, raw.y * cdk.y * E[i].y);
                }
                ptx::fence_proxy_async_smem();
                ptx::named_bar(1, kPrepThreads);
                if (pt == 0) ptx::mbar_arrive(&bar_c3);
            }
        }
        if (FUSED) {
            // ---- P = pi . e (strictly lower): high part over A, remainder over Kt
            {
                const int t = pt >> 2, blk = pt & 3, s0 = 16 * blk;
                float ph[16], pl[16];
                // pi_st = prod_{s<v<t} r_v, walked down from s = s0 + 15, where
                // it is the product of r over [s0 + 16, t)
                float pi = blk < 3 ? sPre[blk + 1][t] : 1.0f;
#pragma unroll
                for (int e = 15; e >= 0; --e) {
                    const int s = s0 + e;
                    float val = 0.0f;
                    if (s < t) {
                        val = pi * sE[s];
                        pi *= sR[s];
                    }
                    ph[e] = __bfloat162float(__float2bfloat16_rn(val));
                    pl[e] = val - ph[e];
                }
                st_row_sw128(sA, C, t, s0, ph, 16);
                st_row_sw128(sKt, C, t, s0, pl, 16);
            }
            // ---- W = K . K once the keys have landed: high part over L, remainder over Xb
            fok = vote_all(wait_poll(&bar_full, 0, &s_abort, st), 1, kPrepThreads);
            if (fok) {
                constexpr int PIECES = C * K * 2 / 16;   // 16-byte pieces of the K rows
                uint8_t *sWh = smem + LY::oL, *sWl = sXb;
                for (int i = pt; i < PIECES; i += kPrepThreads) {
                    const int cb = i >> 9, o = (i & 511) * 16;   // 512 pieces per 64-row block
                    const uint4 u = *reinterpret_cast<const uint4 *>(sKQ + cb * 16384 + o);
                    const uint32_t in[4] = {u.x, u.y, u.z, u.w};
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&in[e]));
                        const float wx = x.x * x.x, wy = x.y * x.y;   // exact: bf16 squared fits fp32
                        hi[e] = pack_bf16x2(wx, wy);
                        const float2 h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hi[e]));
                        lo[e] = pack_bf16x2(wx - h.x, wy - h.y);
                    }
                    *reinterpret_cast<uint4 *>(sWh + cb * 8192 + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(sWl + cb * 8192 + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
                ptx::fence_proxy_async_smem();
                ptx::named_bar(1, kPrepThreads);
                if (pt == 0) ptx::mbar_arrive(&bar_f0);
            }
            // ---- Kt = (rho d_c + P W) . K, over P's remainder (its product has completed)
            fok = fok && vote_all(wait_poll(&bar_f1, 0, &s_abort, st), 1, kPrepThreads);
            if (fok) {
                ptx::tc_fence_after();
                const int mrow = 16 * (warp & 3) + lane;
                const uint32_t loff = static_cast<uint32_t>(32 * (warp & 3)) << 16;
                const int h = warp >> 2;
                float v[NH];
                tmem_ldn<NH>(tmem + loff + h * NH, v);
                if (lane < 16) {
                    const float rho = sPre[0][mrow];
#pragma unroll
                    for (int c = 0; c < NH; c += 16) {
                        float kv[16];
                        ld_row_sw128(sKQ, 128, mrow, h * NH + c, kv, 16);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            kv[e] *= fmaf(rho, sD0[h * NH + c + e], v[c + e]);
                        st_row_sw128(sKt, C, mrow, h * NH + c, kv, 16);
                    }
                }
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before();
                ptx::named_bar(1, kPrepThreads);
                if (pt == 0) ptx::mbar_arrive(&bar_kt);
            }
        }

        // ---- Gram / scores: L (fp32) and A (bf16); then Kt <- D Kt
        bool ok = fok && vote_all(wait_poll(&bar_g, 0, &s_abort, st), 1, kPrepThreads);
        if (ok) {
            ptx::tc_fence_after();
            float g[32];
            if (PCH) {  // lanes 0-15 of the warp read block b0's reference, 16-31 block b0+1's
                const int b0 = 2 * (q4 & 1);
                float g1[32];
                tmem_ld32(tmem + lane_off + 64 * b0 + 32 * half, g);
                tmem_ld32(tmem + lane_off + 64 * (b0 + 1) + 32 * half, g1);
                if (lane >= 16) {
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) g[jj] = g1[jj];
                }
            } else {
                tmem_ld32(tmem + lane_off + 32 * half, g);
            }
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
            if (GATED) {  // Kt rows scaled by g_C / g_t (the Gram product has read Kt)
                constexpr int PIECES = C * K * 2 / 16;
                for (int i = pt; i < PIECES; i += kPrepThreads) {
                    const int row = (i >> 3) & 63;   // 8 pieces per 128-byte row
                    uint4 *q = reinterpret_cast<uint4 *>(sKt + i * 16);
                    uint4 u = *q;
                    const float f = sD[row];
                    uint32_t *wv = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float2 x = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&wv[e]));
                        wv[e] = pack_bf16x2(x.x * f, x.y * f);
                    }
                    *q = u;
                }
            }
            if (PCH) {  // K rows to Gam . K for Kw (the Gram products have read them)
                constexpr int CP = K / 2, QT = kPrepThreads / CP, TPT = C / QT;
                const int f0 = 2 * (pt % CP), grp = pt / CP;
#pragma unroll
                for (int i = 0; i < TPT; ++i) {
                    const int t = grp * TPT + i, off = sw_off(128, t, f0);
                    __nv_bfloat162 *w2 = reinterpret_cast<__nv_bfloat162 *>(sKQ + off);
                    const float2 kv = __bfloat1622float2(*w2);
                    *w2 = __floats2bfloat162_rn(kv.x * sGref[t >> 4][f0], kv.y * sGref[t >> 4][f0 + 1]);
                }
            }
            ptx::tc_fence_before();
            ptx::named_bar(1, kPrepThreads);
            solve_unit_lower(sL, pt);
            // ---- Xb = X diag(beta) and Xb diag(g), bf16 for the MMAs
            const int t = pt >> 2, s0 = 16 * (pt & 3);
            float xb[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int s = s0 + e;
                xb[e] = (s <= t) ? sL[t * kLP + s] * sBeta[s] : 0.0f;
            }
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
        // M=64 accumulators: row 16*q4 + lane (lanes 0-15 of each quarter);
        // an M=K accumulator: row 32*q4 + lane (K = 128) or as M=64 (K = 64)
        const int mrow = 16 * q4 + lane;
        const bool act = lane < 16;
        const int krow = (K == 128) ? 32 * q4 + lane : mrow;
        const bool kact = (K == 128) || act;
        // ---- Kw (bf16 over the K rows), W and Ae (to the workspace)
        if (ok) ok = vote_all(wait_poll(&bar_p1, 0, &s_abort, st), 1, kPrepThreads);
        if (ok) {
            ptx::tc_fence_after();
            {
                float v[NH];
                tmem_ldn<NH>(tmem + lane_off + cKw + half * NH, v);
                if (act) st_row_sw128(sKQ, 128, mrow, half * NH, v, NH);
            }
            {
                float v[32];
                tmem_ld32(tmem + lane_off + cW + 32 * half, v);
                if (kact) st_row_sw128(sW + (krow >> 6) * 8192, 64, krow & 63, 32 * half, v, 32);
                tmem_ld32(tmem + lane_off + cAe + 32 * half, v);
                if (act) st_row_sw128(sXb, 64, mrow, 32 * half, v, 32);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_bar(1, kPrepThreads);
            if (pt == 0) {
                ptx::mbar_arrive(&bar_x3);
#pragma unroll
                for (int rb = 0; rb < K / 64; ++rb) ptx::tma_store_3d(&tm_w, sW + rb * 8192, 0, krow0 + rb * 64, seq);
                ptx::tma_store_3d(&tm_ae, sXb, 0, t0, seq);
                ptx::bulk_commit_group();
            }
        }
        // ---- M = -M' (stored as soon as it is staged), then Qe = diag(g) Q - Qe'
        if (ok) ok = vote_all(wait_poll(&bar_p2, 0, &s_abort, st), 1, kPrepThreads);
        if (ok) {
            ptx::tc_fence_after();
            {
                float v[NH];
                tmem_ldn<NH>(tmem + lane_off + cM + half * NH, v);
#pragma unroll
                for (int e = 0; e < NH; ++e) v[e] = -v[e];
                const int col = half * NH;
                if (kact) st_row_sw128(mbox(krow >> 6, col >> 6), 64, krow & 63, col & 63, v, NH);
            }
            float d[NH];
            tmem_ldn<NH>(tmem + lane_off + cQe + half * NH, d);
            ptx::fence_proxy_async_smem();
            ptx::named_bar(1, kPrepThreads);
            if (pt == 0) {
#pragma unroll
                for (int rb = 0; rb < K / 64; ++rb)
#pragma unroll
                    for (int cb = 0; cb < K / 64; ++cb)
                        ptx::tma_store_3d(&tm_m, mbox(rb, cb), cb * 64, krow0 + rb * 64, seq);
                ptx::bulk_commit_group();
            }
            const float gt = GATED ? __expf(sLg[mrow & 63]) : 1.0f;
            if (act) {
#pragma unroll
                for (int c = 0; c < NH; c += 16) {
                    float qv[16];
                    ld_row_sw128(sKQ, 128, C + mrow, half * NH + c, qv, 16);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        // PCH: Q rows hold (Gam_t / Gam_m) . q_t; Gam_m restores Gam . q
                        const float ge = PCH ? sGref[mrow >> 4][half * NH + c + e] : gt;
                        qv[e] = fmaf(ge, qv[e], -d[c + e]);
                    }
                    st_row_sw128(sKQ, 128, C + mrow, half * NH + c, qv, 16);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::named_bar(1, kPrepThreads);
            if (pt == 0) {
#pragma unroll
                for (int cb = 0; cb < K / 64; ++cb)
                    ptx::tma_store_3d(&tm_qe, sKQ + cb * 16384 + 8192, cb * 64, t0, seq);
                ptx::bulk_commit_group();
            }
        }
        // the stores have read their shared-memory tiles before the CTA exits
        if (pt == 0) ptx::bulk_wait_read_all();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 8) ptx::tmem_dealloc(tmem, kPrepCols);
}

template <int K, bool GATED, bool FUSED, bool PCH>
cudaError_t prep_launch_t(int BH, int T, int c0, int c1, const void *q, const void *k,
                          const void *kt, const float *beta, const float *alpha, const Fused &fz,
                          __nv_bfloat16 *w, __nv_bfloat16 *m, __nv_bfloat16 *qe, __nv_bfloat16 *ae,
                          float *gc, int *status, cudaStream_t stream) {
    const int nch = (T + C - 1) / C, Tp = nch * C;
    CUtensorMap mk, mq, mkt, mw, mm, mqe, mae;
    if (!make_map(&mk, k, BH, T, K) || !make_map(&mq, q, BH, T, K) ||
        !make_map(&mkt, FUSED ? k : kt, BH, T, K) ||   // fused: Kt is built, not loaded
        !make_map(&mw, w, BH, nch * K, C) || !make_map(&mm, m, BH, nch * K, K) ||
        !make_map(&mqe, qe, BH, Tp, K) || !make_map(&mae, ae, BH, Tp, C))
        return cudaErrorInvalidValue;
    constexpr int smem = PrepLay<K>::kAlloc;
    static std::atomic<unsigned long long> attr_done{0};
    {
        cudaError_t e = smem_attr_once((const void *)chunk_prep_kernel<K, GATED, FUSED, PCH>, smem, attr_done);
        if (e != cudaSuccess) return e;
    }
    PrepParams p;
    p.T = T;
    p.nch = nch;
    p.c0 = c0;
    p.beta = beta;
    p.alpha = alpha;
    p.r = fz.r;
    p.ecoef = fz.ecoef;
    p.dchk = fz.dchk;
    p.alpha_k = fz.alpha_k;
    p.gc = gc;
    p.status = status;
    p.BH = BH;
    p.ahead = 2 * sm_count();   // two CTAs per SM
    const dim3 grid = seq_grid(c1 - c0, BH);
    chunk_prep_kernel<K, GATED, FUSED, PCH><<<grid, kPrepBlock, smem, stream>>>(mk, mq, mkt, mw, mm, mqe, mae, p);
    return cudaGetLastError();
}

template <int K>
cudaError_t prep_launch_k(int BH, int T, int c0, int c1, const void *q, const void *k,
                          const void *kt, const float *beta, const float *alpha, const Fused &fz,
                          __nv_bfloat16 *w, __nv_bfloat16 *m, __nv_bfloat16 *qe, __nv_bfloat16 *ae,
                          float *gc, int *status, cudaStream_t stream) {
    if (fz.alpha_k)
        return prep_launch_t<K, false, false, true>(BH, T, c0, c1, q, k, kt, beta, nullptr, fz, w, m, qe, ae, gc, status, stream);
    if (fz.ecoef) {
        if (alpha)
            return prep_launch_t<K, true, true, false>(BH, T, c0, c1, q, k, kt, beta, alpha, fz, w, m, qe, ae, gc, status, stream);
        return prep_launch_t<K, false, true, false>(BH, T, c0, c1, q, k, kt, beta, alpha, fz, w, m, qe, ae, gc, status, stream);
    }
    if (alpha)
        return prep_launch_t<K, true, false, false>(BH, T, c0, c1, q, k, kt, beta, alpha, fz, w, m, qe, ae, gc, status, stream);
    return prep_launch_t<K, false, false, false>(BH, T, c0, c1, q, k, kt, beta, alpha, fz, w, m, qe, ae, gc, status, stream);
}

}  // namespace

// Chunks [c0, c1) of every sequence.  With fz.ecoef given (the fused forward
// pass) Kt is rebuilt from the preconditioner's checkpoints instead of read;
// with fz.alpha_k the decay is per key channel.
cudaError_t chunk_prep_launch(int BH, int T, int K, int c0, int c1, const void *q, const void *k,
                              const void *kt, const float *beta, const float *alpha,
                              const Fused &fz, __nv_bfloat16 *w, __nv_bfloat16 *m,
                              __nv_bfloat16 *qe, __nv_bfloat16 *ae, float *gc, int *status,
                              cudaStream_t stream) {
    if (K == 128)
        return prep_launch_k<128>(BH, T, c0, c1, q, k, kt, beta, alpha, fz, w, m, qe, ae, gc, status, stream);
    return prep_launch_k<64>(BH, T, c0, c1, q, k, kt, beta, alpha, fz, w, m, qe, ae, gc, status, stream);
}

}  // namespace tc
}  // namespace osdn
