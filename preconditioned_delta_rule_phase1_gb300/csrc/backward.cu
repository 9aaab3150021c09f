// backward.cu -- gradients of the OSDN forward pass through both phases, in
// fp32 arithmetic (both I/O types), token by token in reverse time.
//
// The forward ("OSDN: Improving Delta Rule with Provable Online
// Preconditioning in Linear Attention", gist.science summary, sections 2.1,
// 2.2 and 2.3):
//
//     ktilde_t = d_t (.) k_t
//     d_{t+1}  = r_t d_t + c_t w_t,   w_t = k_t^2,  n_t = |k_t|^2,
//                c_t = eta beta_t (1 - beta_t <d_t, w_t>) / n_t  (0 if n_t = 0)
//     S_t      = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) ktilde_t^T
//     o_t      = S_t q_t
//
// Its derivative is taken by hand and run in three kernels:
//
//  1. state_adjoint_kernel -- Phase 2.  The rows of S evolve independently,
//     so one warp owns value row i (lane l holds key columns l*NC..l*NC+NC-1,
//     NC = K/32) and a CTA holds 8 rows.  A forward sweep writes the row's
//     state every 16 tokens; the reverse sweep recomputes each 16-token
//     sub-chunk (states in shared memory) and walks it backwards with the
//     row's state gradient G = dL/dS_t[i,:]:
//         G += dO_t[i] q_t;  du = <G, ktilde_t>;  dSbar = G - beta du k_t
//         dv_t[i] = beta du;  G <- alpha dSbar
//     and the row's shares of the gradients that sum over rows
//         dq_t += dO_t[i] S_t[i],  dktilde_t += u_t[i] G,
//         dk_t += -beta du alpha S_{t-1}[i],  dbeta_t += du e_t[i],
//         dalpha_t += <dSbar, S_{t-1}[i]>      (e = v - alpha S_{t-1} k)
//     which the CTA adds over its 8 rows in warp order and writes as one
//     partial per row block (no atomics: the result is deterministic).
//     With a decay per key channel (alpha_t in R^K scaling the key columns
//     of S, the Kimi-Delta-Attention-style backbone) the same sweep runs with
//     Diag(alpha_t) in place of alpha_t, and dalpha_t is a K-vector:
//     dalpha_t[j] += dSbar[i,j] S_{t-1}[i,j].
//  2. partial_sum_kernel -- adds the row-block partials in a fixed order:
//     dq and dalpha are final; dktilde (plus the caller's cotangent of the
//     ktilde output), Phase 2's share of dk and of dbeta go to scratch.
//  3. precond_adjoint_kernel -- Phase 1.  One warp per sequence runs the
//     adjoint lam = dL/dd_t backwards; the step's Jacobian r I - mu w w^T is
//     symmetric, so the adjoint has the forward's form:
//         dr_t = <lam, d_t>,  dc = <lam, w_t>,  da = -dc eta beta^2 / n
//         dbeta_t += dc eta (1 - 2 beta a) / n,  deta += dc beta (1 - beta a) / n
//         dk_t += g d_t + 2 k_t (c_t lam + da d_t + dn),  dn = -dc c_t / n
//         lam <- r_t lam + da w_t + g k_t,   g = dktilde_t (both shares)
//     with d_t recomputed by 16-token sub-chunks from checkpoints.
//
// Every access is a plain load or store inside the caller's buffers or the
// workspace; there are no waits, so nothing can stall.
#include <atomic>

#include "osdn_device.cuh"

namespace osdn {

constexpr int kBwdSub = 16;    // tokens per recomputed sub-chunk
constexpr int kBwdWindow = 1024;   // tokens per reverse-sweep launch (the partials hold one window)
constexpr int kBwdRows = 8;    // value rows (one warp each) per state-adjoint CTA
constexpr int kBwdSeqs = 4;    // sequences (one warp each) per precond-adjoint CTA
constexpr int kSumTok = 8;     // tokens per partial-sum CTA

// Values a token contributes per row block: dq, dktilde, dk (K each), dbeta,
// then dalpha (1 value, or K with a decay per key channel).
__host__ __device__ constexpr int bwd_part_width(int K, bool pch = false) {
    return 3 * K + 1 + (pch ? K : 1);
}
// row stride of the shared reduction buffer: a multiple of 4 floats keeps the
// vector stores into it 16-byte aligned
__host__ __device__ constexpr int bwd_red_stride(int K, bool pch = false) {
    return (bwd_part_width(K, pch) + 3) & ~3;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(kFullMask, x, m);
    return x;
}
__device__ __forceinline__ float2 warp_sum2(float2 x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        x.x += __shfl_xor_sync(kFullMask, x.x, m);
        x.y += __shfl_xor_sync(kFullMask, x.y, m);
    }
    return x;
}

// NC consecutive elements (NC = 2 or 4) at p, converted to fp32.
template <int NC, typename T>
__device__ __forceinline__ void load_cols(const T *p, float (&x)[NC]) {
    if constexpr (NC == 4) load4(p, x); else load2(p, x);
}
template <int NC, typename T>
__device__ __forceinline__ void store_cols(T *p, const float (&x)[NC]) {
    if constexpr (NC == 4) store4(p, x); else store2(p, x);
}

// The decay of token g for this lane's NC columns: alpha[g] for every
// column (a scalar gate), alpha[g*K + c0 ..] (a decay per key channel), or 1.
template <bool PCH, int NC>
__device__ __forceinline__ void decay_cols(const float *alpha, size_t g, int K, int c0,
                                           float (&a)[NC]) {
    if (!alpha) {
#pragma unroll
        for (int m = 0; m < NC; ++m) a[m] = 1.0f;
    } else if constexpr (PCH) {
        load_cols<NC>(alpha + g * K + c0, a);
    } else {
        const float s = alpha[g];
#pragma unroll
        for (int m = 0; m < NC; ++m) a[m] = s;
    }
}

// The row's prediction <Diag(a) S_{t-1}[i], k_t>, reduced over the warp.  A
// scalar gate multiplies after the reduction, a per-channel decay before it.
template <bool PCH, int NC>
__device__ __forceinline__ float decayed_pred(const float (&S)[NC], const float (&a)[NC],
                                              const float (&kc)[NC]) {
    float sk = 0.0f;
#pragma unroll
    for (int m = 0; m < NC; ++m) sk = fmaf(PCH ? a[m] * S[m] : S[m], kc[m], sk);
    sk = warp_sum(sk);
    return PCH ? sk : a[0] * sk;
}

// ---------------------------------------------------------------- kernel 1
// The CTA's 8 rows all read the same keys, ktilde and queries, so each
// 16-token sub-chunk is staged once in shared memory by cp.async, one
// sub-chunk ahead: keys, ktilde, the CTA's rows of v and dO, beta and a scalar
// decay in two slots, the queries (read by the reverse walk only) in one,
// fetched while the sub-chunk is recomputed.  The arithmetic is the same as
// with the loads from global memory; only where the operands come from moves.
__device__ __forceinline__ void bwd_cp16(void *dst, const void *src, bool valid) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void bwd_cp4(void *dst, const void *src, bool valid) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(s), "l"(src), "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void bwd_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bwd_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Byte layout of the staging area (after the recomputed states and the
// reduction buffer): slots [2] of the per-token operands, one query tile,
// and with a decay per key channel one tile of its [kBwdSub][K] rows.
template <typename io_t, int K, bool PCH>
struct BwdStage {
    static constexpr int ROW = K * (int)sizeof(io_t);                       // one token's key row
    static constexpr int VROW = kBwdRows * (int)sizeof(io_t);               // one token's v (or dO) of the rows
    static constexpr int SK = 0;                                            // [2][kBwdSub][K]
    static constexpr int SKT = SK + 2 * kBwdSub * ROW;                      // [2][kBwdSub][K]
    static constexpr int SQ = SKT + 2 * kBwdSub * ROW;                      // [kBwdSub][K]
    static constexpr int SV = SQ + kBwdSub * ROW;                           // [2][kBwdSub][kBwdRows]
    static constexpr int SDO = SV + 2 * kBwdSub * VROW;                     // [2][kBwdSub][kBwdRows]
    static constexpr int SB = SDO + 2 * kBwdSub * VROW;                     // [2][kBwdSub] beta
    static constexpr int SA = SB + 2 * kBwdSub * 4;                         // [2][kBwdSub] scalar decay
    static constexpr int SAK = SA + 2 * kBwdSub * 4;                        // [kBwdSub][K] per-channel decay
    static constexpr int BYTES = SAK + (PCH ? kBwdSub * K * 4 : 0);
    static_assert(VROW % 16 == 0, "a token's rows of v must be whole 16-byte pieces");
};

// The reduction tile is double-buffered (one barrier a token); with a decay
// per key channel, whose rows are wider, it is single-buffered (two
// barriers a token) so that two CTAs still fit on an SM.
template <bool PCH>
constexpr int bwd_red_bufs() { return PCH ? 1 : 2; }

template <typename io_t, int K, bool PCH>
constexpr int state_adjoint_smem_bytes() {
    return (kBwdRows * kBwdSub * K + bwd_red_bufs<PCH>() * kBwdRows * bwd_red_stride(K, PCH)) * 4 +
           BwdStage<io_t, K, PCH>::BYTES;
}

template <typename io_t, int K, bool PCH>
__global__ void __launch_bounds__(kBwdRows * 32)
state_adjoint_kernel(int BH, int T, int V, int nsub, const io_t *__restrict__ q,
                     const io_t *__restrict__ k, const io_t *__restrict__ kt,
                     const io_t *__restrict__ v, const float *__restrict__ beta,
                     const float *__restrict__ alpha, const float *__restrict__ S0,
                     const io_t *__restrict__ dO, const float *__restrict__ dST,
                     io_t *__restrict__ dv, float *__restrict__ dS0, float *__restrict__ ck,
                     float *__restrict__ part, int fwd, int tw0, int tw1, int Tw,
                     float *__restrict__ gcarry) {
    constexpr int NC = K / 32;
    constexpr int P = bwd_part_width(K, PCH);
    constexpr int PS = bwd_red_stride(K, PCH);
    using SG = BwdStage<io_t, K, PCH>;
    constexpr int EPP = 16 / (int)sizeof(io_t);   // elements per 16-byte piece
    constexpr int PR = K / EPP;                   // pieces per key row
    constexpr int VP = SG::VROW / 16;             // pieces per token of the rows' v
    constexpr int NT = kBwdRows * 32;
    extern __shared__ __align__(16) float smem[];
    float *Sp = smem;                                  // [kBwdRows][kBwdSub][K]
    constexpr int NRED = bwd_red_bufs<PCH>();
    float *red = smem + kBwdRows * kBwdSub * K;        // [NRED][kBwdRows][PS]
    uint8_t *stg = reinterpret_cast<uint8_t *>(red + NRED * kBwdRows * PS);
    auto sk = [&](int s, int tt) { return reinterpret_cast<io_t *>(stg + SG::SK) + (s * kBwdSub + tt) * K; };
    auto skt = [&](int s, int tt) { return reinterpret_cast<io_t *>(stg + SG::SKT) + (s * kBwdSub + tt) * K; };
    auto sq = [&](int tt) { return reinterpret_cast<io_t *>(stg + SG::SQ) + tt * K; };
    auto sv = [&](int s, int tt) { return reinterpret_cast<io_t *>(stg + SG::SV) + (s * kBwdSub + tt) * kBwdRows; };
    auto sdo = [&](int s, int tt) { return reinterpret_cast<io_t *>(stg + SG::SDO) + (s * kBwdSub + tt) * kBwdRows; };
    auto sb = [&](int s) { return reinterpret_cast<float *>(stg + SG::SB) + s * kBwdSub; };
    auto sa = [&](int s) { return reinterpret_cast<float *>(stg + SG::SA) + s * kBwdSub; };
    auto sak = [&](int tt) { return reinterpret_cast<float *>(stg + SG::SAK) + tt * K; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rb = blockIdx.x, nrb = gridDim.x;
    const int i0 = rb * kBwdRows, i = i0 + warp;      // the CTA's first row; this warp's row
    const size_t seq = grid_seq();
    if (seq >= (size_t)BH) return;
    const int c0 = lane * NC;
    const size_t tok0 = seq * (size_t)T;               // first token of the sequence
    float *Spw = Sp + warp * kBwdSub * K;

    // sub-chunk j's keys, ktilde, rows of v (and dO with `rev`), beta and a
    // scalar decay into slot s; tokens past T are zero-filled
    auto stage = [&](int s, int j, bool rev) {
        const int t0 = j * kBwdSub;
        for (int x = threadIdx.x; x < kBwdSub * PR; x += NT) {
            const int tt = x / PR, pc = x % PR;
            const bool ok = t0 + tt < T;
            const size_t g = tok0 + (ok ? t0 + tt : 0);
            bwd_cp16(sk(s, tt) + pc * EPP, k + g * K + pc * EPP, ok);
            bwd_cp16(skt(s, tt) + pc * EPP, kt + g * K + pc * EPP, ok);
        }
        for (int x = threadIdx.x; x < kBwdSub * VP; x += NT) {
            const int tt = x / VP, pc = x % VP;
            const bool ok = t0 + tt < T;
            const size_t g = tok0 + (ok ? t0 + tt : 0);
            bwd_cp16(sv(s, tt) + pc * EPP, v + g * V + i0 + pc * EPP, ok);
            if (rev && dO) bwd_cp16(sdo(s, tt) + pc * EPP, dO + g * V + i0 + pc * EPP, ok);
        }
        if (threadIdx.x < kBwdSub) {
            const int tt = threadIdx.x;
            const bool ok = t0 + tt < T;
            const size_t g = tok0 + (ok ? t0 + tt : 0);
            bwd_cp4(sb(s) + tt, beta + g, ok);
            if (!PCH && alpha) bwd_cp4(sa(s) + tt, alpha + g, ok);
        }
    };
    // sub-chunk j's per-channel decay rows into their one tile (issued when
    // the previous sub-chunk is done with it, ahead of the next prefetch)
    auto stage_alpha = [&](int j) {
        const int t0 = j * kBwdSub;
        for (int x = threadIdx.x; x < kBwdSub * (K / 4); x += NT) {
            const int tt = x / (K / 4), pc = x % (K / 4);
            const bool ok = t0 + tt < T;
            const size_t g = tok0 + (ok ? t0 + tt : 0);
            bwd_cp16(sak(tt) + 4 * pc, alpha + g * K + 4 * pc, ok);
        }
        bwd_commit();
    };
    auto stage_q = [&](int j) {
        const int t0 = j * kBwdSub;
        for (int x = threadIdx.x; x < kBwdSub * PR; x += NT) {
            const int tt = x / PR, pc = x % PR;
            const bool ok = t0 + tt < T;
            const size_t g = tok0 + (ok ? t0 + tt : 0);
            bwd_cp16(sq(tt) + pc * EPP, q + g * K + pc * EPP, ok);
        }
    };
    // the decay of token tt of the sub-chunk in slot s for this lane's columns
    auto decay = [&](int s, int tt, size_t g, float (&a)[NC]) {
        if constexpr (PCH) {
            if (alpha) {
                load_cols<NC>(sak(tt) + c0, a);
            } else {
#pragma unroll
                for (int m = 0; m < NC; ++m) a[m] = 1.0f;
            }
        } else {
            const float x = alpha ? sa(s)[tt] : 1.0f;
#pragma unroll
            for (int m = 0; m < NC; ++m) a[m] = x;
        }
    };

    // forward sweep (its own launch): the row's state every kBwdSub tokens
    float S[NC];
    if (fwd) {
    if (S0) {
        load_cols<NC>(S0 + (seq * V + i) * (size_t)K + c0, S);
    } else {
#pragma unroll
        for (int m = 0; m < NC; ++m) S[m] = 0.0f;
    }
    if (nsub > 0) stage(0, 0, false);
    bwd_commit();
    for (int j = 0; j < nsub; ++j) {
        __syncthreads();   // every warp is done with the other slot (and the decay tile)
        if (PCH && alpha) stage_alpha(j);
        if (j + 1 < nsub) stage((j + 1) & 1, j + 1, false);
        bwd_commit();
        bwd_wait<1>();
        __syncthreads();   // sub-chunk j is in
        const int s = j & 1, t0 = j * kBwdSub, tn = min(kBwdSub, T - t0);
        store_cols<NC>(ck + ((seq * nsub + j) * V + i) * (size_t)K + c0, S);
        for (int tt = 0; tt < tn; ++tt) {
            float kc[NC], tc[NC], a[NC];
            load_cols<NC>(sk(s, tt) + c0, kc);
            load_cols<NC>(skt(s, tt) + c0, tc);
            decay(s, tt, tok0 + t0 + tt, a);
            const float u = sb(s)[tt] * (to_f32(sv(s, tt)[warp]) - decayed_pred<PCH, NC>(S, a, kc));
#pragma unroll
            for (int m = 0; m < NC; ++m) S[m] = fmaf(a[m], S[m], u * tc[m]);
        }
    }
    bwd_wait<0>();
    return;
    }

    // reverse sweep over the window [tw0, tw1) (tw0 a multiple of kBwdWindow,
    // tw1 the next one or T), starting from the state gradient the later
    // window left in gcarry (from d_ST for the last window)
    float G[NC];
    float *grow = gcarry + (seq * V + i) * (size_t)K + c0;
    if (tw1 < T) {
        load_cols<NC>(grow, G);
    } else if (dST) {
        load_cols<NC>(dST + (seq * V + i) * (size_t)K + c0, G);
    } else {
#pragma unroll
        for (int m = 0; m < NC; ++m) G[m] = 0.0f;
    }
    const int jhi = (tw1 - 1) / kBwdSub, jlo = tw0 / kBwdSub;
    int slot = 0;
    stage(slot, jhi, true);
    bwd_commit();
    int buf = 0;
    for (int j = jhi; j >= jlo; --j) {
        __syncthreads();   // every warp is done with the other slot, the queries (and the decay tile)
        if (PCH && alpha) stage_alpha(j);
        if (j > jlo) stage(slot ^ 1, j - 1, true);
        bwd_commit();
        bwd_wait<1>();
        __syncthreads();   // sub-chunk j is in
        stage_q(j);        // for the walk, while the sub-chunk is recomputed
        bwd_commit();
        const int t0 = j * kBwdSub;
        const int tn = min(kBwdSub, T - t0);
        // recompute the sub-chunk: S_{t-1} of each token into shared memory,
        // e_t and u_t of token t0+tt kept by lane tt
        load_cols<NC>(ck + ((seq * nsub + j) * V + i) * (size_t)K + c0, S);
        float my_e = 0.0f, my_u = 0.0f;
        for (int tt = 0; tt < tn; ++tt) {
            const size_t g = tok0 + t0 + tt;
            store_cols<NC>(Spw + tt * K + c0, S);
            float kc[NC], tc[NC], a[NC];
            load_cols<NC>(sk(slot, tt) + c0, kc);
            load_cols<NC>(skt(slot, tt) + c0, tc);
            decay(slot, tt, g, a);
            const float e = to_f32(sv(slot, tt)[warp]) - decayed_pred<PCH, NC>(S, a, kc);
            const float u = sb(slot)[tt] * e;
            if (lane == tt) { my_e = e; my_u = u; }
#pragma unroll
            for (int m = 0; m < NC; ++m) S[m] = fmaf(a[m], S[m], u * tc[m]);
        }
        bwd_wait<0>();
        __syncthreads();   // the queries are in
        // walk it backwards (each lane reads back only its own columns of Spw)
        for (int tt = tn - 1; tt >= 0; --tt) {
            const size_t g = tok0 + t0 + tt;
            const float e = __shfl_sync(kFullMask, my_e, tt);
            const float u = __shfl_sync(kFullMask, my_u, tt);
            float sp[NC], qc[NC], kc[NC], tc[NC], a[NC];
            load_cols<NC>(Spw + tt * K + c0, sp);
            load_cols<NC>(sq(tt) + c0, qc);
            load_cols<NC>(sk(slot, tt) + c0, kc);
            load_cols<NC>(skt(slot, tt) + c0, tc);
            decay(slot, tt, g, a);
            const float b = sb(slot)[tt];
            const float dOi = dO ? to_f32(sdo(slot, tt)[warp]) : 0.0f;
            float du = 0.0f;
#pragma unroll
            for (int m = 0; m < NC; ++m) {
                G[m] = fmaf(dOi, qc[m], G[m]);
                du = fmaf(G[m], tc[m], du);
            }
            du = warp_sum(du);
            float dSb[NC];
#pragma unroll
            for (int m = 0; m < NC; ++m) dSb[m] = G[m] - b * du * kc[m];
            float *rw = red + (buf * kBwdRows + warp) * PS;
            float cq[NC], ct[NC], ck_[NC];
#pragma unroll
            for (int m = 0; m < NC; ++m) {
                cq[m] = dOi * fmaf(a[m], sp[m], u * tc[m]);   // dO_t[i] S_t[i]
                ct[m] = u * G[m];                             // u_t[i] G
                ck_[m] = -b * du * a[m] * sp[m];              // -beta du Sbar[i]
            }
            store_cols<NC>(rw + c0, cq);
            store_cols<NC>(rw + K + c0, ct);
            store_cols<NC>(rw + 2 * K + c0, ck_);
            // dalpha = <dSbar, S_{t-1}[i]>: per key column with a per-channel
            // decay (scalar stores: the columns start at the odd offset 3K + 1),
            // else summed over the row
            // (without a decay there is no dalpha: its columns are left at 0)
            if constexpr (PCH) {
#pragma unroll
                for (int m = 0; m < NC; ++m) rw[3 * K + 1 + c0 + m] = alpha ? dSb[m] * sp[m] : 0.0f;
            } else if (alpha) {
                float dal = 0.0f;
#pragma unroll
                for (int m = 0; m < NC; ++m) dal = fmaf(dSb[m], sp[m], dal);
                dal = warp_sum(dal);
                if (lane == 0) rw[3 * K + 1] = dal;
            } else if (lane == 0) {
                rw[3 * K + 1] = 0.0f;
            }
            if (lane == 0) {
                rw[3 * K] = du * e;
                from_f32(dv[g * V + i], b * du);
            }
#pragma unroll
            for (int m = 0; m < NC; ++m) G[m] = a[m] * dSb[m];
            __syncthreads();
            // the CTA's sum over its rows, in warp order; the next token
            // writes the other buffer, and its barrier orders these reads
            // before this buffer is written again
            const float *rsum = red + buf * kBwdRows * PS;
            float *dst = part + ((seq * nrb + rb) * (size_t)Tw + (t0 + tt - tw0)) * P;
            for (int x = threadIdx.x; x < P; x += kBwdRows * 32) {
                float s = 0.0f;
#pragma unroll
                for (int w = 0; w < kBwdRows; ++w) s += rsum[w * PS + x];
                dst[x] = s;
            }
            if (NRED == 1) __syncthreads();   // the tile is read before the next token writes it
            else buf ^= 1;
        }
        slot ^= 1;
    }
    bwd_wait<0>();
    if (tw0 > 0) store_cols<NC>(grow, G);
    else if (dS0) store_cols<NC>(dS0 + (seq * V + i) * (size_t)K + c0, G);
}

// ---------------------------------------------------------------- kernel 2
template <typename io_t, int K, bool PCH>
__global__ void __launch_bounds__(256)
partial_sum_kernel(int BH, int T, int nrb, int tw0, int tn, int Tw, const float *__restrict__ part,
                   const io_t *__restrict__ dkt_ext, io_t *__restrict__ dq,
                   float *__restrict__ dalpha, float *__restrict__ dkt_tot,
                   float *__restrict__ dk2, float *__restrict__ db2) {
    constexpr int P = bwd_part_width(K, PCH);
    const size_t seq = grid_seq();
    if (seq >= (size_t)BH) return;
    const int tb = blockIdx.x * kSumTok;   // within the window
    for (int x = threadIdx.x; x < kSumTok * P; x += blockDim.x) {
        const int tt = x / P, col = x % P;
        const int tl = tb + tt, t = tw0 + tl;
        if (tl >= tn) continue;
        float s = 0.0f;
        for (int r = 0; r < nrb; ++r) s += part[((seq * nrb + r) * (size_t)Tw + tl) * P + col];
        const size_t g = seq * (size_t)T + t;
        if (col < K) {
            from_f32(dq[g * K + col], s);
        } else if (col < 2 * K) {
            const int c = col - K;
            dkt_tot[g * K + c] = s + (dkt_ext ? to_f32(dkt_ext[g * K + c]) : 0.0f);
        } else if (col < 3 * K) {
            dk2[g * K + col - 2 * K] = s;
        } else if (col == 3 * K) {
            db2[g] = s;
        } else if (dalpha) {
            if constexpr (PCH) dalpha[g * K + col - 3 * K - 1] = s;
            else dalpha[g] = s;
        }
    }
}

// ---------------------------------------------------------------- kernel 3
// Phase 1 adjoint over tokens [tlo, thi) of sequence `seq` (both multiples of
// kBwdSub, or thi = T), walking sub-chunks backwards from lam at thi.  d_t is
// recomputed forward over each 16-token sub-chunk from the checkpoints ck
// (d every kBwdSub tokens, written by the forward scan).  With `emit` the
// token outputs (dk, dbeta, dr) are written and deta accumulated (the same
// value on every lane); `expand`
// is set if some token's step map r_t I - mu_t w w^T (mu = eta beta^2 / n)
// could expand (norm max(|r|, |r - mu |w|^2|) > 1).  One warp.
template <typename io_t, int K>
struct WalkStage {   // one warp's staging area (about 28 KB: two CTAs of 4 warps per SM)
    alignas(16) float dsub[kBwdSub][K];    // d_t of the sub-chunk, recomputed
    alignas(16) io_t sk[kBwdSub][K];       // keys
    alignas(16) float sg[kBwdSub][K];      // the total ktilde cotangent
    alignas(16) float s2[kBwdSub][K];      // Phase 2's share of dk
    alignas(16) float sb[kBwdSub];         // beta
    alignas(16) float sr[kBwdSub];         // r
    alignas(16) float sdb[kBwdSub];        // Phase 2's share of dbeta
};

template <typename io_t, int K>
__device__ void adjoint_walk(int T, int nsub, size_t seq, int tlo, int thi, bool emit,
                             const io_t *__restrict__ k, const float *__restrict__ beta,
                             const float *__restrict__ r, float eta,
                             const float *__restrict__ dkt_tot, const float *__restrict__ dk2,
                             const float *__restrict__ db2, const float *__restrict__ ck,
                             io_t *__restrict__ dk, float *__restrict__ dbeta,
                             float *__restrict__ dr, WalkStage<io_t, K> &ws, float (&lam)[K / 32],
                             float &deta_acc, bool &expand) {
    constexpr int NC = K / 32;
    constexpr int EPP = 16 / (int)sizeof(io_t);   // key elements per 16-byte piece
    constexpr int PR = K / EPP;                   // pieces per key row
    constexpr int PF = K / 4;                     // pieces per fp32 row
    const int lane = threadIdx.x & 31;
    const int c0 = lane * NC;
    const size_t tok0 = seq * (size_t)T;
    // sub-chunk j's keys, beta and r (tokens past T zero-filled)
    auto stage_keys = [&](int j) {
        const int t0 = j * kBwdSub;
        for (int x = lane; x < kBwdSub * PR; x += 32) {
            const int tt = x / PR, pc = x % PR;
            const bool ok = t0 + tt < T;
            const size_t g = tok0 + (ok ? t0 + tt : 0);
            bwd_cp16(&ws.sk[tt][pc * EPP], k + g * K + pc * EPP, ok);
        }
        const int tt = lane & (kBwdSub - 1);
        const bool ok = t0 + tt < T && (lane < kBwdSub || r);
        const size_t g = tok0 + (ok ? t0 + tt : 0);
        if (lane < kBwdSub) bwd_cp4(&ws.sb[tt], beta + g, ok);
        else if (r) bwd_cp4(&ws.sr[tt], r + g, ok);
    };
    // sub-chunk j's cotangents (and, when emitting, Phase 2's shares)
    auto stage_grads = [&](int j) {
        const int t0 = j * kBwdSub;
        for (int x = lane; x < kBwdSub * PF; x += 32) {
            const int tt = x / PF, pc = x % PF;
            const bool ok = t0 + tt < T;
            const size_t g = tok0 + (ok ? t0 + tt : 0);
            bwd_cp16(&ws.sg[tt][4 * pc], dkt_tot + g * K + 4 * pc, ok);
            if (emit) bwd_cp16(&ws.s2[tt][4 * pc], dk2 + g * K + 4 * pc, ok);
        }
        if (emit && lane < kBwdSub) {
            const bool ok = t0 + lane < T;
            bwd_cp4(&ws.sdb[lane], db2 + tok0 + (ok ? t0 + lane : 0), ok);
        }
    };
    float d[NC];
    for (int j = (thi - 1) / kBwdSub; j >= tlo / kBwdSub; --j) {
        const int t0 = j * kBwdSub;
        const int tn = min(kBwdSub, thi - t0);
        stage_keys(j);
        bwd_commit();
        stage_grads(j);    // for the walk, while the sub-chunk is recomputed
        bwd_commit();
        bwd_wait<1>();     // the keys of sub-chunk j are in
        __syncwarp();
        load_cols<NC>(ck + (seq * nsub + j) * K + c0, d);
        float my_n = 0.0f, my_a = 0.0f;
        for (int tt = 0; tt < tn; ++tt) {
            store_cols<NC>(&ws.dsub[tt][c0], d);
            float kc[NC];
            load_cols<NC>(&ws.sk[tt][c0], kc);
            float na[3] = {0.0f, 0.0f, 0.0f};   // n, <d, w>, |w|^2
#pragma unroll
            for (int m = 0; m < NC; ++m) {
                const float w = kc[m] * kc[m];
                na[0] += w;
                na[1] = fmaf(d[m], w, na[1]);
                na[2] = fmaf(w, w, na[2]);
            }
#pragma unroll
            for (int x = 16; x > 0; x >>= 1) {
#pragma unroll
                for (int e = 0; e < 3; ++e) na[e] += __shfl_xor_sync(kFullMask, na[e], x);
            }
            if (lane == tt) { my_n = na[0]; my_a = na[1]; }
            const float b = ws.sb[tt];
            const float c = na[0] > 0.0f ? eta * b * (1.0f - b * na[1]) / na[0] : 0.0f;
            const float rt = r ? ws.sr[tt] : 1.0f;
            const float mu = na[0] > 0.0f ? eta * b * b * na[2] / na[0] : 0.0f;
            if (fmaxf(fabsf(rt), fabsf(rt - mu)) > 1.0f + 1e-6f) expand = true;
#pragma unroll
            for (int m = 0; m < NC; ++m) d[m] = fmaf(rt, d[m], c * (kc[m] * kc[m]));
        }
        bwd_wait<0>();     // this sub-chunk's cotangents are in
        __syncwarp();
        for (int tt = tn - 1; tt >= 0; --tt) {
            const size_t g = tok0 + t0 + tt;
            const float n = __shfl_sync(kFullMask, my_n, tt);
            const float a = __shfl_sync(kFullMask, my_a, tt);
            float dc_[NC], kc[NC], gk[NC];
            load_cols<NC>(&ws.dsub[tt][c0], dc_);
            load_cols<NC>(&ws.sk[tt][c0], kc);
            load_cols<NC>(&ws.sg[tt][c0], gk);
            float2 rc = make_float2(0.0f, 0.0f);       // (<lam, d_t>, <lam, w_t>)
#pragma unroll
            for (int m = 0; m < NC; ++m) {
                rc.x = fmaf(lam[m], dc_[m], rc.x);
                rc.y = fmaf(lam[m], kc[m] * kc[m], rc.y);
            }
            rc = warp_sum2(rc);
            const float b = ws.sb[tt];
            const float rt = r ? ws.sr[tt] : 1.0f;
            float c = 0.0f, da = 0.0f, db1 = 0.0f, dn = 0.0f;
            if (n > 0.0f) {
                const float res = 1.0f - b * a;
                c = eta * b * res / n;
                da = -rc.y * eta * b * b / n;
                db1 = rc.y * eta * (1.0f - 2.0f * b * a) / n;
                if (emit) deta_acc += rc.y * b * res / n;
                dn = -rc.y * c / n;
            }
            if (emit) {
                float k2[NC], out[NC];
                load_cols<NC>(&ws.s2[tt][c0], k2);
#pragma unroll
                for (int m = 0; m < NC; ++m)
                    out[m] = k2[m] + gk[m] * dc_[m] + 2.0f * kc[m] * (c * lam[m] + da * dc_[m] + dn);
                store_cols<NC>(dk + g * K + c0, out);
                if (lane == 0) {
                    dbeta[g] = ws.sdb[tt] + db1;
                    if (dr) dr[g] = rc.x;
                }
            }
#pragma unroll
            for (int m = 0; m < NC; ++m) lam[m] = fmaf(rt, lam[m], fmaf(da, kc[m] * kc[m], gk[m] * kc[m]));
        }
        __syncwarp();      // every lane is done with this sub-chunk's buffers
    }
}

// One warp per (time segment, sequence) of L tokens, walking backwards.  The
// last segment starts from the exact lam_T = d_dT; every other one starts
// from lam = 0 kWarmAdj tokens past its end (or from the exact lam_T when the
// sequence ends sooner), walks that warm-up without output, records the lam
// it reaches at its end (its speculative start), then walks its own tokens
// with output and records lam at its first token, its share of deta and
// whether a map could expand.  With one segment (nseg = 1) the results are
// final: dd0 and deta are written here.
constexpr int kWarmAdj = 128;
template <typename io_t, int K>
__global__ void __launch_bounds__(kBwdSeqs * 32)
precond_adjoint_kernel(int BH, int T, int nsub, int L, int nseg, const io_t *__restrict__ k,
                       const float *__restrict__ beta, const float *__restrict__ r, float eta,
                       const float *__restrict__ dkt_tot, const float *__restrict__ ddT,
                       const float *__restrict__ dk2, const float *__restrict__ db2,
                       const float *__restrict__ ck, io_t *__restrict__ dk,
                       float *__restrict__ dbeta, float *__restrict__ dr,
                       float *__restrict__ dd0, float *__restrict__ deta,
                       float *__restrict__ ws_start, float *__restrict__ ws_end,
                       int *__restrict__ ws_flag, float *__restrict__ ws_eta) {
    constexpr int NC = K / 32;
    extern __shared__ __align__(16) uint8_t smem_walk[];
    WalkStage<io_t, K> *stages = reinterpret_cast<WalkStage<io_t, K> *>(smem_walk);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t id = (size_t)blockIdx.x * kBwdSeqs + warp;
    if (id >= (size_t)BH * nseg) return;        // whole warps only: no block barrier below
    const size_t seq = id / nseg;
    const int seg = (int)(id % nseg), c0 = lane * NC;
    const int tlo = seg * L, thi = min(T, tlo + L);
    float lam[NC];
    const int tend = seg == nseg - 1 ? T : min(T, thi + kWarmAdj);
    if (ddT && tend == T) {
        load_cols<NC>(ddT + seq * K + c0, lam);
    } else {
#pragma unroll
        for (int m = 0; m < NC; ++m) lam[m] = 0.0f;   // the warm-up forgets this
    }
    float deta_acc = 0.0f;
    bool expand = false;
    if (tend > thi)
        adjoint_walk<io_t, K>(T, nsub, seq, thi, tend, false, k, beta, r, eta, dkt_tot, dk2, db2,
                              ck, dk, dbeta, dr, stages[warp], lam, deta_acc, expand);
    if (nseg > 1) store_cols<NC>(ws_start + id * K + c0, lam);
    adjoint_walk<io_t, K>(T, nsub, seq, tlo, thi, true, k, beta, r, eta, dkt_tot, dk2, db2, ck,
                          dk, dbeta, dr, stages[warp], lam, deta_acc, expand);
    expand = __any_sync(kFullMask, expand);   // (deta_acc is the same on every lane)
    if (nseg > 1) {
        store_cols<NC>(ws_end + id * K + c0, lam);
        if (lane == 0) {
            ws_flag[id] = expand ? 1 : 0;
            ws_eta[id] = deta_acc;
        }
    } else {
        if (dd0) store_cols<NC>(dd0 + seq * K + c0, lam);
        if (deta && lane == 0) deta[seq] = deta_acc;
    }
}

// One warp per sequence: check each segment's speculative start (lam at its
// end) against the lam its successor reached at its first token, walking
// down from the last segment (whose start is exact), and recompute from that
// exact value every segment whose start is off by more than the acceptance
// bound relative to the largest entry (2^-21 fp32 I/O, 2^-13 bf16 I/O, as in
// the forward scan), or every segment when some map could expand.  Then
// dd0 = lam at token 0 and deta = the segments' shares in segment order.
template <typename io_t, int K>
__global__ void __launch_bounds__(32)
precond_adjoint_verify_kernel(int BH, int T, int nsub, int L, int nseg, const io_t *__restrict__ k,
                              const float *__restrict__ beta, const float *__restrict__ r,
                              float eta, const float *__restrict__ dkt_tot,
                              const float *__restrict__ dk2, const float *__restrict__ db2,
                              const float *__restrict__ ck, io_t *__restrict__ dk,
                              float *__restrict__ dbeta, float *__restrict__ dr,
                              float *__restrict__ dd0, float *__restrict__ deta,
                              const float *__restrict__ ws_start, float *__restrict__ ws_end,
                              const int *__restrict__ ws_flag, float *__restrict__ ws_eta) {
    constexpr int NC = K / 32;
    constexpr float tol = sizeof(io_t) == 2 ? 1.220703125e-04f : 4.76837158203125e-07f;
    extern __shared__ __align__(16) uint8_t smem_walk[];
    WalkStage<io_t, K> &stage = *reinterpret_cast<WalkStage<io_t, K> *>(smem_walk);
    const size_t seq = blockIdx.x;
    const int lane = threadIdx.x, c0 = lane * NC;
    const size_t base = seq * nseg;
    int f = 0;
    for (int i = lane; i < nseg; i += 32) f |= ws_flag[base + i];
    const bool all = __any_sync(kFullMask, f != 0);
    float prev[NC];   // the exact lam at the first token of segment i + 1
    load_cols<NC>(ws_end + (base + nseg - 1) * K + c0, prev);
    for (int i = nseg - 2; i >= 0; --i) {
        float cur[NC];
        load_cols<NC>(ws_start + (base + i) * K + c0, cur);
        float diff = 0.0f, mag = 0.0f;
#pragma unroll
        for (int m = 0; m < NC; ++m) {
            diff = fmaxf(diff, fabsf(cur[m] - prev[m]));
            mag = fmaxf(mag, fabsf(prev[m]));
        }
#pragma unroll
        for (int x = 16; x > 0; x >>= 1) {
            diff = fmaxf(diff, __shfl_xor_sync(kFullMask, diff, x));
            mag = fmaxf(mag, __shfl_xor_sync(kFullMask, mag, x));
        }
        if (all || !(diff <= tol * mag)) {   // recompute segment i from the exact start
            const int tlo = i * L, thi = min(T, tlo + L);
            float deta_acc = 0.0f;
            bool unused = false;
            adjoint_walk<io_t, K>(T, nsub, seq, tlo, thi, true, k, beta, r, eta, dkt_tot, dk2,
                                  db2, ck, dk, dbeta, dr, stage, prev, deta_acc, unused);
            store_cols<NC>(ws_end + (base + i) * K + c0, prev);
            if (lane == 0) ws_eta[base + i] = deta_acc;
        } else {
            load_cols<NC>(ws_end + (base + i) * K + c0, prev);
        }
        __syncwarp();
    }
    if (dd0) store_cols<NC>(dd0 + seq * K + c0, prev);
    if (deta) {
        __syncwarp();
        float e = 0.0f;
        for (int i = lane; i < nseg; i += 32) e += ws_eta[base + i];
        e = warp_sum(e);
        if (lane == 0) deta[seq] = e;
    }
}

// ---------------------------------------------------------------- host side
static size_t pad256(size_t x) { return (x + 255) & ~size_t(255); }

int precond_segments(int BH, int T, bool has_r, int *L_out);
size_t precond_scratch_bytes(int BH, int T, int K);
cudaError_t precond_checkpoint_launch(int io, int BH, int T, int K, const void *k,
                                      const float *beta, const float *r, float eta,
                                      const float *d0, float *dT, float *ecoef, float *dchk,
                                      int chk_shift, void *scratch, int *status,
                                      cudaStream_t stream);

// Scratch: Phase 2's state checkpoints (ck2) and row-block partials, the
// summed dktilde, Phase 2's shares of dk and dbeta, Phase 1's checkpoints of
// d every kBwdSub tokens (ck1) and the forward scan's segment scratch (p1),
// and the adjoint's time segments: lam at each segment's end (speculative
// start) and first token, flags and deta shares (the segments of the forward
// scan's rule, with a retention gate; sized for it in any case).
struct BwdScratch {
    float *ck2, *part, *gcarry, *dkt_tot, *dk2, *db2, *ck1, *p1, *a_start, *a_end, *a_flag, *a_eta;
};

static size_t bwd_layout(int BH, int T, int K, int V, bool pch, char *base, BwdScratch *s) {
    const size_t nsub = ((size_t)T + kBwdSub - 1) / kBwdSub;
    const size_t tw = T < kBwdWindow ? (size_t)T : (size_t)kBwdWindow;   // tokens of one window
    const size_t n = (size_t)BH * precond_segments(BH, T, true, nullptr);
    const size_t sz[12] = {
        pad256((size_t)BH * nsub * V * K * 4),                                   // ck2
        pad256((size_t)BH * (V / kBwdRows) * tw * bwd_part_width(K, pch) * 4),   // part
        pad256((size_t)BH * V * K * 4),                                           // gcarry
        pad256((size_t)BH * T * K * 4),                                           // dkt_tot
        pad256((size_t)BH * T * K * 4),                                           // dk2
        pad256((size_t)BH * T * 4),                                               // db2
        pad256((size_t)BH * nsub * K * 4),                                        // ck1
        pad256(precond_scratch_bytes(BH, T, K)),                                  // p1
        pad256(n * K * 4), pad256(n * K * 4), pad256(n * 4), pad256(n * 4),       // a_*
    };
    size_t off = 0;
    float **dst[12] = {&s->ck2, &s->part, &s->gcarry, &s->dkt_tot, &s->dk2, &s->db2, &s->ck1,
                       &s->p1, &s->a_start, &s->a_end, &s->a_flag, &s->a_eta};
    for (int a = 0; a < 12; ++a) {
        if (base) *dst[a] = reinterpret_cast<float *>(base + off);
        off += sz[a];
    }
    return off;
}

size_t backward_scratch_bytes(int BH, int T, int K, int V, bool per_channel) {
    BwdScratch s;
    return bwd_layout(BH, T, K, V, per_channel, nullptr, &s);
}

template <typename io_t, int K, bool PCH>
static cudaError_t launch_backward(int BH, int T, int V, const void *q, const void *k,
                                   const void *kt, const void *v, const float *beta,
                                   const float *r, float eta, const float *d0,
                                   const float *alpha, const float *S0, const void *dO,
                                   const float *dST, const float *ddT, const void *dkt_ext,
                                   void *dq, void *dk, void *dv, float *dbeta, float *dr,
                                   float *dalpha, float *dd0, float *dS0, float *deta,
                                   void *scratch, int *status, cudaStream_t stream) {
    static std::atomic<unsigned long long> attr_done{0};
    BwdScratch s;
    bwd_layout(BH, T, K, V, PCH, static_cast<char *>(scratch), &s);
    // Phase 1's d every kBwdSub tokens, by the (time-parallel) forward scan
    cudaError_t e = precond_checkpoint_launch(sizeof(io_t) == 2 ? OSDN_BF16 : OSDN_F32, BH, T, K, k,
                                              beta, r, eta, d0, nullptr, nullptr, s.ck1, 4, s.p1,
                                              status, stream);
    if (e != cudaSuccess) return e;
    const int nsub = T / kBwdSub + (T % kBwdSub != 0);   // no overflow near INT_MAX
    const int nrb = V / kBwdRows;
    const int smem = state_adjoint_smem_bytes<io_t, K, PCH>();
    auto *k1 = state_adjoint_kernel<io_t, K, PCH>;
    e = smem_attr_once(reinterpret_cast<const void *>(k1), smem, attr_done);
    if (e != cudaSuccess) return e;
    // the forward sweep, then the reverse sweep window by window (newest
    // first), each window's row-block partials summed before the next one
    // reuses their buffer
    const int Tw = T < kBwdWindow ? T : kBwdWindow;
    auto sweep = [&](int fwd, int tw0, int tw1) {
        k1<<<seq_grid(nrb, BH), kBwdRows * 32, smem, stream>>>(
            BH, T, V, nsub, static_cast<const io_t *>(q), static_cast<const io_t *>(k),
            static_cast<const io_t *>(kt), static_cast<const io_t *>(v), beta, alpha, S0,
            static_cast<const io_t *>(dO), dST, static_cast<io_t *>(dv), dS0, s.ck2, s.part, fwd,
            tw0, tw1, Tw, s.gcarry);
        return cudaGetLastError();
    };
    if ((e = sweep(1, 0, T)) != cudaSuccess) return e;
    for (int tw1 = T; tw1 > 0;) {
        const int tw0 = ((tw1 - 1) / kBwdWindow) * kBwdWindow, tn = tw1 - tw0;
        if ((e = sweep(0, tw0, tw1)) != cudaSuccess) return e;
        partial_sum_kernel<io_t, K, PCH><<<seq_grid(tn / kSumTok + (tn % kSumTok != 0), BH), 256, 0, stream>>>(
            BH, T, nrb, tw0, tn, Tw, s.part, static_cast<const io_t *>(dkt_ext),
            static_cast<io_t *>(dq), dalpha, s.dkt_tot, s.dk2, s.db2);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        tw1 = tw0;
    }
    // the Phase 1 adjoint in time segments (one per sequence without a
    // retention gate), then their verification
    int L = T;
    const int nseg = precond_segments(BH, T, r != nullptr, &L);
    const long long nw = (long long)BH * nseg;
    int *aflag = reinterpret_cast<int *>(s.a_flag);
    static std::atomic<unsigned long long> attr_adj{0}, attr_ver{0};
    constexpr int kWalk = (int)sizeof(WalkStage<io_t, K>);
    if ((e = smem_attr_once(reinterpret_cast<const void *>(precond_adjoint_kernel<io_t, K>),
                            kBwdSeqs * kWalk, attr_adj)) != cudaSuccess ||
        (e = smem_attr_once(reinterpret_cast<const void *>(precond_adjoint_verify_kernel<io_t, K>),
                            kWalk, attr_ver)) != cudaSuccess)
        return e;
    precond_adjoint_kernel<io_t, K><<<(unsigned)((nw + kBwdSeqs - 1) / kBwdSeqs), kBwdSeqs * 32,
                                      kBwdSeqs * kWalk, stream>>>(
        BH, T, nsub, L, nseg, static_cast<const io_t *>(k), beta, r, eta, s.dkt_tot, ddT, s.dk2,
        s.db2, s.ck1, static_cast<io_t *>(dk), dbeta, dr, dd0, deta, s.a_start, s.a_end, aflag,
        s.a_eta);
    if ((e = cudaGetLastError()) != cudaSuccess || nseg == 1) return e;
    precond_adjoint_verify_kernel<io_t, K><<<BH, 32, kWalk, stream>>>(
        BH, T, nsub, L, nseg, static_cast<const io_t *>(k), beta, r, eta, s.dkt_tot, s.dk2, s.db2,
        s.ck1, static_cast<io_t *>(dk), dbeta, dr, dd0, deta, s.a_start, s.a_end, aflag, s.a_eta);
    return cudaGetLastError();
}

cudaError_t backward_launch(int io, int BH, int T, int K, int V, const void *q, const void *k,
                            const void *kt, const void *v, const float *beta, const float *r,
                            float eta, const float *d0, const float *alpha, const float *S0,
                            const void *dO, const float *dST, const float *ddT,
                            const void *dkt_ext, void *dq, void *dk, void *dv, float *dbeta,
                            float *dr, float *dalpha, float *dd0, float *dS0, float *deta,
                            bool per_channel, void *scratch, int *status, cudaStream_t stream) {
#define OSDN_BWD(T_, K_, P_)                                                                  \
    return launch_backward<T_, K_, P_>(BH, T, V, q, k, kt, v, beta, r, eta, d0, alpha, S0,   \
                                       dO, dST, ddT, dkt_ext, dq, dk, dv, dbeta, dr, dalpha, \
                                       dd0, dS0, deta, scratch, status, stream)
#define OSDN_BWD_K(T_, P_)          \
    do {                            \
        if (K == 64) OSDN_BWD(T_, 64, P_); \
        OSDN_BWD(T_, 128, P_);      \
    } while (0)
    if (io == OSDN_BF16) {
        if (per_channel) OSDN_BWD_K(__nv_bfloat16, true);
        OSDN_BWD_K(__nv_bfloat16, false);
    }
    if (per_channel) OSDN_BWD_K(float, true);
    OSDN_BWD_K(float, false);
#undef OSDN_BWD_K
#undef OSDN_BWD
}

}  // namespace osdn
