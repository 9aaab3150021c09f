// phase1_scan.cu -- Phase 1 of OSDN: the O(K) preconditioner scan over the
// key stream (gist.science summary of arXiv 2605.13473, sections 2.2-2.3).
//
// Per sequence and token t, with w_t = k_t (.) k_t and n_t = ||k_t||^2:
//     ktilde_t = d_t (.) k_t
//     d_{t+1}  = r_t d_t + e_t w_t,   e_t = c_t (1 - beta_t <d_t, w_t>),
//     c_t      = eta beta_t / n_t      (c_t = 0 for a zero key)
// i.e. a descent step on h_t(d) = ((1 - beta_t <d, w_t>)^2 - 1) / (2 n_t)
// with retention r_t.
//
// Chunked evaluation (16 tokens per step; exact algebra, no approximation).
// Inside a chunk starting from d, with p_t = <d, w_t>, G_tu = <w_t, w_u>,
// rho_t = prod_{v<t} r_v and pi_ut = prod_{u<v<t} r_v:
//     <d_t, w_t> = rho_t p_t + sum_{u<t} pi_ut e_u G_tu
// so the 16 scalars e_t follow from one lower-triangular substitution,
//     e_t = c_t (1 - beta_t rho_t p_t) - c_t beta_t sum_{u<t} pi_ut G_tu e_u,
// after which every column of d steps through the chunk independently
// (ktilde_t = d (.) k_t, d <- r_t d + e_t w_t).  G only enters through the
// small coupling c beta G, so it is formed on the tensor cores (mma.sync,
// tf32 inputs, fp32 accumulation); p and n, which enter e directly, are
// reduced in fp32.
//
// One warp scans one stretch of one sequence: lane l owns the K/32
// consecutive columns from l K/32 (its part of d stays in registers), so a
// chunk needs no block barrier.  Per chunk the warp stages the keys in its
// own shared-memory ring (cp.async, four chunks in flight), reduces p and n
// by one transpose-reduce of 32 partial sums, forms G from the staged keys,
// runs the substitution on lanes 0..15 and steps its columns with packed
// fp32x2 arithmetic.
//
// Time segments.  With a retention gate the map d -> d_{t+1} contracts, so a
// segment can start from a state estimated by running the scan over the W
// tokens before it from d = 0 ("warm-up", 128 tokens).  Every segment
// records its estimated start and its end state; a
// second kernel checks each start against the predecessor's end and
// recomputes any segment whose estimate is off by more than a bound relative
// to the largest entry of that end state (2^-21 for fp32 I/O; 2^-13 for bf16
// I/O, a sixteenth of the rounding its ktilde is stored with), or all
// segments after a token whose one-step map could expand (||A_t||_2 > 1).
// An accepted start therefore differs from the state the sequential scan
// would carry into the segment by at most that bound; the maps contract
// (that is what the check on ||A_t|| guarantees), so such a difference
// shrinks through the segment and the differences of the accepted segments
// add up to at most about nseg times the bound, on top of fp32 rounding.
// Speculation only decides how much runs in parallel.
//
// Checkpoint mode (the fused forward pass).  Instead of (or besides)
// ktilde, the scan can write the coefficient e_t of every token and d at
// every 64-token boundary.  From those a later kernel rebuilds the
// preconditioner of any token of a 64-token chunk without a scan:
//     d_t = rho_t d_c + sum_{u<t} pi_ut e_u w_u   (rho, pi within the chunk)
// -- one small matrix product, which is how the fused forward's chunk
// preparation forms ktilde on chip.
//
// Residual diagnostic (optional).  Writing ktilde_t into the state scales
// the token's residual S k_t - v_t by 1 - beta_t <d_t, w_t> (section 3,
// theorem 5.2: f_t(S_t) / f_t(S_{t-1}) = (1 - beta_t <d_t, w_t>)^2), and the
// substitution above already forms that factor.  On request each sequence
// also gets sum_t log((1 - beta_t <d_t, w_t>)^2); its exp over T is the
// geometric-mean residual ratio q_geo of section 4.2.
#include <mutex>

#include "osdn_device.cuh"

namespace osdn {
namespace p1 {

constexpr int C = 16;          // tokens per chunk
constexpr int NST = 4;         // key chunks in flight per warp
constexpr int kWarm = 128;     // longest warm-up in front of a speculative segment
constexpr int kMinSeg = 256;   // shortest segment
constexpr int kMaxWarps = 4;   // warps (segments) per CTA
constexpr int kDefaultSms = 152;  // GB300; used only when no device can be queried
constexpr float kRelTol = 4.76837158203125e-07f;  // 2^-21

// The acceptance bound of a speculative start, relative to the largest entry
// of the predecessor's end state: 2^-21 for fp32 I/O; for bf16 I/O, whose
// ktilde carries a rounding of 2^-9 anyway, 2^-13 (a sixteenth of that), so
// that a retention too slow to forget the guess to fp32 precision in the
// warm-up does not force a repair the output could not tell from it.
template <typename io_t>
struct Spec {
    static constexpr int warm = kWarm;
    static constexpr float tol = sizeof(io_t) == 2 ? 1.220703125e-04f : kRelTol;
};

// One warp's staging area.  Key rows are padded by 8 elements so that the
// Gram fragment loads (rows g and g+8, two columns per lane) hit 32 banks.
template <typename io_t, int K>
struct WarpSmem {
    static constexpr int KP = K + 8;
    alignas(16) io_t keys[NST][C][KP];
    alignas(16) float gb[NST][C];   // beta of the staged chunk
    alignas(16) float gr[NST][C];   // r of the staged chunk
    alignas(16) float sG[2][C][20]; // Gram (and n_t in column 16) of two chunks
    alignas(16) float4 sER[C];      // (e_t, e_t, r_t, r_t)
};

struct Params {
    int BH, T, L, nseg;
    const void *k;
    const float *beta, *r, *d0;
    float eta;
    void *ktilde;               // or NULL (checkpoint mode without ktilde)
    float *dT;
    float *ecoef;               // [BH][T] e_t, or NULL
    float *dchk;                // [BH][ceil(T/I)][K] d at tokens 0, I, 2 I, ..., or NULL
    int chk_shift;              // log2 of the checkpoint interval I (6: 64 tokens; 4: 16)
    float *ws_start, *ws_end;   // [BH][nseg][K]
    int *ws_flag;               // [BH][nseg]
    float *ws_lr;               // [BH][nseg] residual log-ratio of each segment
    float *logratio;            // [BH] residual log-ratio of each sequence, or NULL
    int *status;
};

__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    const int sz = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(src), "r"(sz)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src, bool valid) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    const int sz = valid ? 4 : 0;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(s), "l"(src), "r"(sz)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void mbar_init_cta(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(bar))),
                 "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_cta(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(bar)))
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_parity(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar))), "r"(parity)
        : "memory");
    return ok != 0;
}
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// fp32 -> tf32 operand, rounded to nearest (ties away from zero): add half a
// tf32 unit in the last place; the tensor core ignores the 13 low bits.  One
// integer add instead of the conversion instruction's NaN handling; operands
// here are squares of finite keys.
__device__ __forceinline__ uint32_t to_tf32(float x) { return __float_as_uint(x) + 0x1000u; }
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
}
__device__ __forceinline__ uint32_t f2_to_bf2(float2 x) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x.x, x.y);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float2 splat(float x) { return make_float2(x, x); }
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(kFullMask, x, m);
    return x;
}
__device__ __forceinline__ float2 ld_pair(const float *p) { return *reinterpret_cast<const float2 *>(p); }
__device__ __forceinline__ float2 ld_pair(const __nv_bfloat16 *p) {
    return bf2_to_f2(*reinterpret_cast<const uint32_t *>(p));
}

// EP consecutive element pairs (a lane's columns) as fp32.
template <int EP>
__device__ __forceinline__ void ld_pairs(const float *p, float2 (&x)[EP]) {
    if constexpr (EP == 2) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        x[0] = make_float2(v.x, v.y);
        x[1] = make_float2(v.z, v.w);
    } else {
        x[0] = *reinterpret_cast<const float2 *>(p);
    }
}
template <int EP>
__device__ __forceinline__ void ld_pairs(const __nv_bfloat16 *p, float2 (&x)[EP]) {
    if constexpr (EP == 2) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        x[0] = bf2_to_f2(u.x);
        x[1] = bf2_to_f2(u.y);
    } else {
        x[0] = bf2_to_f2(*reinterpret_cast<const uint32_t *>(p));
    }
}
template <int EP>
__device__ __forceinline__ void st_pairs(float *p, const float2 (&x)[EP]) {
    if constexpr (EP == 2)
        *reinterpret_cast<float4 *>(p) = make_float4(x[0].x, x[0].y, x[1].x, x[1].y);
    else
        *reinterpret_cast<float2 *>(p) = x[0];
}
template <int EP>
__device__ __forceinline__ void st_pairs(__nv_bfloat16 *p, const float2 (&x)[EP]) {
    if constexpr (EP == 2)
        *reinterpret_cast<uint2 *>(p) = make_uint2(f2_to_bf2(x[0]), f2_to_bf2(x[1]));
    else
        *reinterpret_cast<uint32_t *>(p) = f2_to_bf2(x[0]);
}

// The half of a chunk's step that does not depend on d, formed while the
// previous chunk runs its chain.
//
// Gram: G_tu = <w_t, w_u> on the tensor cores, and n_t = ||k_t||^2 summed
// in fp32 from the same fragments.  The reduction index of k-step s8 visits
// columns 8 s8 .. 8 s8 + 7 in the order that puts a lane's two A elements
// next to each other (positions q and q + 4 are columns 8 s8 + 2q and
// 8 s8 + 2q + 1); any order gives the same sum.  B = A^T, so its fragments
// are A's.  Two accumulators per tile (even and odd k-steps) halve the mma
// chain.  finish() leaves G in sG and n_t in column 16 of row t.
template <typename io_t, int K>
struct GramPass {
    float acc[2][2][4];
    float2 n0, n1;
    __device__ __forceinline__ void start() {
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[a][b][i] = 0.f;
        n0 = n1 = make_float2(0.f, 0.f);
    }
    __device__ __forceinline__ void step(const io_t (*kr)[K + 8], int g, int q, int s8) {
        float2 x0 = ld_pair(&kr[g][8 * s8 + 2 * q]);
        float2 x1 = ld_pair(&kr[g + 8][8 * s8 + 2 * q]);
        x0 = __fmul2_rn(x0, x0);
        x1 = __fmul2_rn(x1, x1);
        n0 = __fadd2_rn(n0, x0);
        n1 = __fadd2_rn(n1, x1);
        const uint32_t a[4] = {to_tf32(x0.x), to_tf32(x1.x), to_tf32(x0.y), to_tf32(x1.y)};
        mma_tf32(acc[s8 & 1][0], a, a[0], a[2]);
        mma_tf32(acc[s8 & 1][1], a, a[1], a[3]);
    }
    __device__ __forceinline__ void finish(float (*sG)[20], int g, int q) {
        float ng = n0.x + n0.y, ng8 = n1.x + n1.y;   // rows g and g + 8, this lane's columns
        ng += __shfl_xor_sync(kFullMask, ng, 1);
        ng8 += __shfl_xor_sync(kFullMask, ng8, 1);
        ng += __shfl_xor_sync(kFullMask, ng, 2);
        ng8 += __shfl_xor_sync(kFullMask, ng8, 2);
        float gs[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) gs[nt][i] = acc[0][nt][i] + acc[1][nt][i];
        *reinterpret_cast<float2 *>(&sG[g][2 * q]) = make_float2(gs[0][0], gs[0][1]);
        *reinterpret_cast<float2 *>(&sG[g][8 + 2 * q]) = make_float2(gs[1][0], gs[1][1]);
        *reinterpret_cast<float2 *>(&sG[g + 8][2 * q]) = make_float2(gs[0][2], gs[0][3]);
        *reinterpret_cast<float2 *>(&sG[g + 8][8 + 2 * q]) = make_float2(gs[1][2], gs[1][3]);
        if (q == 0) {
            sG[g][C] = ng;
            sG[g + 8][C] = ng8;
        }
    }
};

// Coupling row of token t = lane & 15: coef_u = c_t beta_t pi_ut G_tu (u < t),
// c_t, and c_t beta_t rho_t, so that on the chain
//     e_t = c_t - c_t beta_t rho_t p_t - sum_u coef_u e_u.
// Also flags a token whose one-step map could expand
// (||A_t|| = max(|r_t|, |r_t - lambda_t|), lambda_t = eta beta_t^2 |w_t|^2 / n_t).
// step(u) runs u = C-1 down to 0.  With LR it also keeps the same row
// without the factor c_t (coefy, by), for the residual factor
//     y_t = 1 - beta_t <d_t, w_t> = 1 - beta_t rho_t p_t - sum_u coefy_u e_u.
template <bool HAS_R, bool LR>
struct CoefPass {
    float coef[C], coefy[LR ? C : 1];
    float ct, cbr, by, rt;
    float grow[C], rr[C], cb, bt, pi;
    __device__ __forceinline__ void start(const float *gb, const float *gr, const float (*sG)[20],
                                          int t, int nv, float eta, bool &expand) {
#pragma unroll
        for (int u = 0; u < C; u += 4) {
            const float4 g4 = *reinterpret_cast<const float4 *>(&sG[t][u]);
            grow[u] = g4.x; grow[u + 1] = g4.y; grow[u + 2] = g4.z; grow[u + 3] = g4.w;
            if (HAS_R) {
                const float4 r4 = *reinterpret_cast<const float4 *>(&gr[u]);
                rr[u] = r4.x; rr[u + 1] = r4.y; rr[u + 2] = r4.z; rr[u + 3] = r4.w;
            }
        }
        const float nt = sG[t][C];
        const float gtt = sG[t][t];
        bt = gb[t];
        rt = HAS_R ? gr[t] : 1.0f;
        const float inv_n = nt > 0.0f ? __frcp_rn(nt) : 0.0f;
        ct = eta * bt * inv_n;
        cb = ct * bt;
        pi = 1.0f;
        const float lam = cb * gtt;
        const float nrm = fmaxf(fabsf(rt), fabsf(rt - lam));
        if (t < nv && nrm > 1.0f + 1e-6f) expand = true;
    }
    __device__ __forceinline__ void step(int t, int u) {
        coef[u] = (u < t) ? cb * pi * grow[u] : 0.0f;
        if (LR) coefy[u] = (u < t) ? bt * pi * grow[u] : 0.0f;
        if (HAS_R && u < t) pi *= rr[u];
    }
    __device__ __forceinline__ void finish() {
        cbr = cb * pi;
        by = bt * pi;
    }
};

// Scan tokens [tb, te) of sequence `seq` with one warp, starting from this
// lane's part of the state in `d`; ktilde is written for tokens >= tseg.
// Returns the state after te in `d`; sets `expand` if some token's one-step
// map could expand.  All 32 lanes call this together.
//
// Software-pipelined: while chunk j runs its chain (p from d, the 16-step
// substitution, the column steps), the warp forms chunk j+1's Gram, n and
// coupling rows, which do not depend on d.
//
// With LR, lanes 0..15 add log(y_t^2) of every token >= tseg to `lr`.
template <typename io_t, int K, bool HAS_R, bool LR>
__device__ void warp_scan(const Params &p, WarpSmem<io_t, K> &st, int seq, int tb, int tseg,
                          int te, float2 (&d)[K / 64], bool &expand, float &lr) {
    constexpr int EP = K / 64;                      // element pairs per lane
    constexpr int E = 2 * EP;                       // columns per lane
    constexpr int EPP = 16 / (int)sizeof(io_t);     // elements per 16-byte piece
    constexpr int PR = K / EPP;                     // pieces per key row
    constexpr int KS = K / 8;                       // Gram k-steps
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;   // mma fragment coordinates
    const int t = lane & (C - 1);            // the token this lane solves for
    const io_t *kseq = static_cast<const io_t *>(p.k) + (size_t)seq * p.T * K;
    io_t *ktseq = p.ktilde ? static_cast<io_t *>(p.ktilde) + (size_t)seq * p.T * K : nullptr;
    const float *bseq = p.beta + (size_t)seq * p.T;
    const float *rseq = HAS_R ? p.r + (size_t)seq * p.T : nullptr;
    const int nc = (te - tb + C - 1) / C;
    const int cs = p.chk_shift;
    const size_t nchk = ((size_t)p.T + (1u << cs) - 1) >> cs;   // checkpoints per sequence

    auto issue = [&](int j) {
        if (j < nc) {
            const int s = j % NST, t0 = tb + j * C;
#pragma unroll
            for (int i = lane; i < C * PR; i += 32) {
                const int tt = i / PR, pc = i % PR;
                const bool valid = t0 + tt < te;
                const io_t *src = valid ? kseq + (size_t)(t0 + tt) * K + pc * EPP : kseq;
                cp_async16(&st.keys[s][tt][pc * EPP], src, valid);
            }
            // lanes 0..15 fetch beta, lanes 16..31 r (when there is one)
            const bool valid = t0 + t < te && (HAS_R || lane < C);
            const float *src = lane < C ? bseq : rseq;
            float *dst = lane < C ? &st.gb[s][t] : &st.gr[s][t];
            cp_async4(dst, valid ? src + t0 + t : bseq, valid);
        }
        cp_commit();
    };
#pragma unroll
    for (int j = 0; j < NST - 1; ++j) issue(j);

    GramPass<io_t, K> gp;
    CoefPass<HAS_R, LR> cf;
    // chunk 0's input-only half
    cp_wait<NST - 2>();
    __syncwarp();
    gp.start();
#pragma unroll
    for (int s8 = 0; s8 < KS; ++s8) gp.step(st.keys[0], g, q, s8);
    gp.finish(st.sG[0], g, q);
    __syncwarp();
    cf.start(st.gb[0], st.gr[0], st.sG[0], t, min(C, te - tb), p.eta, expand);
#pragma unroll
    for (int u = C - 1; u >= 0; --u) cf.step(t, u);
    cf.finish();

    for (int j = 0; j < nc; ++j) {
        issue(j + NST - 1);
        cp_wait<NST - 2>();   // chunks j and j+1 have landed
        __syncwarp();
        const int s = j % NST, s1 = (j + 1) % NST, t0 = tb + j * C;
        const int nv = min(C, te - t0);
        // chunk j+1's stage may be empty past the end; its results are then unused
        const io_t(*kr1)[K + 8] = st.keys[s1];

        // ---- chain: this lane's columns, w = k^2, partial p --------------------
        float2 kk[C][EP], w[C][EP];
        float v[C];
#pragma unroll
        for (int u = 0; u < C; ++u) {
            ld_pairs<EP>(&st.keys[s][u][E * lane], kk[u]);
            float2 pp = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                w[u][e] = __fmul2_rn(kk[u][e], kk[u][e]);
                pp = __ffma2_rn(d[e], w[u][e], pp);
            }
            v[u] = pp.x + pp.y;
        }

        // ---- off the chain: chunk j+1's Gram and n ------------------------------
        gp.start();
#pragma unroll
        for (int s8 = 0; s8 < KS; ++s8) gp.step(kr1, g, q, s8);
        gp.finish(st.sG[(j + 1) & 1], g, q);

        // ---- chain: reduce p; lanes 2t and 2t+1 end with p_t --------------------
#pragma unroll
        for (int off = 16, n = 8; off >= 2; off >>= 1, n >>= 1) {
            const bool hi = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < n; ++i) {
                const float keep = hi ? v[i + n] : v[i];
                const float send = hi ? v[i] : v[i + n];
                v[i] = keep + __shfl_xor_sync(kFullMask, send, off);
            }
        }
        v[0] += __shfl_xor_sync(kFullMask, v[0], 1);
        const float pt = __shfl_sync(kFullMask, v[0], 2 * t);

        // ---- chain: the 16-step substitution for e_t ----------------------------
        float acc = cf.ct - cf.cbr * pt;
        float accy = 1.0f - cf.by * pt;
#pragma unroll
        for (int u = 0; u < C - 1; ++u) {
            const float eu = __shfl_sync(kFullMask, acc, u);
            acc = fmaf(-cf.coef[u], eu, acc);
            if (LR) accy = fmaf(-cf.coefy[u], eu, accy);
        }
        if (LR && lane < C && t < nv && t0 + t >= tseg) lr += logf(accy * accy);
        if (lane < C) {
            const float et = t < nv ? acc : 0.0f, rt = t < nv ? cf.rt : 1.0f;
            st.sER[t] = make_float4(et, et, rt, rt);
            if (p.ecoef && t < nv && t0 >= tseg) p.ecoef[(size_t)seq * p.T + t0 + t] = et;
        }
        if (p.dchk && (t0 & ((1 << cs) - 1)) == 0 && t0 >= tseg)   // d entering a checkpoint interval
            st_pairs<EP>(p.dchk + ((size_t)seq * nchk + (t0 >> cs)) * K + E * lane, d);
        __syncwarp();

        // ---- chain: this lane's columns through the chunk; emit ktilde ----------
        const int nst = (t0 >= tseg && ktseq) ? nv : 0;   // tokens of this chunk to emit
        io_t *kst = ktseq ? ktseq + (size_t)t0 * K + E * lane : nullptr;
#pragma unroll
        for (int u = 0; u < C; ++u) {
            const float4 er = st.sER[u];
            float2 kt[EP];
#pragma unroll
            for (int e = 0; e < EP; ++e) kt[e] = __fmul2_rn(d[e], kk[u][e]);
            if (u < nst) st_pairs<EP>(kst + u * K, kt);
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                const float2 rd = HAS_R ? __fmul2_rn(make_float2(er.z, er.w), d[e]) : d[e];
                d[e] = __ffma2_rn(make_float2(er.x, er.y), w[u][e], rd);
            }
        }

        // ---- off the chain: chunk j+1's coupling rows ---------------------------
        cf.start(st.gb[s1], st.gr[s1], st.sG[(j + 1) & 1], t, min(C, te - t0 - C), p.eta, expand);
#pragma unroll
        for (int u = C - 1; u >= 0; --u) cf.step(t, u);
        cf.finish();
    }
    cp_wait<0>();
    __syncwarp();
}

// ---------------------------------------------------------------------------
// A whole sequence on one CTA, for scans that run in a single segment (no
// retention gate, or too few tokens to segment).  The state then has no
// other parallelism, so the chunk's work is split to shorten its serial
// path:
//   chain warps 0 .. K/32-1   lane l of warp w owns column 32 w + l of d;
//                             per chunk: the partial p_t = <d, w_t> over its
//                             columns, one cross-warp sum, e = X b (a 16 x 16
//                             mat-vec, computed by every chain warp alike),
//                             then its column's 16 steps and ktilde stores;
//   solver warps K/32 .. +3   take every fourth chunk, ahead of the chain:
//                             the Gram, n_t and the coupling rows (as in the
//                             warp scan above), then X = (I + N)^-1 of the
//                             coupling matrix N by column substitution, handed
//                             over in shared memory.
// With b_t = c_t - c_t beta_t rho_t p_t the coefficients of the chunk are
// e = X b, the same numbers the warp scan's substitution forms on its chain.
constexpr int kSolvers = 4;
constexpr int kSolverStages = 3;   // key chunks in flight per solver warp
constexpr int kChainStages = 4;    // key chunks in flight per chain warp

template <typename io_t, int K>
struct CtaSmem {
    static constexpr int KP = K + 8;
    static constexpr int NW = K / 32;
    alignas(16) io_t skeys[kSolvers][kSolverStages][C][KP];   // solver key rings
    alignas(16) float sgb[kSolvers][kSolverStages][C];
    alignas(16) float sgr[kSolvers][kSolverStages][C];
    alignas(16) float sG[kSolvers][C][20];                    // Gram and n_t (column 16)
    alignas(16) float sN[kSolvers][C][C + 4];                 // coupling rows, then X
    alignas(16) float sNy[kSolvers][C][C + 4];                // coupling rows without c (LR)
    alignas(16) float4 sS[kSolvers][C];                       // (c_t, c_t b_t rho_t, r_t, b_t rho_t)
    alignas(16) io_t ckeys[NW][kChainStages][C][32];          // chain key rings: own columns
    alignas(16) float part[2][NW][C];                         // per-warp partial p_t
    alignas(16) float sR[kSolvers][C];                        // r_t (1 past T)
    alignas(16) float be[NW][2][C];                           // per chain warp: b, then e
    uint64_t xr[kSolvers], xc[kSolvers];                      // X ready / consumed
    int abort_flag;
};

__device__ __forceinline__ bool cta_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         int *status) {
    for (uint32_t i = 0; i < (1u << 26); ++i) {
        if (mbar_try_wait_parity(bar, parity)) return true;
        if ((i & 255u) == 255u && *abort_flag) return false;
    }
    report_status(status, OSDN_ERR_TIMEOUT);
    *abort_flag = 1;
    return false;
}

// CHK: checkpoint mode (e_t and d every 2^chk_shift tokens; ktilde may be NULL).
template <typename io_t, int K, bool HAS_R, bool LR, bool CHK>
__global__ void __launch_bounds__(32 * (K / 32 + kSolvers)) precond_cta_kernel(Params p) {
    using SM = CtaSmem<io_t, K>;
    constexpr int NW = K / 32;
    constexpr int EPP = 16 / (int)sizeof(io_t);   // elements per 16-byte piece
    constexpr int PR = K / EPP;                   // pieces per key row
    constexpr int KS = K / 8;                     // Gram k-steps
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SM &sm = *reinterpret_cast<SM *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seq = blockIdx.x, T = p.T, nc = (T + C - 1) / C;
    const io_t *kseq = static_cast<const io_t *>(p.k) + (size_t)seq * T * K;
    volatile int *abort_flag = &sm.abort_flag;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSolvers; ++i) {
            mbar_init_cta(&sm.xr[i], 1);
            mbar_init_cta(&sm.xc[i], NW);
        }
        sm.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp >= NW) {
        // ================================================= solver warp
        const int sv = warp - NW;
        const int g = lane >> 2, q = lane & 3, t = lane & (C - 1);
        const float *bseq = p.beta + (size_t)seq * T;
        const float *rseq = HAS_R ? p.r + (size_t)seq * T : nullptr;
        const int nmine = nc > sv ? (nc - sv + kSolvers - 1) / kSolvers : 0;
        auto issue = [&](int m) {
            if (m < nmine) {
                const int s = m % kSolverStages, t0 = (sv + m * kSolvers) * C;
#pragma unroll
                for (int i = lane; i < C * PR; i += 32) {
                    const int tt = i / PR, pc = i % PR;
                    const bool valid = t0 + tt < T;
                    const io_t *src = valid ? kseq + (size_t)(t0 + tt) * K + pc * EPP : kseq;
                    cp_async16(&sm.skeys[sv][s][tt][pc * EPP], src, valid);
                }
                const bool valid = t0 + t < T && (HAS_R || lane < C);
                const float *src = lane < C ? bseq : rseq;
                float *dst = lane < C ? &sm.sgb[sv][s][t] : &sm.sgr[sv][s][t];
                cp_async4(dst, valid ? src + t0 + t : bseq, valid);
            }
            cp_commit();
        };
#pragma unroll
        for (int m = 0; m < kSolverStages - 1; ++m) issue(m);
        GramPass<io_t, K> gp;
        CoefPass<HAS_R, LR> cf;
        bool unused = false;
        for (int m = 0; m < nmine; ++m) {
            issue(m + kSolverStages - 1);
            cp_wait<kSolverStages - 1>();
            __syncwarp();
            const int s = m % kSolverStages, t0 = (sv + m * kSolvers) * C, nv = min(C, T - t0);
            gp.start();
#pragma unroll
            for (int s8 = 0; s8 < KS; ++s8) gp.step(sm.skeys[sv][s], g, q, s8);
            // the chain has consumed this solver's previous X
            bool ok = true;
            if (m >= 1) ok = cta_wait(&sm.xc[sv], (m - 1) & 1, abort_flag, p.status);
            if (!__all_sync(kFullMask, ok)) break;
            gp.finish(sm.sG[sv], g, q);
            __syncwarp();
            cf.start(sm.sgb[sv][s], sm.sgr[sv][s], sm.sG[sv], t, nv, p.eta, unused);
#pragma unroll
            for (int u = C - 1; u >= 0; --u) cf.step(t, u);
            cf.finish();
            if (lane < C) {
#pragma unroll
                for (int u = 0; u < C; ++u) {
                    sm.sN[sv][t][u] = cf.coef[u];
                    if (LR) sm.sNy[sv][t][u] = cf.coefy[u];
                }
                sm.sS[sv][t] = make_float4(cf.ct, cf.cbr, t < nv ? cf.rt : 1.0f, cf.by);
                sm.sR[sv][t] = t < nv ? cf.rt : 1.0f;
            }
            __syncwarp();
            // X = (I + N)^-1, lane u < 16 forming column u; rows of N read
            // before the column overwrites them (every lane reads row i
            // while the lanes' x_i of earlier rows are in registers)
            float x[C];
#pragma unroll
            for (int i = 0; i < C; ++i) {
                float part4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int k4 = 0; k4 < i; k4 += 4) {
                    const float4 n4 = *reinterpret_cast<const float4 *>(&sm.sN[sv][i][k4]);
                    const float nn[4] = {n4.x, n4.y, n4.z, n4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (k4 + e < i) part4[e] = fmaf(nn[e], x[k4 + e], part4[e]);
                }
                x[i] = ((i == t) ? 1.0f : 0.0f) - ((part4[0] + part4[1]) + (part4[2] + part4[3]));
            }
            __syncwarp();
            if (lane < C) {
#pragma unroll
                for (int i = 0; i < C; ++i) sm.sN[sv][i][t] = x[i];   // X[i][t]
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_cta(&sm.xr[sv]);
        }
        cp_wait<0>();
        __syncwarp();
    } else {
        // ================================================= chain warp
        const int w = warp, col = 32 * w + lane;
        io_t *ktseq = (!CHK || p.ktilde) ? static_cast<io_t *>(p.ktilde) + (size_t)seq * T * K : nullptr;
        const int chs = p.chk_shift;
        const size_t nchk = ((size_t)T + (1u << chs) - 1) >> chs;   // checkpoints per sequence
        // this warp's 32 columns of a chunk's 16 keys, staged by cp.async:
        // 4-byte pieces, lane l copying piece l of every row (bf16: 16 lanes
        // cover the 64-byte row, fp32: 32 lanes the 128-byte row)
        constexpr int PW = 32 * (int)sizeof(io_t) / 4;   // 4-byte pieces per row
        auto issue = [&](int j) {
            if (j < nc) {
                const int s = j % kChainStages, t0 = j * C;
#pragma unroll
                for (int i = lane; i < C * PW; i += 32) {
                    const int tt = i / PW, pc = i % PW;
                    const bool valid = t0 + tt < T;
                    const io_t *src = valid ? kseq + (size_t)(t0 + tt) * K + 32 * w + pc * (4 / (int)sizeof(io_t)) : kseq;
                    cp_async4(reinterpret_cast<uint8_t *>(&sm.ckeys[w][s][tt][0]) + 4 * pc, src, valid);
                }
            }
            cp_commit();
        };
#pragma unroll
        for (int j = 0; j < kChainStages - 1; ++j) issue(j);
        float d = p.d0 ? p.d0[(size_t)seq * K + col] : 1.0f;
        float lr = 0.0f;
        for (int j = 0; j < nc; ++j) {
            issue(j + kChainStages - 1);
            cp_wait<kChainStages - 1>();
            __syncwarp();
            const int s = j % kChainStages, sv = j % kSolvers, t0 = j * C, nv = min(C, T - t0);
            float kk[C], ww[C], v[C];
#pragma unroll
            for (int u = 0; u < C; ++u) {
                kk[u] = to_f32(sm.ckeys[w][s][u][lane]);
                ww[u] = kk[u] * kk[u];
                v[u] = d * ww[u];
            }
            // p_t over this warp's columns: lanes 2t and 2t+1 end with it
#pragma unroll
            for (int off = 16, n = 8; off >= 2; off >>= 1, n >>= 1) {
                const bool hi = (lane & off) != 0;
#pragma unroll
                for (int i = 0; i < n; ++i) {
                    const float keep = hi ? v[i + n] : v[i];
                    const float send = hi ? v[i] : v[i + n];
                    v[i] = keep + __shfl_xor_sync(kFullMask, send, off);
                }
            }
            v[0] += __shfl_xor_sync(kFullMask, v[0], 1);
            if ((lane & 1) == 0) sm.part[j & 1][w][lane >> 1] = v[0];
            const bool ok = cta_wait(&sm.xr[sv], (j / kSolvers) & 1, abort_flag, p.status);
            asm volatile("bar.sync 1, %0;" ::"n"(32 * NW) : "memory");
            if (!__all_sync(kFullMask, ok) || *abort_flag) break;
            // e = X b: lane t < 16 forms b_t, every lane reads all of b and
            // its row of X as float4 (this warp's own copy of b and e)
            const int t = lane & (C - 1);
            const float4 cs = sm.sS[sv][t];
            float pt = 0.0f;
#pragma unroll
            for (int ww2 = 0; ww2 < NW; ++ww2) pt += sm.part[j & 1][ww2][t];
            if (lane < C) sm.be[w][0][t] = cs.x - cs.y * pt;
            __syncwarp();
            float acc4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int u4 = 0; u4 < C; u4 += 4) {
                const float4 x4 = *reinterpret_cast<const float4 *>(&sm.sN[sv][t][u4]);
                const float4 b4 = *reinterpret_cast<const float4 *>(&sm.be[w][0][u4]);
                acc4[0] = fmaf(x4.x, b4.x, acc4[0]);
                acc4[1] = fmaf(x4.y, b4.y, acc4[1]);
                acc4[2] = fmaf(x4.z, b4.z, acc4[2]);
                acc4[3] = fmaf(x4.w, b4.w, acc4[3]);
            }
            const float et = t < nv ? (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]) : 0.0f;
            if (lane < C) sm.be[w][1][t] = et;
            if (CHK && p.ecoef && w == 0 && lane < C && t < nv) p.ecoef[(size_t)seq * T + t0 + t] = et;
            if (CHK && p.dchk && (t0 & ((1 << chs) - 1)) == 0)   // d entering a checkpoint interval
                p.dchk[((size_t)seq * nchk + (t0 >> chs)) * K + col] = d;
            __syncwarp();
            if (LR) {   // the residual factor y_t = 1 - b_t rho_t p_t - sum_u Ny_tu e_u
                float y4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int u4 = 0; u4 < C; u4 += 4) {
                    const float4 n4 = *reinterpret_cast<const float4 *>(&sm.sNy[sv][t][u4]);
                    const float4 e4 = *reinterpret_cast<const float4 *>(&sm.be[w][1][u4]);
                    y4[0] = fmaf(n4.x, e4.x, y4[0]);
                    y4[1] = fmaf(n4.y, e4.y, y4[1]);
                    y4[2] = fmaf(n4.z, e4.z, y4[2]);
                    y4[3] = fmaf(n4.w, e4.w, y4[3]);
                }
                const float y = 1.0f - cs.w * pt - ((y4[0] + y4[1]) + (y4[2] + y4[3]));
                if (w == 0 && lane < C && t < nv) lr += logf(y * y);
            }
            // this column through the chunk
            io_t *kst = (!CHK || ktseq) ? ktseq + (size_t)t0 * K + col : nullptr;
            const int nst = (!CHK || ktseq) ? nv : 0;   // tokens of this chunk to emit
#pragma unroll
            for (int u4 = 0; u4 < C; u4 += 4) {
                const float4 e4 = *reinterpret_cast<const float4 *>(&sm.be[w][1][u4]);
                const float4 r4 = HAS_R ? *reinterpret_cast<const float4 *>(&sm.sR[sv][u4])
                                        : make_float4(1.f, 1.f, 1.f, 1.f);
                const float ev[4] = {e4.x, e4.y, e4.z, e4.w}, rv[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int u = u4 + e;
                    if (u < nst) from_f32(kst[(size_t)u * K], d * kk[u]);
                    d = fmaf(ev[e], ww[u], HAS_R ? rv[e] * d : d);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_cta(&sm.xc[sv]);
        }
        cp_wait<0>();
        __syncwarp();
        if (p.dT) p.dT[(size_t)seq * K + col] = d;
        if (LR && w == 0) {
            lr = warp_sum(lr);
            if (lane == 0) p.logratio[seq] = lr;
        }
    }
}

// Warm-up length of speculative segment starting at tseg (all 32 lanes call
// this).  The start is estimated by scanning the W tokens before it from
// d = 0; the estimate's error is the exact state at tseg - W carried through
// those W steps, whose maps have norm max(|r_t|, |r_t - lambda_t|) -- r_t
// unless a step is so large that the map may expand, and then the verify
// kernel recomputes every segment anyway.  So the error is at most the
// product of r over the W tokens times the 2-norm of that state, which is
// at most sqrt(K) <= 2^4 times its largest entry.  W is the shortest
// multiple of 16 up to kWarm whose product of r lies below the acceptance
// bound / 2^5 (a margin of 2 for the state's drift over the warm-up).  A
// start that still misses the bound is recomputed, so W only decides speed.
template <typename io_t>
__device__ __forceinline__ int warm_tokens(const Params &p, int seq, int tseg, int lane) {
    // lane l: the product of r over the four tokens tseg - 4 (l + 1) .. tseg - 4 l - 1
    const float *rs = p.r + (size_t)seq * p.T + tseg - 4 * (lane + 1);
    float pr = (rs[0] * rs[1]) * (rs[2] * rs[3]);
    // inclusive product over lanes 0..l: the product of r over the last 4 (l + 1) tokens
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(kFullMask, pr, off);
        if (lane >= off) pr *= y;
    }
    const float bound = Spec<io_t>::tol * (1.0f / 32.0f);
    const unsigned ok = __ballot_sync(kFullMask, (lane & 3) == 3 && fabsf(pr) <= bound);
    return ok ? 4 * (__ffs(ok)) : kWarm;   // first lane 4 m + 3 that passes: W = 16 (m + 1)
}

// One warp per (segment, sequence): warp id = segment + nseg * sequence.
template <typename io_t, int K, bool HAS_R, bool LR>
__global__ void __launch_bounds__(32 * kMaxWarps) precond_segment_kernel(Params p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    constexpr int EP = K / 64, E = 2 * EP;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int id = blockIdx.x * (blockDim.x >> 5) + warp;
    if (id >= p.BH * p.nseg) return;
    WarpSmem<io_t, K> &st = reinterpret_cast<WarpSmem<io_t, K> *>(smem_raw)[warp];
    const int seq = id / p.nseg, seg = id % p.nseg;
    const int tseg = seg * p.L;
    const int te = min(p.T, tseg + p.L);
    float2 d[EP];
    int tb;
    if (seg == 0) {
        if (p.d0) {
            ld_pairs<EP>(p.d0 + (size_t)seq * K + E * lane, d);
        } else {
#pragma unroll
            for (int e = 0; e < EP; ++e) d[e] = make_float2(1.0f, 1.0f);
        }
        tb = 0;
    } else {
#pragma unroll
        for (int e = 0; e < EP; ++e) d[e] = make_float2(0.0f, 0.0f);   // the warm-up forgets this
        tb = tseg - (HAS_R ? warm_tokens<io_t>(p, seq, tseg, lane) : Spec<io_t>::warm);
    }
    bool expand = false;
    float lr = 0.0f;   // warm-up tokens (< tseg) add nothing
    if (seg > 0) warp_scan<io_t, K, HAS_R, LR>(p, st, seq, tb, tseg, tseg, d, expand, lr);
    const size_t slot = (size_t)seq * p.nseg + seg;
    if (p.nseg > 1) st_pairs<EP>(p.ws_start + slot * K + E * lane, d);
    warp_scan<io_t, K, HAS_R, LR>(p, st, seq, tseg, tseg, te, d, expand, lr);
    expand = __any_sync(kFullMask, expand);
    if (LR) lr = warp_sum(lr);
    if (p.nseg > 1) {
        st_pairs<EP>(p.ws_end + slot * K + E * lane, d);
        if (lane == 0) p.ws_flag[slot] = expand ? 1 : 0;
        if (LR && lane == 0) p.ws_lr[slot] = lr;
    } else {
        if (p.dT) st_pairs<EP>(p.dT + (size_t)seq * K + E * lane, d);
        if (LR && lane == 0) p.logratio[seq] = lr;
    }
}

// Largest |a_i - b_i| and |b_i| over a K-vector held as this lane's pairs.
template <int EP>
__device__ __forceinline__ void warp_diff(const float2 (&a)[EP], const float2 (&b)[EP], float &diff,
                                          float &mag) {
    diff = 0.f;
    mag = 0.f;
#pragma unroll
    for (int e = 0; e < EP; ++e) {
        diff = fmaxf(diff, fmaxf(fabsf(a[e].x - b[e].x), fabsf(a[e].y - b[e].y)));
        mag = fmaxf(mag, fmaxf(fabsf(b[e].x), fabsf(b[e].y)));
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        diff = fmaxf(diff, __shfl_xor_sync(kFullMask, diff, m));
        mag = fmaxf(mag, __shfl_xor_sync(kFullMask, mag, m));
    }
}

// Grid (BH), kMaxWarps warps: verify every speculative segment start against
// its predecessor's end; recompute (exactly) the segments that do not match;
// write d_T.  Without a repair every boundary check is independent (the
// predecessor's end is then exact), so the warps check all boundaries at
// once; warp 0 then walks sequentially from the first one that fails.
template <typename io_t, int K, bool HAS_R, bool LR>
__global__ void __launch_bounds__(32 * kMaxWarps) precond_verify_kernel(Params p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    constexpr int EP = K / 64, E = 2 * EP;
    WarpSmem<io_t, K> &st = *reinterpret_cast<WarpSmem<io_t, K> *>(smem_raw);
    const int seq = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const size_t base = (size_t)seq * p.nseg;
    __shared__ int first_bad;
    int f = 0;
    for (int i = threadIdx.x; i < p.nseg; i += blockDim.x) f |= p.ws_flag[base + i];
    const bool all_suspect = __syncthreads_or(f) != 0;
    if (threadIdx.x == 0) first_bad = all_suspect ? 1 : p.nseg;
    __syncthreads();
    if (!all_suspect) {
        // kB boundaries per warp and pass, all loads in flight before the checks
        constexpr int kB = 8;
        for (int b0 = 1 + warp * kB; b0 < p.nseg; b0 += nw * kB) {
            float2 prev[kB][EP], cur[kB][EP];
#pragma unroll
            for (int m = 0; m < kB; ++m) {
                const int i = min(b0 + m, p.nseg - 1);   // past the end: a repeat of the last
                ld_pairs<EP>(p.ws_end + (base + i - 1) * K + E * lane, prev[m]);
                ld_pairs<EP>(p.ws_start + (base + i) * K + E * lane, cur[m]);
            }
#pragma unroll
            for (int m = 0; m < kB; ++m) {
                float diff, mag;
                warp_diff<EP>(prev[m], cur[m], diff, mag);
                if (lane == 0 && b0 + m < p.nseg && !(diff <= Spec<io_t>::tol * mag))
                    atomicMin(&first_bad, b0 + m);
            }
        }
    }
    __syncthreads();
    if (warp != 0) return;   // the walk below is warp 0's alone
    const int start = first_bad;
    float2 prev_end[EP];
    ld_pairs<EP>(p.ws_end + (base + start - 1) * K + E * lane, prev_end);
    for (int i = start; i < p.nseg; ++i) {
        float2 cur[EP];
        ld_pairs<EP>(p.ws_start + (base + i) * K + E * lane, cur);
        float diff, mag;
        warp_diff<EP>(prev_end, cur, diff, mag);
        const bool ok = !all_suspect && diff <= Spec<io_t>::tol * mag;
        float2 dd[EP];
        if (ok) {
            ld_pairs<EP>(p.ws_end + (base + i) * K + E * lane, dd);
        } else {   // recompute segment i from the exact end of segment i-1
#pragma unroll
            for (int e = 0; e < EP; ++e) dd[e] = prev_end[e];
            const int tseg = i * p.L, te = min(p.T, tseg + p.L);
            bool unused = false;
            float lr = 0.0f;
            warp_scan<io_t, K, HAS_R, LR>(p, st, seq, tseg, tseg, te, dd, unused, lr);
            st_pairs<EP>(p.ws_end + (base + i) * K + E * lane, dd);
            if (LR) {
                lr = warp_sum(lr);
                if (lane == 0) p.ws_lr[base + i] = lr;
            }
        }
#pragma unroll
        for (int e = 0; e < EP; ++e) prev_end[e] = dd[e];
    }
    if (p.dT) st_pairs<EP>(p.dT + (size_t)seq * K + E * lane, prev_end);
    if (LR) {   // the segments' sums, in segment order within each lane
        __syncwarp();
        float lr = 0.0f;
        for (int i = lane; i < p.nseg; i += 32) lr += p.ws_lr[base + i];
        lr = warp_sum(lr);
        if (lane == 0) p.logratio[seq] = lr;
    }
}

// T == 0: the final preconditioner is the initial one.
__global__ void copy_or_fill_kernel(size_t n, const float *__restrict__ src, float fill,
                                    float *__restrict__ dst) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src ? src[i] : fill;
}

// Streaming multiprocessors of the current device (the segment count and
// the CTA shape are sized for one wave); the GB300 count when there is none.
static int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
        cudaGetLastError();   // clear the error a device-less query leaves behind
        return kDefaultSms;
    }
    return n;
}

template <typename io_t, int K, bool HAS_R, bool LR>
static cudaError_t launch_t(const Params &p, cudaStream_t stream) {
    constexpr int kStage = (int)sizeof(WarpSmem<io_t, K>);
    static std::atomic<unsigned long long> attr_seg{0}, attr_ver{0}, attr_cta{0}, attr_chk{0};
    if (p.nseg == 1 && p.BH <= 2 * sm_count()) {
        // one segment a sequence and few sequences: a CTA per sequence
        constexpr int kCta = (int)sizeof(CtaSmem<io_t, K>);
        if constexpr (!LR) {
            if (p.ecoef || p.dchk) {   // checkpoint mode (never with the residual sums)
                cudaError_t e = smem_attr_once(
                    (const void *)precond_cta_kernel<io_t, K, HAS_R, false, true>, kCta, attr_chk);
                if (e != cudaSuccess) return e;
                precond_cta_kernel<io_t, K, HAS_R, false, true>
                    <<<p.BH, 32 * (K / 32 + kSolvers), kCta, stream>>>(p);
                return cudaGetLastError();
            }
        }
        cudaError_t e = smem_attr_once((const void *)precond_cta_kernel<io_t, K, HAS_R, LR, false>,
                                       kCta, attr_cta);
        if (e != cudaSuccess) return e;
        precond_cta_kernel<io_t, K, HAS_R, LR, false><<<p.BH, 32 * (K / 32 + kSolvers), kCta, stream>>>(p);
        return cudaGetLastError();
    }
    cudaError_t e0 = smem_attr_once((const void *)precond_segment_kernel<io_t, K, HAS_R, LR>,
                                    kMaxWarps * kStage, attr_seg);
    if (e0 == cudaSuccess)
        e0 = smem_attr_once((const void *)precond_verify_kernel<io_t, K, HAS_R, LR>, kStage, attr_ver);
    if (e0 != cudaSuccess) return e0;
    // few segments: one per CTA, so that they spread over the SMs
    const long long nwarps = (long long)p.BH * p.nseg;
    const int wpc = nwarps >= 2LL * sm_count() ? kMaxWarps : 1;
    const unsigned grid = (unsigned)((nwarps + wpc - 1) / wpc);
    precond_segment_kernel<io_t, K, HAS_R, LR><<<grid, 32 * wpc, wpc * kStage, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.nseg == 1) return e;
    precond_verify_kernel<io_t, K, HAS_R, LR><<<p.BH, 32 * kMaxWarps, kStage, stream>>>(p);
    return cudaGetLastError();
}

template <typename io_t, int K>
static cudaError_t launch(const Params &p, cudaStream_t stream) {
    if (p.logratio)
        return p.r ? launch_t<io_t, K, true, true>(p, stream) : launch_t<io_t, K, false, true>(p, stream);
    return p.r ? launch_t<io_t, K, true, false>(p, stream) : launch_t<io_t, K, false, false>(p, stream);
}

}  // namespace p1

// Segment length: each segment is one warp, and about 8 of them are resident
// per SM (two CTAs of four), so segments are halved from 1024 tokens while
// all of them still fit in that one wave: more warps hide more latency, a
// second wave costs a whole segment time, and below 256 tokens the 128-token
// warm-up would double the work.  Only a retention gate (r != NULL) makes the
// warm-up converge, so without one there is a single segment per sequence.
int precond_segments(int BH, int T, bool has_r, int *L_out) {
    // ceil(a / b) in 64 bits: T may be within a segment of INT_MAX
    auto cdiv = [](long long a, long long b) { return (a + b - 1) / b; };
    int L = T;
    if (has_r && T > p1::kMinSeg) {
        L = 1024;
        const long long sms = p1::sm_count();
        while (L > p1::kMinSeg && (long long)BH * cdiv(T, L / 2) <= 8LL * sms)
            L >>= 1;
        if (L >= T) L = T;
    }
    if (L < 1) L = 1;
    if (L_out) *L_out = L;
    return (int)cdiv(T, L);
}

// Scratch of the segmented scan: segment starts and ends [n][K] fp32, then
// the flags [n] int and the residual sums [n] fp32, each padded to 256 bytes
// (n = BH * nseg).
static size_t segment_scratch_bytes(size_t n, int K) {
    return n * K * 4 * 2 + 2 * (((n * 4 + 255) / 256) * 256);
}

size_t precond_scratch_bytes(int BH, int T, int K) {
    int L;
    const int nseg = precond_segments(BH, T, true, &L);
    if (nseg <= 1) return 0;
    return segment_scratch_bytes((size_t)BH * nseg, K);
}

static cudaError_t scan_launch(int io, int BH, int T, int K, const void *k, const float *beta,
                               const float *r, float eta, const float *d0, void *ktilde,
                               float *dT, float *logratio, float *ecoef, float *dchk,
                               int chk_shift, void *scratch, int *status, cudaStream_t stream) {
    if (T == 0) {   // d_T = d_0; an empty product of residual ratios is 1
        if (logratio) {
            p1::copy_or_fill_kernel<<<(unsigned)((BH + 255) / 256), 256, 0, stream>>>(
                (size_t)BH, nullptr, 0.0f, logratio);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        if (!dT) return cudaSuccess;
        size_t n = (size_t)BH * K;
        p1::copy_or_fill_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(n, d0, 1.0f, dT);
        return cudaGetLastError();
    }
    p1::Params p;
    p.BH = BH;
    p.T = T;
    p.nseg = precond_segments(BH, T, r != nullptr, &p.L);
    p.k = k;
    p.beta = beta;
    p.r = r;
    p.d0 = d0;
    p.eta = eta;
    p.ktilde = ktilde;
    p.dT = dT;
    p.ecoef = ecoef;
    p.dchk = dchk;
    p.chk_shift = chk_shift;
    p.logratio = logratio;
    p.status = status;
    float *f = static_cast<float *>(scratch);
    const size_t n = (size_t)BH * p.nseg;
    const size_t pad = ((n * 4 + 255) / 256) * 256 / 4;   // floats per padded [n] array
    p.ws_start = p.nseg > 1 ? f : nullptr;
    p.ws_end = p.nseg > 1 ? f + n * K : nullptr;
    p.ws_flag = p.nseg > 1 ? reinterpret_cast<int *>(f + 2 * n * K) : nullptr;
    p.ws_lr = p.nseg > 1 ? f + 2 * n * K + pad : nullptr;
    if (io == OSDN_BF16)
        return K == 64 ? p1::launch<__nv_bfloat16, 64>(p, stream)
                       : p1::launch<__nv_bfloat16, 128>(p, stream);
    return K == 64 ? p1::launch<float, 64>(p, stream) : p1::launch<float, 128>(p, stream);
}

cudaError_t precond_scan_launch(int io, int BH, int T, int K, const void *k, const float *beta,
                                const float *r, float eta, const float *d0, void *ktilde,
                                float *dT, float *logratio, void *scratch, int *status,
                                cudaStream_t stream) {
    return scan_launch(io, BH, T, K, k, beta, r, eta, d0, ktilde, dT, logratio, nullptr, nullptr,
                       6, scratch, status, stream);
}

// Checkpoint mode: e_t of every token ([BH][T]) and d entering every
// interval of 2^chk_shift tokens ([BH][ceil(T / 2^chk_shift)][K]) instead of
// ktilde (either may be NULL); d_T as usual.
cudaError_t precond_checkpoint_launch(int io, int BH, int T, int K, const void *k,
                                      const float *beta, const float *r, float eta,
                                      const float *d0, float *dT, float *ecoef, float *dchk,
                                      int chk_shift, void *scratch, int *status,
                                      cudaStream_t stream) {
    return scan_launch(io, BH, T, K, k, beta, r, eta, d0, nullptr, dT, nullptr, ecoef, dchk,
                       chk_shift, scratch, status, stream);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the scan, for callers that may not allocate
// device memory.  Its scratch (the speculative segment starts and ends) lives
// in this file-scope device array instead of a caller workspace.  The array
// exists on every GPU that loads the library until the process exits.  All
// calls share it and it keeps the last call's contents; the scan writes every
// entry it later reads, so nothing needs clearing between calls, but calls
// whose kernels overlap on the GPU (different streams, no ordering) race on it.
constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

size_t precond_noalloc_capacity() { return kNoAllocScratchBytes; }

// Device address of the scratch array on the current device.  Resolved once
// per device (with that device current) on the first call there; host code
// must not pass the array's name itself to a kernel.
static cudaError_t noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

cudaError_t precond_scan_noalloc_launch(int io, int BH, int T, int K, const void *k,
                                        const float *beta, const float *r, float eta,
                                        const float *d0, void *ktilde, float *dT,
                                        cudaStream_t stream) {
    void *scratch = nullptr;
    cudaError_t e = noalloc_scratch(&scratch);
    if (e != cudaSuccess) return e;
    return precond_scan_launch(io, BH, T, K, k, beta, r, eta, d0, ktilde, dT, nullptr, scratch,
                               nullptr, stream);
}

// Bytes of scratch the scan needs for this call (0 without a retention gate).
size_t precond_scratch_bytes_for(int BH, int T, int K, bool has_r) {
    int L;
    const int nseg = precond_segments(BH, T, has_r, &L);
    if (nseg <= 1 || T == 0) return 0;
    return segment_scratch_bytes((size_t)BH * nseg, K);
}

cudaError_t fill_state_launch(size_t n, const float *src, float fill, float *dst,
                              cudaStream_t stream) {
    if (n == 0 || !dst) return cudaSuccess;
    unsigned blocks = (unsigned)((n + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    p1::copy_or_fill_kernel<<<blocks, 256, 0, stream>>>(n, src, fill, dst);
    return cudaGetLastError();
}

}  // namespace osdn
