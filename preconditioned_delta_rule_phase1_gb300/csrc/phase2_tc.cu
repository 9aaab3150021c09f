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
//   L  = tril(diag(b) (G . K Kt^T), -1),   X = (I + L)^-1,   Xb = X diag(b)
//   U  = Xb V - Xb diag(g) K S^T                    (the chunk's scaled residuals)
//   O  = diag(g) Q S^T + tril(G . Q Kt^T) U
//   S' = g_C S + U^T diag(g_C / g) Kt
//
// One CTA per (sequence, 64-row slice of S), 448 threads in four roles that
// run concurrently and hand work over through mbarriers:
//   warp 0      TMA producer: Q/Kt tiles (3-deep ring) and K/V tiles (2-deep
//               ring), plus the chunk's gates (beta, cumulative log alpha);
//   warp 1      MMA issuer (one thread): every tcgen05.mma and commit;
//   warps 2-9   "prep", one chunk ahead of the chain: Gram and scores out of
//               TMEM, L and the masked scores A, the diagonal gate scalings of
//               Q, K and Kt in place, X = (I + L)^-1 (16x16 diagonal blocks in
//               fp32, off-diagonal blocks with mma.sync tf32), Xb, and
//               Kw^T = (Xb diag(g) K)^T back to shared memory;
//   warps 10-13 "chain": U, the state S (fp32 accumulator in TMEM, bf16 copy
//               in shared memory for the MMAs) and the output O.
// Tensor-core products (bf16 operands, fp32 accumulation in TMEM):
//   prep : K Kt^T, Q Kt^T (M=64, N=64);  K^T Xb^T -> Kw^T (M=K);  V^T Xb^T -> U^T init
//   chain: U^T -= S Kw^T;  O^T = S Q^T;  S += U^T Kt;  O^T += U^T A^T   (M=64)
// Every wait is bounded: a wait that runs out records OSDN_ERR_TIMEOUT in the
// status word and all roles leave their loops.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "osdn_device.cuh"
#include "ptx.cuh"

namespace osdn {
namespace tc {

constexpr int C = 64;     // tokens per chunk
constexpr int BV = 64;    // rows of S per CTA
constexpr int NS = 2;     // depth of the input ring (one slot per chunk)
constexpr int kThreads = 448;
constexpr int kPrepThreads = 256;
constexpr int kChainThreads = 128;
constexpr int kLP = 68;   // fp32 pitch of the solver tile
constexpr uint32_t kWaitLimit = 1u << 15;      // sleeping polls before a wait gives up
constexpr uint32_t kSleepNs = 1u << 16;         // longest sleep per poll (~65 us)

// TMEM columns
constexpr uint32_t kColG = 0;      // [K;Q] Kt^T (M=128): Gram rows 0-63, score rows 64-127
constexpr uint32_t kColKw = 64;    // Kw^T (M=K)
constexpr uint32_t kColU = 128;    // U^T, two buffers of 64 (M=64)
constexpr uint32_t kColO = 256;    // O^T, two buffers of 64 (M=64)
constexpr uint32_t kColS = 384;    // S (M=64, K columns)
constexpr uint32_t kTmemCols = 512;

// Input slot: [K;Q] stacked in 128-row blocks of 64 columns (K rows 0-63,
// Q rows 64-127), then Kt (64-row blocks), then the value slice.
template <int K>
struct Lay {
    static constexpr int kKQ = 128 * K * 2;
    static constexpr int kKt = C * K * 2;
    static constexpr int kV = C * BV * 2;
    static constexpr int kSlot = kKQ + kKt + kV;
    static constexpr int oKt = kKQ;                   // within a slot
    static constexpr int oVv = kKQ + kKt;
    static constexpr int oL = NS * kSlot;             // fp32 64 x kLP
    static constexpr int oA = oL + C * kLP * 4;       // bf16 64 x 64, two buffers
    static constexpr int oKw = oA + 2 * C * C * 2;    // bf16 K rows x 64
    static constexpr int oXb = oKw + K * 128;         // bf16 64 x 64
    static constexpr int oS = oXb + C * C * 2;        // bf16 BV x K
    static constexpr int oU = oS + BV * K * 2;        // bf16 BV x 64 (also O staging)
    static constexpr int kBytes = oU + BV * C * 2;
    static constexpr int kAlloc = kBytes + 1024;
};

struct Params {
    int T, V, nchunks;
    const float *beta, *alpha, *S0;
    __nv_bfloat16 *o;
    float *ST;
    int *status;
};

struct Bars {
    uint64_t full[NS], empty[NS];
    uint64_t g_full, x1, x2, kw_full, x3, u_full, u_sm, s_full, s_ready;
    uint64_t a_free[2], o_free[2];
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// n (multiple of 8) consecutive bf16 of row r, columns [c0, c0+n) within one
// 64-column block, into a 128B-swizzled tile whose blocks hold `rows` rows.
__device__ __forceinline__ void st_row_sw128(uint8_t *tile, int rows, int r, int c0,
                                             const float *vals, int n) {
    uint8_t *rowp = tile + (c0 >> 6) * rows * 128 + r * 128;
    const int cb = (c0 & 63) >> 3;
#pragma unroll
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

// Descriptors are built once per operand (dk0 / dmn0) and advanced per
// k-slice by adding the byte offset in 16-byte units to the start-address
// field (all tiles sit below 256 KB, so the 14-bit field never carries).
__device__ __forceinline__ uint64_t dk0(uint32_t base) { return ptx::sdesc(base, 16, 1024, 2); }
__device__ __forceinline__ uint64_t dmn0(uint32_t base, int block_bytes) {
    return ptx::sdesc(base, block_bytes, 1024, 2);
}
// k-slice ks of a K-major tile whose 64-column blocks hold `rows` rows
__host__ __device__ constexpr uint64_t koff(int rows, int ks) {
    return static_cast<uint64_t>(((ks >> 2) * rows * 128 + (ks & 3) * 32) >> 4);
}
// k-slice ks (16 rows) of an MN-major tile
__host__ __device__ constexpr uint64_t mnoff(int ks) { return static_cast<uint64_t>((ks * 2048) >> 4); }

// Barrier over `count` threads of barrier `id` that also ANDs a predicate:
// every participant gets the same answer, so a role leaves its loop together.
__device__ __forceinline__ bool vote_all(bool v, int id, int count) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(out)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(count)
        : "memory");
    return out != 0;
}

// Bounded wait that also gives up as soon as another thread has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         int *status) {
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        if (ptx::mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
        if (*abort_flag) return false;
    }
    report_status(status, OSDN_ERR_TIMEOUT);
    *abort_flag = 1;
    return false;
}

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
// scratch).  Recursive doubling: 4x4 diagonal blocks in closed form, then
// X21 = -X22 L21 X11 on 8x8 and 16x16 blocks in fp32 SIMT, and on 32x32 and
// 64x64 with mma.sync (tf32 inputs, fp32 accumulation).  sP: 256 floats of
// scratch.  Called by the 256 prep threads.
__device__ void solve_unit_lower(float *sL, float *sP, int pt) {
    const int pw = pt >> 5, lane = pt & 31;
    if (pt < 64) {  // 16x16 diagonal blocks: lane (blk, c) forms column c
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

// Scale rows of a 64-row bf16 tile (K/64 blocks of 8 KB) in place: row t by f[t].
template <int K>
__device__ __forceinline__ void scale_rows(uint8_t *tile, const float *f, int pt) {
    constexpr int PIECES = C * K * 2 / 16;   // 16-byte pieces
    for (int i = pt; i < PIECES; i += kPrepThreads) {
        const int row = (i >> 3) & 63;        // 8 pieces per 128-byte row
        uint4 *p = reinterpret_cast<uint4 *>(tile + i * 16);
        uint4 u = *p;
        const float s = f[row];
        uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float2 x = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&w[e]));
            w[e] = pack_bf16x2(x.x * s, x.y * s);
        }
        *p = u;
    }
}

template <int K, bool GATED>
__global__ void __launch_bounds__(kThreads, 1)
delta_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_v,
                Params p) {
    using LY = Lay<K>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned start, by pointer arithmetic so accesses stay in the
    // shared state space (an integer round trip would make them generic)
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ Bars bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ float sBeta[NS][C], sLg[NS][C];
    __shared__ float sScale[2][C];        // prep: g_t, g_C / g_t of the chunk being scaled
    __shared__ float sP[256];             // solver scratch
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3;
    const int seq = blockIdx.y, v0 = blockIdx.x * BV;
    const int T = p.T, nch = p.nchunks;
    float *sL = reinterpret_cast<float *>(smem + LY::oL);
    uint8_t *sKw = smem + LY::oKw, *sXb = smem + LY::oXb;
    uint8_t *sS = smem + LY::oS, *sU = smem + LY::oU;
    auto slot = [&](int j) { return smem + (j % NS) * LY::kSlot; };
    auto tA = [&](int j) { return smem + LY::oA + (j & 1) * C * C * 2; };

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            ptx::mbar_init(&bars.full[i], 1);
            ptx::mbar_init(&bars.empty[i], 1);
        }
        uint64_t *one[] = {&bars.g_full, &bars.x1, &bars.x2, &bars.kw_full, &bars.x3,
                           &bars.u_full, &bars.u_sm, &bars.s_full, &bars.s_ready,
                           &bars.a_free[0], &bars.a_free[1], &bars.o_free[0], &bars.o_free[1]};
        for (uint64_t *b : one) ptx::mbar_init(b, 1);
        ptx::fence_mbar_init();
        s_abort = 0;
    }
    if (warp == 1) {
        ptx::tmem_alloc(&tmem_base_sh, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    int *st = p.status;

    if (warp == 0) {
        // ======================================================== producer
        int last = -1;
        for (int j = 0; j < nch; ++j) {
            const int sl = j % NS, t0 = j * C;
            // gates: beta (0 past T) and the inclusive cumulative log alpha,
            // fetched before waiting for the slot so the load latency overlaps
            float bb[2], lg[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = t0 + 2 * lane + e;
                const bool valid = t < T;
                bb[e] = valid ? p.beta[(size_t)seq * T + t] : 0.0f;
                lg[e] = (GATED && valid) ? logf(p.alpha[(size_t)seq * T + t]) : 0.0f;
            }
            if (j >= NS &&
                !__all_sync(kFullMask, wait_bar(&bars.empty[sl], ((j / NS) - 1) & 1, &s_abort, st)))
                break;
            float sc = lg[0] + lg[1];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(kFullMask, sc, off);
                if (lane >= off) sc += y;
            }
            const float excl = sc - (lg[0] + lg[1]);
            sBeta[sl][2 * lane] = bb[0];
            sBeta[sl][2 * lane + 1] = bb[1];
            sLg[sl][2 * lane] = excl + lg[0];
            sLg[sl][2 * lane + 1] = excl + lg[0] + lg[1];
            __syncwarp();
            if (lane == 0) {
                uint8_t *sb = slot(j);
                ptx::mbar_arrive_expect_tx(&bars.full[sl], LY::kSlot);
#pragma unroll
                for (int cb = 0; cb < K / 64; ++cb) {
                    ptx::tma_load_3d(sb + cb * 16384, &tm_k, &bars.full[sl], cb * 64, t0, seq);
                    ptx::tma_load_3d(sb + cb * 16384 + 8192, &tm_q, &bars.full[sl], cb * 64, t0, seq);
                    ptx::tma_load_3d(sb + LY::oKt + cb * 8192, &tm_kt, &bars.full[sl], cb * 64, t0, seq);
                }
                ptx::tma_load_3d(sb + LY::oVv, &tm_v, &bars.full[sl], v0, t0, seq);
            }
            last = j;
        }
        // bulk copies still in flight (only after an abort) must land before exit
        if (lane == 0 && s_abort) {
            for (int j = (last > NS - 1 ? last - NS + 1 : 0); j <= last; ++j)
                for (uint32_t i = 0; i < kWaitLimit; ++i)
                    if (ptx::mbar_try_wait_sleep(&bars.full[j % NS], (j / NS) & 1, kSleepNs)) break;
        }
    } else if (warp == 1) {
        // ======================================================== MMA issuer
        if (lane == 0) {
            const uint32_t aXb = ptx::smem_u32(sXb), aKw = ptx::smem_u32(sKw);
            const uint32_t aS = ptx::smem_u32(sS), aU = ptx::smem_u32(sU);
            auto gram = [&](int j) {  // [K;Q] Kt^T of chunk j into G
                const uint32_t aKQ = ptx::smem_u32(slot(j)), aKt = aKQ + LY::oKt;
                const uint32_t id = ptx::idesc_bf16(128, 64, 0, 0);
                const uint64_t da = dk0(aKQ), db = dk0(aKt);
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks)
                    ptx::umma_bf16(tmem + kColG, da + koff(128, ks), db + koff(C, ks), id, ks > 0);
                ptx::umma_commit(&bars.g_full);
            };
            bool ok = wait_bar(&bars.full[0], 0, &s_abort, st);
            if (ok) {
                ptx::tc_fence_after();
                gram(0);
            }
            for (int j = 0; ok && j <= nch; ++j) {
                // Order per iteration: chain of chunk j-1 (frees the slot chunk j+1
                // is loaded into), Kw/V' of chunk j, then Gram of chunk j+1.
                if (j >= 1) {  // chain of chunk c = j - 1
                    const int c = j - 1;
                    if (!wait_bar(&bars.x3, c & 1, &s_abort, st)) break;
                    if (!wait_bar(&bars.s_ready, c & 1, &s_abort, st)) break;
                    if (c >= 2 && !wait_bar(&bars.o_free[c & 1], ((c >> 1) + 1) & 1, &s_abort, st)) break;
                    ptx::tc_fence_after();
                    const uint32_t aKQ = ptx::smem_u32(slot(c)), aKt = aKQ + LY::oKt;
                    const uint32_t aA = ptx::smem_u32(tA(c));
                    const uint32_t dU = tmem + kColU + 64 * (c & 1), dO = tmem + kColO + 64 * (c & 1);
                    const uint32_t idu = ptx::idesc_bf16(64, 64, 0, 1, 1), ido = ptx::idesc_bf16(64, 64, 0, 0);
                    const uint64_t dS = dk0(aS), dKw = dmn0(aKw, 8192), dQ = dk0(aKQ + 8192);
#pragma unroll
                    for (int ks = 0; ks < K / 16; ++ks) {  // U^T -= S Kw^T, O^T = S Q^T
                        ptx::umma_bf16(dU, dS + koff(BV, ks), dKw + mnoff(ks), idu, 1);
                        ptx::umma_bf16(dO, dS + koff(BV, ks), dQ + koff(128, ks), ido, ks > 0);
                    }
                    ptx::umma_commit(&bars.u_full);
                    if (!wait_bar(&bars.u_sm, c & 1, &s_abort, st)) break;
                    ptx::tc_fence_after();
                    const uint32_t ids = ptx::idesc_bf16(64, K, 0, 1), ida = ptx::idesc_bf16(64, 64, 0, 0);
                    const uint64_t dUa = dk0(aU), dKt = dmn0(aKt, 8192), dA = dk0(aA);
#pragma unroll
                    for (int ks = 0; ks < C / 16; ++ks) {  // S += U^T Kt, O^T += U^T A^T
                        ptx::umma_bf16(tmem + kColS, dUa + koff(BV, ks), dKt + mnoff(ks), ids, 1);
                        ptx::umma_bf16(dO, dUa + koff(BV, ks), dA + koff(C, ks), ida, 1);
                    }
                    ptx::umma_commit(&bars.s_full);
                    ptx::umma_commit(&bars.a_free[c & 1]);
                    ptx::umma_commit(&bars.empty[c % NS]);
                }
                if (j < nch) {  // Kw^T = K^T Xb^T (K scaled by g) and U^T = V^T Xb^T of chunk j
                    if (!wait_bar(&bars.x2, j & 1, &s_abort, st)) break;
                    ptx::tc_fence_after();
                    const uint32_t aKQ = ptx::smem_u32(slot(j)), aV = aKQ + LY::oVv;
                    const uint32_t idk = ptx::idesc_bf16(K, 64, 1, 0), idv = ptx::idesc_bf16(64, 64, 1, 0);
                    const uint32_t dU = tmem + kColU + 64 * (j & 1);
                    const uint64_t dK = dmn0(aKQ, 16384), dV = dmn0(aV, 8192), dX = dk0(aXb);
#pragma unroll
                    for (int ks = 0; ks < C / 16; ++ks) {
                        ptx::umma_bf16(tmem + kColKw, dK + mnoff(ks), dX + koff(C, ks), idk, ks > 0);
                        ptx::umma_bf16(dU, dV + mnoff(ks), dX + koff(C, ks), idv, ks > 0);
                    }
                    ptx::umma_commit(&bars.kw_full);
                }
                if (j + 1 < nch) {  // Gram of the next chunk: slot loaded, G read by prep
                    if (!wait_bar(&bars.full[(j + 1) % NS], ((j + 1) / NS) & 1, &s_abort, st)) break;
                    if (!wait_bar(&bars.x1, j & 1, &s_abort, st)) break;
                    ptx::tc_fence_after();
                    gram(j + 1);
                }
            }
        }
        __syncwarp();
    } else if (warp < 10) {
        // ======================================================== prep
        const int pt = tid - 64, pw = warp - 2, half = pw >> 2;
        const int grow = 32 * q4 + lane;       // row of the M=128 Gram/score accumulator
        // G epilogue of chunk j: L (fp32) into sL, masked scores A into tA(j),
        // the gate scalings of chunk j into sScale; ends by releasing G.
        auto g_epilogue = [&](int j) -> bool {
            const int sl = j % NS;
            bool ok = wait_bar(&bars.full[sl], (j / NS) & 1, &s_abort, st) &&
                      wait_bar(&bars.g_full, j & 1, &s_abort, st) &&
                      (j < 2 || wait_bar(&bars.a_free[j & 1], ((j >> 1) + 1) & 1, &s_abort, st));
            if (!vote_all(ok, 1, kPrepThreads)) return false;
            ptx::tc_fence_after();
            float g[32];
            tmem_ld32(tmem + lane_off + kColG + 32 * half, g);
            if (grow < C) {  // L = tril(diag(beta) (G . K Kt^T), -1)
                const int i = grow;
                const float bi = sBeta[sl][i], lgi = sLg[sl][i];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int col = 32 * half + jj;
                    float val = 0.0f;
                    if (col < i) val = bi * (GATED ? __expf(lgi - sLg[sl][col]) : 1.0f) * g[jj];
                    sL[i * kLP + col] = val;
                }
            } else {  // A = tril(G . Q Kt^T)
                const int t = grow - C;
                const float lgt = sLg[sl][t];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int col = 32 * half + jj;
                    g[jj] = (col <= t) ? (GATED ? __expf(lgt - sLg[sl][col]) : 1.0f) * g[jj] : 0.0f;
                }
                st_row_sw128(tA(j), C, t, 32 * half, g, 32);
            }
            if (GATED && pt < C) {
                const float lgC = sLg[sl][C - 1], lgt = sLg[sl][pt];
                sScale[0][pt] = __expf(lgt);
                sScale[1][pt] = __expf(lgC - lgt);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_bar(1, kPrepThreads);
            if (pt == 0) ptx::mbar_arrive(&bars.x1);
            return true;
        };
        bool ok = true;
        for (int j = 0; ok && j < nch; ++j) {
            const int sl = j % NS;
            if (!g_epilogue(j)) break;
            if (GATED) {  // [K;Q] <- diag(g) [K;Q], Kt <- diag(g_C / g) Kt (in place)
                scale_rows<2 * K>(slot(j), sScale[0], pt);
                scale_rows<K>(slot(j) + LY::oKt, sScale[1], pt);
            }
            solve_unit_lower(sL, sP, pt);
            {  // Xb = X diag(beta): row t, columns s <= t (bf16 B operand)
                const int t = pt >> 2, s0 = 16 * (pt & 3);
                float xb[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int s = s0 + e;
                    xb[e] = (s <= t) ? sL[t * kLP + s] * sBeta[sl][s] : 0.0f;
                }
                st_row_sw128(sXb, C, t, s0, xb, 16);
            }
            ptx::fence_proxy_async_smem();
            ptx::named_bar(1, kPrepThreads);
            if (pt == 0) ptx::mbar_arrive(&bars.x2);
            // Kw^T out of TMEM into the MN-major B operand of the chain
            ok = wait_bar(&bars.kw_full, j & 1, &s_abort, st) &&
                 (j < 1 || wait_bar(&bars.u_full, (j - 1) & 1, &s_abort, st));
            if (!vote_all(ok, 1, kPrepThreads)) break;
            ptx::tc_fence_after();
            {
                float kw[32];
                tmem_ld32(tmem + lane_off + kColKw + 32 * half, kw);
                const int krow = (K == 128) ? 32 * q4 + lane : 16 * q4 + lane;
                if (K == 128 || lane < 16) st_row_sw128(sKw, K, krow, 32 * half, kw, 32);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_bar(1, kPrepThreads);
            if (pt == 0) ptx::mbar_arrive(&bars.x3);
        }
    } else {
        // ======================================================== chain
        const int ct = tid - 320;
        const bool act = lane < 16;
        const int vrow = 16 * q4 + lane;
        // initial state: TMEM S = g_C(0) S0, bf16 copy = S0
        {
            float gC = 1.0f;
            const bool ok0 = !GATED || wait_bar(&bars.full[0], 0, &s_abort, st);
            if (vote_all(ok0, 2, kChainThreads) && GATED) gC = __expf(sLg[0][C - 1]);
#pragma unroll
            for (int c0 = 0; c0 < K; c0 += 32) {
                float sv[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    sv[e] = (act && p.S0) ? p.S0[((size_t)seq * p.V + v0 + vrow) * K + c0 + e] : 0.0f;
                if (act) st_row_sw128(sS, BV, vrow, c0, sv, 32);
                float lo[16], hi[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    lo[e] = gC * sv[e];
                    hi[e] = gC * sv[16 + e];
                }
                ptx::tmem_st16(tmem + lane_off + kColS + c0, lo);
                ptx::tmem_st16(tmem + lane_off + kColS + c0 + 16, hi);
            }
            ptx::tmem_wait_st();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_bar(2, kChainThreads);
            if (ct == 0) ptx::mbar_arrive(&bars.s_ready);
        }
        for (int c = 0; c < nch; ++c) {
            // ---- U^T to shared memory (A operand of the state and output MMAs)
            if (!vote_all(wait_bar(&bars.u_full, c & 1, &s_abort, st), 2, kChainThreads)) break;
            ptx::tc_fence_after();
            {
                float u[32], u2[32];
                tmem_ld32(tmem + lane_off + kColU + 64 * (c & 1), u);
                tmem_ld32(tmem + lane_off + kColU + 64 * (c & 1) + 32, u2);
                if (act) {
                    st_row_sw128(sU, BV, vrow, 0, u, 32);
                    st_row_sw128(sU, BV, vrow, 32, u2, 32);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_bar(2, kChainThreads);
            if (ct == 0) ptx::mbar_arrive(&bars.u_sm);
            // ---- state: bf16 copy for the next chunk, g_C(next) folded into TMEM
            bool okc = wait_bar(&bars.s_full, c & 1, &s_abort, st) &&
                       (!GATED || c + 1 >= nch ||
                        wait_bar(&bars.full[(c + 1) % NS], ((c + 1) / NS) & 1, &s_abort, st));
            if (!vote_all(okc, 2, kChainThreads)) break;
            ptx::tc_fence_after();
            const float gN = (GATED && c + 1 < nch) ? __expf(sLg[(c + 1) % NS][C - 1]) : 1.0f;
#pragma unroll
            for (int c0 = 0; c0 < K; c0 += 32) {
                float sv[32];
                tmem_ld32(tmem + lane_off + kColS + c0, sv);
                if (act) {
                    st_row_sw128(sS, BV, vrow, c0, sv, 32);
                    if (c == nch - 1 && p.ST) {
                        float *dst = p.ST + ((size_t)seq * p.V + v0 + vrow) * K + c0;
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4 *>(dst + e) = make_float4(sv[e], sv[e + 1], sv[e + 2], sv[e + 3]);
                    }
                }
                if (GATED) {
                    float lo[16], hi[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        lo[e] = gN * sv[e];
                        hi[e] = gN * sv[16 + e];
                    }
                    ptx::tmem_st16(tmem + lane_off + kColS + c0, lo);
                    ptx::tmem_st16(tmem + lane_off + kColS + c0 + 16, hi);
                }
            }
            if (GATED) ptx::tmem_wait_st();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_bar(2, kChainThreads);
            if (ct == 0) ptx::mbar_arrive(&bars.s_ready);
            // ---- output: O^T out of TMEM, staged [t][v] in the free U tile
            {
                float o1[32], o2[32];
                tmem_ld32(tmem + lane_off + kColO + 64 * (c & 1), o1);
                tmem_ld32(tmem + lane_off + kColO + 64 * (c & 1) + 32, o2);
                __nv_bfloat16 *sO = reinterpret_cast<__nv_bfloat16 *>(sU);
                if (act) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        sO[e * BV + vrow] = __float2bfloat16_rn(o1[e]);
                        sO[(32 + e) * BV + vrow] = __float2bfloat16_rn(o2[e]);
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::named_bar(2, kChainThreads);
            if (ct == 0) ptx::mbar_arrive(&bars.o_free[c & 1]);
            {
                const __nv_bfloat16 *sO = reinterpret_cast<const __nv_bfloat16 *>(sU);
                const int r = ct >> 3, part = ct & 7;   // 16 rows x 8 pieces per pass
#pragma unroll
                for (int rr = 0; rr < C; rr += 16) {
                    const int t = c * C + r + rr;
                    if (t < T)
                        *reinterpret_cast<uint4 *>(p.o + ((size_t)seq * T + t) * p.V + v0 + part * 8) =
                            *reinterpret_cast<const uint4 *>(sO + (r + rr) * BV + part * 8);
                }
            }
            // the next chunk's U epilogue overwrites this staging tile
            ptx::named_bar(2, kChainThreads);
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
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
    constexpr int smem = Lay<K>::kAlloc;
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
