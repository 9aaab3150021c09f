// phase2_tc.cu -- Phase 2 of OSDN on the sm_103a tensor cores (tcgen05 +
// TMEM + TMA): the chunkwise delta-rule pass with the stored keys replaced by
// the preconditioned keys Ktilde in the chunk Gram matrix and in the
// intra-chunk scores (gist.science summary of arXiv 2605.13473, section 2.1).
//
// Recurrence (per sequence):  S_t = a_t S_{t-1} + b_t (v_t - a_t S_{t-1} k_t) kt_t^T,
//                             o_t = S_t q_t        (a = alpha, b = beta, kt = ktilde)
//
// Two kernels.  chunk_prep_kernel (phase2_prep.cu) does, for every chunk of
// every sequence in parallel, all the work that does not involve the state:
// the Gram matrix, the unit-lower triangular inverse and the products that
// fold it into the per-chunk operands W, M, Qe, Ae.  The chain kernel here
// then runs the state recurrence, one chunk of C = 64 tokens after another:
//   S'^T = g_C S^T + [W | M] [V; S^T]           (the only product on the chain)
//   O    = [Ae | Qe] [V; S^T]                   (off the chain)
// with S^T kept as an fp32 accumulator in TMEM and as a bf16 copy in shared
// memory (the B operand of both products; three copies rotate, so the
// output product may still read one while the next is written).
//
// One CTA per (sequence, 64 columns of V), 480 threads in five roles:
//   warp 0      TMA producer: [W | M] and V (2-deep ring), [Ae | Qe] and V
//               (2-deep ring; V is loaded twice so that each ring stage is
//               released by one product);
//   warp 1      state MMA issuer (one thread): the chain's product only;
//   warp 2      output MMA issuer (one thread): a chunk's output product,
//               issued right behind its state product so that it never
//               delays the chain;
//   warps 3-6   O out of TMEM to global memory as bf16;
//   warps 7-14  the state: S^T out of TMEM, its bf16 copy, the decay g_C of
//               the next chunk, and the final state.
// The issuers and the state readout poll their barriers without sleeping:
// their waits sit on the chain's critical path.
// Every wait is bounded: a wait that runs out records OSDN_ERR_TIMEOUT in the
// status word and all roles leave their loops.
#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "tc_common.cuh"

namespace osdn {
namespace tc {

cudaError_t chunk_prep_launch(int BH, int T, int K, int c0, int c1, const void *q, const void *k,
                              const void *kt, const float *beta, const float *alpha,
                              const Fused &fz, __nv_bfloat16 *w, __nv_bfloat16 *m,
                              __nv_bfloat16 *qe, __nv_bfloat16 *ae, float *gc, int *status,
                              cudaStream_t stream);

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
        cudaGetLastError();
        return 152;
    }
    return n;
}

namespace {

constexpr int BV = 64;          // columns of V (rows of S) per CTA
constexpr int NS = 2;           // depth of both input rings
constexpr int NSB = 3;          // bf16 copies of the state
constexpr int kThreads = 480;
constexpr uint32_t kColS = 0;   // S^T (M=K), 64 columns
constexpr uint32_t kColO = 64;  // O (M=64), two buffers of 64 columns
constexpr uint32_t kTmemCols = 256;
constexpr float kSpecTol = 1.52587890625e-05f;   // 2^-16: a speculative start accepted this close

// Shared memory: ring X stages ([W | M] as K-row blocks of 64 columns, then
// V), ring Y stages ([Ae | Qe] as 64-row blocks of 64 columns, then V), and
// the bf16 copies of S^T (K rows of 64 values each).
template <int K>
struct Lay {
    static constexpr int oVx = (1 + K / 64) * K * 128;   // within a ring X stage
    static constexpr int oVy = (1 + K / 64) * C * 128;   // within a ring Y stage
    static constexpr int kX = oVx + C * 128;
    static constexpr int kY = oVy + C * 128;
    static constexpr int oX = 0;
    static constexpr int oY = NS * kX;
    static constexpr int oS = oY + NS * kY;
    static constexpr int kBytes = oS + NSB * K * 128;
    static constexpr int kAlloc = kBytes + 1024;
};

struct Params {
    int BH, T, V, nch, c0, ncs;   // sequences, length, V, its chunks; this launch: chunks [c0, c0 + ncs)
    int nz;                       // z-slices of the grid that hold sequences (segments: the rest)
    const float *S0, *gc;
    __nv_bfloat16 *o;
    float *ST;
    // Speculative time segments (seg_len > 0; grid z = segment): segment z
    // owns chunks [z L, (z+1) L); for z > 0 it starts from a zero state `warm`
    // chunks early, records the state it reaches at z L in seg_spec[z] and
    // writes O only from z L on.  Its end state goes to seg_end[z], the last
    // segment's to ST.
    int seg_len, warm, nseg;
    float *seg_spec, *seg_end;   // [nseg][BH][V][K]
    // Repair launch: when `check` is given, a CTA first compares its rows of
    // `check` (a speculative start) with S0 (the exact start) and leaves at
    // once if they agree to kSpecTol of S0's largest entry.
    const float *check;
    int *status;
    // Test word (the second word of the workspace header, status[1]): when it
    // is nonzero the producer issues nothing and the waits are shortened, so
    // that they run out and the kernel ends with OSDN_ERR_TIMEOUT.
};

// Barriers.  The bf16 state copy entering chunk c sits in buffer c % NSB:
// s_issued[b] completes when the state product reading it has been issued
// (so the copy is complete), o_read[b] when the output product reading it
// has completed (the buffer may then be overwritten).  s_tmem completes when
// every state warp has read the accumulator (and, gated, rescaled it): the
// part of the next state product that does not read S (W V) may then start,
// while the bf16 copy is still being written (s_ready).
struct Bars {
    uint64_t fullX[NS], emptyX[NS], fullY[NS], emptyY[NS];
    uint64_t s_full, s_ready, s_tmem, done_s, done_o;
    uint64_t s_issued[NSB], o_read[NSB];
    uint64_t o_full[2], o_free[2];
};

// GATED: a decay; PCH: the decay is per key channel (g_C is then a K-vector
// per chunk, and row k of S^T decays by its own entry).
template <int K, bool GATED, bool PCH>
__global__ void __launch_bounds__(kThreads, 1)
chunk_chain_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_m,
                   const __grid_constant__ CUtensorMap tm_ae, const __grid_constant__ CUtensorMap tm_qe,
                   const __grid_constant__ CUtensorMap tm_v, Params p) {
    using LY = Lay<K>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    __shared__ Bars bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3;
    if (grid_seq(p.nz) >= (size_t)p.BH) return;
    const int seq = (int)grid_seq(p.nz), v0 = blockIdx.x * BV;
    const int T = p.T, nch = p.nch;
    const int stall = p.status ? *reinterpret_cast<volatile int *>(p.status + 1) : 0;
    const uint32_t bar_limit = stall ? 64u : kWaitLimit;
    const uint32_t poll_limit = stall ? (1u << 14) : (kWaitLimit << 11);
    // this CTA's chunks, the first whose output it writes, the chunk whose
    // entering state it records (-1: none), and its start and end states
    int cbase = p.c0, ncs = p.ncs, emit_from = p.c0, record_c = -1;
    const float *S0 = p.S0;
    float *ST = p.ST;
    float *spec = nullptr;
    const size_t sstride = (size_t)p.BH * p.V * K;   // one [BH][V][K] state
    if (p.seg_len > 0) {
        const int z = blockIdx.z / p.nz, L = p.seg_len;
        cbase = z == 0 ? 0 : z * L - p.warm;
        ncs = min(nch, (z + 1) * L) - cbase;
        emit_from = z * L;
        record_c = z == 0 ? -1 : z * L;
        S0 = z == 0 ? p.S0 : nullptr;
        ST = z == p.nseg - 1 ? p.ST : p.seg_end + z * sstride;
        spec = z == 0 ? nullptr : p.seg_spec + z * sstride;
    }
    if (p.check) {
        // repair launch: leave if this CTA's rows of the speculative start
        // agree with the exact start (the predecessor's end) already
        __shared__ unsigned s_diff, s_mag;
        if (tid == 0) s_diff = s_mag = 0u;
        __syncthreads();
        float diff = 0.0f, mag = 0.0f;
        for (int i = tid; i < BV * K; i += kThreads) {
            const size_t at = ((size_t)seq * p.V + v0 + i / K) * K + i % K;
            const float a = S0[at], b = p.check[at];
            diff = fmaxf(diff, fabsf(a - b));
            mag = fmaxf(mag, fabsf(a));
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            diff = fmaxf(diff, __shfl_xor_sync(kFullMask, diff, m));
            mag = fmaxf(mag, __shfl_xor_sync(kFullMask, mag, m));
        }
        // non-negative floats order like their bit patterns (a NaN compares high)
        if (lane == 0) {
            atomicMax(&s_diff, __float_as_uint(diff));
            atomicMax(&s_mag, __float_as_uint(mag));
        }
        __syncthreads();
        if (__uint_as_float(s_diff) <= kSpecTol * __uint_as_float(s_mag)) return;
    }
    auto stX = [&](int j) { return smem + LY::oX + (j % NS) * LY::kX; };
    auto stY = [&](int j) { return smem + LY::oY + (j % NS) * LY::kY; };
    // the bf16 copy of the state entering chunk c
    auto sS = [&](int c) { return smem + LY::oS + (c % NSB) * K * 128; };
    int *st = p.status;

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            ptx::mbar_init(&bars.fullX[i], 1);
            ptx::mbar_init(&bars.emptyX[i], 1);
            ptx::mbar_init(&bars.fullY[i], 1);
            ptx::mbar_init(&bars.emptyY[i], 1);
        }
        uint64_t *one[] = {&bars.s_full, &bars.s_ready, &bars.done_s, &bars.done_o,
                           &bars.o_full[0], &bars.o_full[1], &bars.o_free[0], &bars.o_free[1]};
        for (uint64_t *b : one) ptx::mbar_init(b, 1);
        ptx::mbar_init(&bars.s_tmem, 8);   // one arrival per state warp
        for (int i = 0; i < NSB; ++i) {
            ptx::mbar_init(&bars.s_issued[i], 1);
            ptx::mbar_init(&bars.o_read[i], 1);
        }
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

    if (warp == 0) {
        // ======================================================== producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_w);
            ptx::prefetch_tmap(&tm_m);
            ptx::prefetch_tmap(&tm_ae);
            ptx::prefetch_tmap(&tm_qe);
            ptx::prefetch_tmap(&tm_v);
            int lastX = -1, lastY = -1;
            for (int j = 0; j < (stall ? 0 : ncs); ++j) {
                // rows of global chunk cbase + j in (Qe, Ae, V) and (W, M)
                const int t0 = (cbase + j) * C, r0 = (cbase + j) * K;
                if (j >= NS && !wait_bar(&bars.emptyX[j % NS], ((j / NS) - 1) & 1, &s_abort, st, bar_limit)) break;
                uint8_t *x = stX(j);
                ptx::mbar_arrive_expect_tx(&bars.fullX[j % NS], LY::kX);
#pragma unroll
                for (int rb = 0; rb < K / 64; ++rb) {
                    ptx::tma_load_3d(x + rb * 8192, &tm_w, &bars.fullX[j % NS], 0, r0 + rb * 64, seq);
#pragma unroll
                    for (int cb = 0; cb < K / 64; ++cb)
                        ptx::tma_load_3d(x + (1 + cb) * K * 128 + rb * 8192, &tm_m, &bars.fullX[j % NS],
                                         cb * 64, r0 + rb * 64, seq);
                }
                ptx::tma_load_3d(x + LY::oVx, &tm_v, &bars.fullX[j % NS], v0, t0, seq);
                lastX = j;
                if (j >= NS && !wait_bar(&bars.emptyY[j % NS], ((j / NS) - 1) & 1, &s_abort, st, bar_limit)) break;
                uint8_t *y = stY(j);
                ptx::mbar_arrive_expect_tx(&bars.fullY[j % NS], LY::kY);
                ptx::tma_load_3d(y, &tm_ae, &bars.fullY[j % NS], 0, t0, seq);
#pragma unroll
                for (int cb = 0; cb < K / 64; ++cb)
                    ptx::tma_load_3d(y + (1 + cb) * 8192, &tm_qe, &bars.fullY[j % NS], cb * 64, t0, seq);
                ptx::tma_load_3d(y + LY::oVy, &tm_v, &bars.fullY[j % NS], v0, t0, seq);
                lastY = j;
            }
            // bulk copies still in flight (only after an abort) land before exit
            if (s_abort) {
                for (int j = (lastX >= NS ? lastX - NS + 1 : 0); j <= lastX; ++j)
                    drain_bar(&bars.fullX[j % NS], (j / NS) & 1);
                for (int j = (lastY >= NS ? lastY - NS + 1 : 0); j <= lastY; ++j)
                    drain_bar(&bars.fullY[j % NS], (j / NS) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ======================================================== state MMA issuer
        if (lane == 0) {
            const uint32_t id_s = ptx::idesc_bf16(K, BV, 0, 1);    // K-major A, MN-major B
            for (int j = 0; j < ncs; ++j) {
                // S^T += [W | M] [V; S^T]; releases ring X.  W V as soon as the
                // accumulator has been read, M S^T once the bf16 copy is in place.
                if (!wait_poll(&bars.fullX[j % NS], (j / NS) & 1, &s_abort, st, poll_limit) ||
                    !wait_poll(&bars.s_tmem, j & 1, &s_abort, st, poll_limit))
                    break;
                ptx::tc_fence_after();
                const uint32_t x = ptx::smem_u32(stX(j));
                const uint64_t da = dk0(x), dV = dmn0(x + LY::oVx, 8192);
                const uint64_t dSp = dmn0(ptx::smem_u32(sS(j)), 8192);
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    ptx::umma_bf16(tmem + kColS, da + koff(K, ks), dV + mnoff(ks), id_s, 1);
                if (!wait_poll(&bars.s_ready, j & 1, &s_abort, st, poll_limit)) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks)
                    ptx::umma_bf16(tmem + kColS, da + koff(K, 4 + ks), dSp + mnoff(ks), id_s, 1);
                ptx::umma_commit(&bars.s_full);
                ptx::mbar_arrive(&bars.s_issued[j % NSB]);
                ptx::umma_commit(&bars.emptyX[j % NS]);
            }
            // every product issued has completed before TMEM is released
            ptx::umma_commit(&bars.done_s);
            drain_bar(&bars.done_s, 0);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ======================================================== output MMA issuer
        if (lane == 0) {
            const uint32_t id_o = ptx::idesc_bf16(64, BV, 0, 1);
            for (int c = 0; c < ncs; ++c) {
                // O = [Ae | Qe] [V; S^T] of chunk c, behind chunk c's state product
                if (!wait_poll(&bars.fullY[c % NS], (c / NS) & 1, &s_abort, st, poll_limit) ||
                    !wait_poll(&bars.s_issued[c % NSB], (c / NSB) & 1, &s_abort, st, poll_limit) ||
                    (c >= 2 && !wait_poll(&bars.o_free[c & 1], ((c >> 1) - 1) & 1, &s_abort, st, poll_limit)))
                    break;
                ptx::tc_fence_after();
                const uint32_t y = ptx::smem_u32(stY(c));
                const uint64_t da = dk0(y), dV = dmn0(y + LY::oVy, 8192);
                const uint64_t dSp = dmn0(ptx::smem_u32(sS(c)), 8192);
                const uint32_t d = tmem + kColO + 64 * (c & 1);
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    ptx::umma_bf16(d, da + koff(C, ks), dV + mnoff(ks), id_o, ks > 0);
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks)
                    ptx::umma_bf16(d, da + koff(C, 4 + ks), dSp + mnoff(ks), id_o, 1);
                ptx::umma_commit(&bars.o_full[c & 1]);
                ptx::umma_commit(&bars.emptyY[c % NS]);
                ptx::umma_commit(&bars.o_read[c % NSB]);
            }
            ptx::umma_commit(&bars.done_o);
            drain_bar(&bars.done_o, 0);
        }
        __syncwarp();
    } else if (warp < 7) {
        // ======================================================== O readout
        const int ot = tid - 96;
        const int trow = 16 * q4 + lane;   // M=64 accumulator: lanes 0-15 of each quarter
        for (int j = 0; j < ncs; ++j) {
            if (!vote_all(wait_bar(&bars.o_full[j & 1], (j >> 1) & 1, &s_abort, st, bar_limit), 3, 128)) break;
            ptx::tc_fence_after();
            float o[64];
            tmem_ld64(tmem + lane_off + kColO + 64 * (j & 1), o);
            ptx::tc_fence_before();
            ptx::named_bar(3, 128);
            if (ot == 0) ptx::mbar_arrive(&bars.o_free[j & 1]);
            const int t = (cbase + j) * C + trow;
            if (lane < 16 && t < T && cbase + j >= emit_from)
                st_global_bf16(p.o + ((size_t)seq * T + t) * p.V + v0, o, 64);
        }
    } else {
        // ======================================================== state
        const int sti = tid - 224, half = (warp - 7) >> 2, c0 = 32 * half;
        // S^T row k: TMEM lane k (M=128) or 32*(k/16) + k%16 (M=64); columns c0..c0+31
        const int krow = (K == 128) ? 32 * q4 + lane : 16 * q4 + lane;
        const bool act = (K == 128) || lane < 16;
        const uint32_t tS = tmem + lane_off + kColS + c0;
        {  // initial state: TMEM S^T = g_C(0) S0^T, bf16 copy = S0^T
            const float g0 = !GATED ? 1.0f
                             : PCH ? (act ? p.gc[((size_t)seq * nch + cbase) * K + krow] : 1.0f)
                                   : p.gc[(size_t)seq * nch + cbase];
            float sv[32];
#pragma unroll
            for (int e = 0; e < 32; ++e)
                sv[e] = (act && S0) ? S0[((size_t)seq * p.V + v0 + c0 + e) * K + krow] : 0.0f;
            if (act) st_row_sw128(sS(0), K, krow, c0, sv, 32);
            float lo[16], hi[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                lo[e] = g0 * sv[e];
                hi[e] = g0 * sv[16 + e];
            }
            ptx::tmem_st16(tS, lo);
            ptx::tmem_st16(tS + 16, hi);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bars.s_tmem);
            ptx::fence_proxy_async_smem();
            ptx::named_bar(1, 256);
            if (sti == 0) ptx::mbar_arrive(&bars.s_ready);
        }
        for (int j = 0; j < ncs; ++j) {
            const bool last = (j == ncs - 1);
            const float gN = (!GATED || last) ? 1.0f
                             : PCH ? (act ? p.gc[((size_t)seq * nch + cbase + j + 1) * K + krow] : 1.0f)
                                   : p.gc[(size_t)seq * nch + cbase + j + 1];
            // the copy entering chunk j+1 overwrites the one chunk j-2's output read
            const int n = j + 1;
            const bool okw = (last || n < NSB ||
                              wait_poll(&bars.o_read[n % NSB], ((n / NSB) - 1) & 1, &s_abort, st, poll_limit)) &&
                             wait_poll(&bars.s_full, j & 1, &s_abort, st, poll_limit);
            if (!vote_all(okw, 1, 256)) break;
            ptx::tc_fence_after();
            float sv[32];
            tmem_ld32(tS, sv);
            if (last) {
                if (act && ST) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) ST[((size_t)seq * p.V + v0 + c0 + e) * K + krow] = sv[e];
                }
                break;
            }
            if (act && cbase + j + 1 == record_c) {   // the state entering the segment's first chunk
#pragma unroll
                for (int e = 0; e < 32; ++e) spec[((size_t)seq * p.V + v0 + c0 + e) * K + krow] = sv[e];
            }
            if (GATED) {  // the next chunk's decay, applied before its update
                float lo[16], hi[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    lo[e] = gN * sv[e];
                    hi[e] = gN * sv[16 + e];
                }
                ptx::tmem_st16(tS, lo);
                ptx::tmem_st16(tS + 16, hi);
                ptx::tmem_wait_st();
            }
            // this warp is done with the accumulator
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bars.s_tmem);
            if (act) st_row_sw128(sS(n), K, krow, c0, sv, 32);
            ptx::fence_proxy_async_smem();
            ptx::named_bar(1, 256);
            if (sti == 0) ptx::mbar_arrive(&bars.s_ready);
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
}

// What a chain launch does beyond its chunk range: the speculative pass over
// time segments (grid z = segment), or a repair launch that first checks
// each CTA's speculative start (see Params).
struct ChainOpt {
    int seg_len = 0, warm = 0, nseg = 0;
    float *seg_spec = nullptr, *seg_end = nullptr;
    const float *check = nullptr;
};

// Chunks [c0, c1) of every sequence, from the state S0 (NULL: zeros) to ST
// (NULL: not written).
template <int K, bool GATED, bool PCH>
cudaError_t chain_launch_t(int BH, int T, int V, int c0, int c1, const void *v,
                           const __nv_bfloat16 *w, const __nv_bfloat16 *m,
                           const __nv_bfloat16 *qe, const __nv_bfloat16 *ae, const float *gc,
                           const float *S0, void *o, float *ST, int *status, cudaStream_t stream,
                           const ChainOpt &opt) {
    const int nch = (T + C - 1) / C, Tp = nch * C;
    CUtensorMap mw, mm, mae, mqe, mv;
    if (!make_map(&mw, w, BH, nch * K, C) || !make_map(&mm, m, BH, nch * K, K) ||
        !make_map(&mae, ae, BH, Tp, C) || !make_map(&mqe, qe, BH, Tp, K) ||
        !make_map(&mv, v, BH, T, V))
        return cudaErrorInvalidValue;
    constexpr int smem = Lay<K>::kAlloc;
    static std::atomic<unsigned long long> attr_done{0};
    {
        cudaError_t e = smem_attr_once((const void *)chunk_chain_kernel<K, GATED, PCH>, smem, attr_done);
        if (e != cudaSuccess) return e;
    }
    Params p;
    p.T = T;
    p.V = V;
    p.nch = nch;
    p.c0 = c0;
    p.ncs = c1 - c0;
    p.S0 = S0;
    p.gc = gc;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.ST = ST;
    p.seg_len = opt.seg_len;
    p.warm = opt.warm;
    p.nseg = opt.nseg;
    p.seg_spec = opt.seg_spec;
    p.seg_end = opt.seg_end;
    p.check = opt.check;
    p.status = status;
    p.BH = BH;
    const dim3 grid = seq_grid(V / BV, BH, opt.seg_len > 0 ? opt.nseg : 1);
    p.nz = (int)((BH + grid.y - 1) / grid.y);
    chunk_chain_kernel<K, GATED, PCH><<<grid, kThreads, smem, stream>>>(mw, mm, mae, mqe, mv, p);
    return cudaGetLastError();
}

// Time segments of the chain with a decay (the state then forgets its start):
// as many as keep one wave of chain CTAs (one per SM), with at least
// kMinSegChunks chunks each; 1 when that leaves a single segment.
constexpr int kMinSegChunks = 16;
constexpr int kWarmChunks = 4;   // warm-up of a speculative segment: 256 tokens
int chain_segments(int BH, int T, int V) {
    const long long nch = ((long long)T + C - 1) / C;
    const long long ctas = (long long)BH * (V / BV);
    long long n = ctas > 0 ? sm_count() / ctas : 1;
    n = std::min(n, nch / kMinSegChunks);
    return (int)std::max(1LL, n);
}

// Workspace carve-up: the prepared operands (W and M per chunk, K rows each;
// Qe and Ae per token, chunk-padded; g_C per chunk), two fp32 states
// [BH][V][K] that carry S from one slab of chunks to the next, and, where the
// chain may run in time segments, each segment's speculative start and end
// state.
struct Carve {
    __nv_bfloat16 *w, *m, *qe, *ae;
    float *gc, *state[2], *seg_spec, *seg_end;
    int nseg;
    size_t bytes;
};
size_t round256(size_t x) { return (x + 255) / 256 * 256; }
Carve carve(void *base, int BH, int T, int K, int V, bool pch = false) {
    const size_t nch = (size_t)(T + C - 1) / C, Tp = nch * C;
    const int nseg = chain_segments(BH, T, V);
    const size_t segb = nseg > 1 ? round256((size_t)nseg * BH * V * K * 4) : 0;
    const size_t sz[9] = {round256((size_t)BH * nch * K * C * 2), round256((size_t)BH * nch * K * K * 2),
                          round256((size_t)BH * Tp * K * 2), round256((size_t)BH * Tp * C * 2),
                          round256((size_t)BH * nch * (pch ? K : 1) * 4), round256((size_t)BH * V * K * 4),
                          round256((size_t)BH * V * K * 4), segb, segb};
    char *b = static_cast<char *>(base);
    char *ptrs[9];
    size_t off = 0;
    for (int i = 0; i < 9; ++i) {
        ptrs[i] = b ? b + off : nullptr;
        off += sz[i];
    }
    Carve c;
    c.w = reinterpret_cast<__nv_bfloat16 *>(ptrs[0]);
    c.m = reinterpret_cast<__nv_bfloat16 *>(ptrs[1]);
    c.qe = reinterpret_cast<__nv_bfloat16 *>(ptrs[2]);
    c.ae = reinterpret_cast<__nv_bfloat16 *>(ptrs[3]);
    c.gc = reinterpret_cast<float *>(ptrs[4]);
    c.state[0] = reinterpret_cast<float *>(ptrs[5]);
    c.state[1] = reinterpret_cast<float *>(ptrs[6]);
    c.seg_spec = reinterpret_cast<float *>(ptrs[7]);
    c.seg_end = reinterpret_cast<float *>(ptrs[8]);
    c.nseg = nseg;
    c.bytes = off;
    return c;
}

// Slabs of chunks: preparation of slab s+1 runs on the SMs the chain of slab
// s leaves idle.  Two internal streams per device (the chain at the highest
// priority, so its CTAs take SMs first) and a pool of events, set up once;
// the enqueue is serialised so that concurrent calls do not share events.
constexpr int kSlabChunks = 64;     // chunks per slab (at least)
constexpr int kMaxSlabs = 64;
struct Overlap {
    cudaStream_t chain = nullptr, prep = nullptr;
    cudaEvent_t ev[kMaxSlabs + 2] = {};
    bool ready = false;
};
constexpr int kMaxDevices = 64;
Overlap g_overlap[kMaxDevices];
std::mutex g_overlap_mu;

cudaError_t overlap_for(int dev, Overlap **out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    Overlap &o = g_overlap[dev];
    if (!o.ready) {
        int least = 0, greatest = 0;
        cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&o.chain, cudaStreamNonBlocking, greatest);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&o.prep, cudaStreamNonBlocking, least);
        for (int i = 0; e == cudaSuccess && i < kMaxSlabs + 2; ++i)
            e = cudaEventCreateWithFlags(&o.ev[i], cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
        o.ready = true;
    }
    *out = &o;
    return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

}  // namespace

bool tensor_map_encoder_ready() {
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

bool make_map(CUtensorMap *m, const void *ptr, int BH, int rows, int width) {
    cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)rows, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * (cuuint64_t)rows};
    cuuint32_t box[3] = {64, (cuuint32_t)C, 1}, es[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace tc

size_t delta_tc_scratch_bytes(int BH, int T, int K, int V) {
    return tc::carve(nullptr, BH, T, K, V).bytes;
}

size_t delta_tc_kda_scratch_bytes(int BH, int T, int K, int V) {
    return tc::carve(nullptr, BH, T, K, V, true).bytes;
}

namespace {
cudaError_t prep_range(int BH, int T, int K, int c0, int c1, const void *q, const void *k,
                       const void *kt, const float *beta, const float *alpha, const tc::Fused &fz,
                       const tc::Carve &w, int *status, cudaStream_t stream) {
    return tc::chunk_prep_launch(BH, T, K, c0, c1, q, k, kt, beta, alpha, fz, w.w, w.m, w.qe, w.ae,
                                 w.gc, status, stream);
}
template <int K>
cudaError_t chain_range_k(int BH, int T, int V, int c0, int c1, const void *v, const float *alpha,
                          bool pch, const tc::Carve &w, const float *S0, void *o, float *ST,
                          int *status, cudaStream_t stream, const tc::ChainOpt &opt) {
    if (pch)
        return tc::chain_launch_t<K, true, true>(BH, T, V, c0, c1, v, w.w, w.m, w.qe, w.ae, w.gc, S0, o, ST, status, stream, opt);
    if (alpha)
        return tc::chain_launch_t<K, true, false>(BH, T, V, c0, c1, v, w.w, w.m, w.qe, w.ae, w.gc, S0, o, ST, status, stream, opt);
    return tc::chain_launch_t<K, false, false>(BH, T, V, c0, c1, v, w.w, w.m, w.qe, w.ae, w.gc, S0, o, ST, status, stream, opt);
}
// `alpha` is a scalar decay [BH][T] or, with pch, one per key channel [BH][T][K].
cudaError_t chain_range(int BH, int T, int K, int V, int c0, int c1, const void *v, const float *alpha,
                        bool pch, const tc::Carve &w, const float *S0, void *o, float *ST,
                        int *status, cudaStream_t stream, const tc::ChainOpt &opt = tc::ChainOpt()) {
    if (K == 128)
        return chain_range_k<128>(BH, T, V, c0, c1, v, alpha, pch, w, S0, o, ST, status, stream, opt);
    return chain_range_k<64>(BH, T, V, c0, c1, v, alpha, pch, w, S0, o, ST, status, stream, opt);
}

// With a decay the state forgets where it started, so the chain can run in
// time segments: every segment but the first starts from a zero state a few
// chunks early (speculative pass, all segments at once); then, in segment
// order, each segment's recorded start is compared with its predecessor's
// end and, where they differ by more than 2^-16 of that end's largest entry,
// the segment is recomputed from that exact end.  Every accepted start is
// therefore that close to the state the unsegmented chain would carry in.
cudaError_t chain_segmented(int BH, int T, int K, int V, int nch, const void *v, const float *alpha,
                            bool pch, const tc::Carve &w, const float *S0, void *o, float *ST, int *status,
                            cudaStream_t stream) {
    const int nseg = w.nseg, L = (nch + nseg - 1) / nseg;
    const size_t sstride = (size_t)BH * V * K;
    tc::ChainOpt spec;
    spec.seg_len = L;
    spec.warm = tc::kWarmChunks;
    spec.nseg = (nch + L - 1) / L;
    spec.seg_spec = w.seg_spec;
    spec.seg_end = w.seg_end;
    cudaError_t e = chain_range(BH, T, K, V, 0, nch, v, alpha, pch, w, S0, o, ST, status, stream, spec);
    for (int i = 1; e == cudaSuccess && i < spec.nseg; ++i) {
        tc::ChainOpt rep;
        rep.check = w.seg_spec + i * sstride;
        const int c0 = i * L, c1 = std::min(nch, c0 + L);
        float *sout = i == spec.nseg - 1 ? ST : w.seg_end + i * sstride;
        e = chain_range(BH, T, K, V, c0, c1, v, alpha, pch, w, w.seg_end + (i - 1) * sstride, o, sout,
                        status, stream, rep);
    }
    return e;
}
}  // namespace

namespace {
cudaError_t delta_tc_impl(int BH, int T, int K, int V, const void *q, const void *k,
                          const void *kt, const void *v, const float *beta, const float *alpha,
                          const tc::Fused &fz, const float *S0, void *o, float *ST, void *scratch,
                          int *status, cudaStream_t stream) {
    if (!tc::tensor_map_encoder_ready()) return cudaErrorNotSupported;
    const bool pch = fz.alpha_k != nullptr;        // a decay per key channel
    const float *decay = pch ? fz.alpha_k : alpha;
    const tc::Carve w = tc::carve(scratch, BH, T, K, V, pch);
    const int nch = (T + tc::C - 1) / tc::C;
    int per = tc::kSlabChunks;
    while ((nch + per - 1) / per > tc::kMaxSlabs) per *= 2;
    // a sequence of one slab is still split in two when the chain leaves at
    // least half the SMs to the preparation of its second half
    if (nch <= per && nch >= 32 && (long long)BH * (V / tc::BV) * 2 <= tc::sm_count())
        per = (nch + 1) / 2;
    const int nslab = (nch + per - 1) / per;
    if (decay && w.nseg > 1) {  // a decay: every chunk prepared, then the chain in time segments
        cudaError_t e = prep_range(BH, T, K, 0, nch, q, k, kt, beta, alpha, fz, w, status, stream);
        if (e != cudaSuccess) return e;
        return chain_segmented(BH, T, K, V, nch, v, decay, pch, w, S0, o, ST, status, stream);
    }
    if (nslab <= 1) {  // one slab: preparation, then the chain, on the caller's stream
        cudaError_t e = prep_range(BH, T, K, 0, nch, q, k, kt, beta, alpha, fz, w, status, stream);
        if (e != cudaSuccess) return e;
        return chain_range(BH, T, K, V, 0, nch, v, decay, pch, w, S0, o, ST, status, stream);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(tc::g_overlap_mu);
    tc::Overlap *ov = nullptr;
    if ((e = tc::overlap_for(dev, &ov)) != cudaSuccess) return e;
    cudaEvent_t *ev = ov->ev;
    // fork: both internal streams start after the caller's prior work
    if ((e = cudaEventRecord(ev[0], stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ov->chain, ev[0], 0)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ov->prep, ev[0], 0)) != cudaSuccess) return e;
    // slab 0 prepared ahead of the chain; slabs 1.. prepared behind it
    if ((e = prep_range(BH, T, K, 0, per, q, k, kt, beta, alpha, fz, w, status, ov->chain)) != cudaSuccess)
        return e;
    for (int s = 1; s < nslab; ++s) {
        const int c0 = s * per, c1 = std::min(nch, c0 + per);
        if ((e = prep_range(BH, T, K, c0, c1, q, k, kt, beta, alpha, fz, w, status, ov->prep)) != cudaSuccess)
            return e;
        if ((e = cudaEventRecord(ev[1 + s], ov->prep)) != cudaSuccess) return e;
    }
    for (int s = 0; s < nslab; ++s) {
        const int c0 = s * per, c1 = std::min(nch, c0 + per);
        if (s >= 1 && (e = cudaStreamWaitEvent(ov->chain, ev[1 + s], 0)) != cudaSuccess) return e;
        const float *sin = s == 0 ? S0 : w.state[(s - 1) & 1];
        float *sout = s == nslab - 1 ? ST : w.state[s & 1];
        if ((e = chain_range(BH, T, K, V, c0, c1, v, decay, pch, w, sin, o, sout, status, ov->chain)) !=
            cudaSuccess)
            return e;
    }
    // join: the caller's stream continues after the last chain slab (which
    // itself waited for the last preparation slab)
    if ((e = cudaEventRecord(ev[1], ov->chain)) != cudaSuccess) return e;
    return cudaStreamWaitEvent(stream, ev[1], 0);
}
}  // namespace

cudaError_t delta_tc_launch(int BH, int T, int K, int V, const void *q, const void *k,
                            const void *kt, const void *v, const float *beta, const float *alpha,
                            const float *S0, void *o, float *ST, void *scratch, int *status,
                            cudaStream_t stream) {
    return delta_tc_impl(BH, T, K, V, q, k, kt, v, beta, alpha, tc::Fused(), S0, o, ST, scratch,
                         status, stream);
}

// The fused forward pass's Phase 2: Kt is rebuilt chunk by chunk from the
// preconditioner scan's checkpoints (e_t of every token, d entering every
// chunk) and never read from or written to global memory.
cudaError_t delta_tc_fused_launch(int BH, int T, int K, int V, const void *q, const void *k,
                                  const void *v, const float *beta, const float *r,
                                  const float *ecoef, const float *dchk, const float *alpha,
                                  const float *S0, void *o, float *ST, void *scratch, int *status,
                                  cudaStream_t stream) {
    tc::Fused fz;
    fz.r = r;
    fz.ecoef = ecoef;
    fz.dchk = dchk;
    return delta_tc_impl(BH, T, K, V, q, k, nullptr, v, beta, alpha, fz, S0, o, ST, scratch, status,
                         stream);
}

// Phase 2 with a decay per key channel (alpha_k [BH][T][K]) on the tensor
// cores: the same preparation and chain, with the decay folded into the
// operands per channel (see phase2_prep.cu) and applied per state row.
cudaError_t delta_tc_kda_launch(int BH, int T, int K, int V, const void *q, const void *k,
                                const void *kt, const void *v, const float *beta,
                                const float *alpha_k, const float *S0, void *o, float *ST,
                                void *scratch, int *status, cudaStream_t stream) {
    tc::Fused fz;
    fz.alpha_k = alpha_k;
    return delta_tc_impl(BH, T, K, V, q, k, kt, v, beta, nullptr, fz, S0, o, ST, scratch, status,
                         stream);
}

}  // namespace osdn
