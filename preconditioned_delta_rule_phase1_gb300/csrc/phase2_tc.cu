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
// fold it into the operands Kwn, Qe, Xb, Ae.  The chain kernel here then runs
// the state recurrence, one chunk of C = 64 tokens after the other:
//   [U; O] = [Xb; Ae] V + [Kwn; Qe] S^T          (one M=128 accumulator)
//   S'^T   = g_C S^T + Kt^T (diag(g_C / g) U)
// with S^T kept as an fp32 accumulator in TMEM and as a bf16 copy in shared
// memory (the B operand of the next chunk's product).
//
// One CTA per (sequence, 64 columns of V), 320 threads in five roles:
//   warp 0      TMA producer: V and [Xb; Ae] (2-deep ring), [Kwn; Qe] and Kt
//               (3- or 4-deep ring);
//   warp 1      MMA issuer (one thread): every tcgen05.mma and commit;
//   warps 2-3   O out of TMEM (rows 64-127) to global memory as bf16;
//   warps 4-7   the state: S^T out of TMEM, its bf16 copy, the decay g_C,
//               and the final state;
//   warps 8-9   U out of TMEM (rows 0-63), scaled by g_C / g, as the bf16 B
//               operand of the state update.
// The chain per chunk is: product into [U; O] -> U to shared memory -> state
// update -> S^T to shared memory; the product of the next chunk's V term and
// the O readout overlap it.  Every wait is bounded: a wait that runs out
// records OSDN_ERR_TIMEOUT in the status word and all roles leave their loops.
#include "tc_common.cuh"

namespace osdn {
namespace tc {

cudaError_t chunk_prep_launch(int BH, int T, int K, const void *q, const void *k, const void *kt,
                              const float *beta, const float *alpha, __nv_bfloat16 *kwn,
                              __nv_bfloat16 *qe, __nv_bfloat16 *xb, __nv_bfloat16 *ae, float *gk,
                              float *gc, int *status, cudaStream_t stream);

namespace {

constexpr int BV = 64;          // columns of V (rows of S) per CTA
constexpr int NA = 2;           // depth of the V / [Xb; Ae] ring
constexpr int kThreads = 320;
constexpr uint32_t kColUO = 0;  // [U; O] (M=128), two buffers of 64 columns
constexpr uint32_t kColS = 128; // S^T (M=K), 64 columns
constexpr uint32_t kTmemCols = 256;

// Shared memory: ring A stages ([Xb; Ae] as one 128-row K-major block, then
// V), ring B stages ([Kwn; Qe] as 128-row blocks of 64 columns, then Kt in
// 64-row blocks), the bf16 copy of S^T (K rows of 64 values) and the scaled
// U (64 rows of 64 values).
template <int K>
struct Lay {
    static constexpr int NB = (K == 128) ? 3 : 4;
    static constexpr int kA = 3 * C * 128;
    static constexpr int kB = 128 * K * 2 + C * K * 2;
    static constexpr int oKt = 128 * K * 2;    // within a ring B stage
    static constexpr int oV = 2 * C * 128;     // within a ring A stage
    static constexpr int oA = 0;
    static constexpr int oB = NA * kA;
    static constexpr int oS = oB + NB * kB;
    static constexpr int oU = oS + K * 128;
    static constexpr int kBytes = oU + C * 128;
    static constexpr int kAlloc = kBytes + 1024;
};

struct Params {
    int T, V, nch, Tp;
    const float *S0, *gk, *gc;
    __nv_bfloat16 *o;
    float *ST;
    int *status;
};

template <int NB>
struct Bars {
    uint64_t fullA[NA], emptyA[NA], fullB[NB], emptyB[NB];
    uint64_t u_full, u_sm, s_full, s_ready, done;
    uint64_t o_full[2], acc_free[2];
};

template <int K, bool GATED>
__global__ void __launch_bounds__(kThreads, 1)
chunk_chain_kernel(const __grid_constant__ CUtensorMap tm_xb, const __grid_constant__ CUtensorMap tm_ae,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kwn,
                   const __grid_constant__ CUtensorMap tm_qe, const __grid_constant__ CUtensorMap tm_kt,
                   Params p) {
    using LY = Lay<K>;
    constexpr int NB = LY::NB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    __shared__ Bars<NB> bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3;
    const int seq = blockIdx.y, v0 = blockIdx.x * BV;
    const int T = p.T, nch = p.nch;
    uint8_t *sS = smem + LY::oS, *sU = smem + LY::oU;
    auto stA = [&](int j) { return smem + LY::oA + (j % NA) * LY::kA; };
    auto stB = [&](int j) { return smem + LY::oB + (j % NB) * LY::kB; };
    int *st = p.status;

    if (tid == 0) {
        for (int i = 0; i < NA; ++i) {
            ptx::mbar_init(&bars.fullA[i], 1);
            ptx::mbar_init(&bars.emptyA[i], 1);
        }
        for (int i = 0; i < NB; ++i) {
            ptx::mbar_init(&bars.fullB[i], 1);
            ptx::mbar_init(&bars.emptyB[i], 1);
        }
        uint64_t *one[] = {&bars.u_full, &bars.u_sm, &bars.s_full, &bars.s_ready, &bars.done,
                           &bars.o_full[0], &bars.o_full[1], &bars.acc_free[0], &bars.acc_free[1]};
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

    if (warp == 0) {
        // ======================================================== producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_xb);
            ptx::prefetch_tmap(&tm_ae);
            ptx::prefetch_tmap(&tm_v);
            ptx::prefetch_tmap(&tm_kwn);
            ptx::prefetch_tmap(&tm_qe);
            ptx::prefetch_tmap(&tm_kt);
            int lastA = -1, lastB = -1;
            for (int j = 0; j < nch; ++j) {
                const int t0 = j * C;
                if (j >= NA && !wait_bar(&bars.emptyA[j % NA], ((j / NA) - 1) & 1, &s_abort, st)) break;
                uint8_t *a = stA(j);
                ptx::mbar_arrive_expect_tx(&bars.fullA[j % NA], LY::kA);
                ptx::tma_load_3d(a, &tm_xb, &bars.fullA[j % NA], 0, t0, seq);
                ptx::tma_load_3d(a + C * 128, &tm_ae, &bars.fullA[j % NA], 0, t0, seq);
                ptx::tma_load_3d(a + LY::oV, &tm_v, &bars.fullA[j % NA], v0, t0, seq);
                lastA = j;
                if (j >= NB && !wait_bar(&bars.emptyB[j % NB], ((j / NB) - 1) & 1, &s_abort, st)) break;
                uint8_t *b = stB(j);
                ptx::mbar_arrive_expect_tx(&bars.fullB[j % NB], LY::kB);
#pragma unroll
                for (int cb = 0; cb < K / 64; ++cb) {
                    ptx::tma_load_3d(b + cb * 16384, &tm_kwn, &bars.fullB[j % NB], cb * 64, t0, seq);
                    ptx::tma_load_3d(b + cb * 16384 + 8192, &tm_qe, &bars.fullB[j % NB], cb * 64, t0, seq);
                    ptx::tma_load_3d(b + LY::oKt + cb * 8192, &tm_kt, &bars.fullB[j % NB], cb * 64, t0, seq);
                }
                lastB = j;
            }
            // bulk copies still in flight (only after an abort) land before exit
            if (s_abort) {
                for (int j = (lastA >= NA ? lastA - NA + 1 : 0); j <= lastA; ++j)
                    drain_bar(&bars.fullA[j % NA], (j / NA) & 1);
                for (int j = (lastB >= NB ? lastB - NB + 1 : 0); j <= lastB; ++j)
                    drain_bar(&bars.fullB[j % NB], (j / NB) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ======================================================== MMA issuer
        if (lane == 0) {
            const uint32_t aS = ptx::smem_u32(sS), aU = ptx::smem_u32(sU);
            const uint32_t id_uo = ptx::idesc_bf16(128, BV, 0, 1);   // K-major A, MN-major B
            const uint32_t id_s = ptx::idesc_bf16(K, BV, 1, 1);      // Kt^T (MN-major) x U
            const uint64_t dS = dmn0(aS, 8192), dU = dmn0(aU, 8192);
            auto vterm = [&](int j) {  // [U; O] of chunk j = [Xb; Ae] V
                const uint32_t a = ptx::smem_u32(stA(j));
                const uint64_t da = dk0(a), dv = dmn0(a + LY::oV, 8192);
                const uint32_t d = tmem + kColUO + 64 * (j & 1);
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    ptx::umma_bf16(d, da + koff(128, ks), dv + mnoff(ks), id_uo, ks > 0);
                ptx::umma_commit(&bars.emptyA[j % NA]);
            };
            bool ok = wait_bar(&bars.fullA[0], 0, &s_abort, st);
            if (ok) {
                ptx::tc_fence_after();
                vterm(0);
            }
            for (int j = 0; ok && j < nch; ++j) {
                if (!wait_bar(&bars.fullB[j % NB], (j / NB) & 1, &s_abort, st)) break;
                if (!wait_bar(&bars.s_ready, j & 1, &s_abort, st)) break;
                ptx::tc_fence_after();
                const uint32_t b = ptx::smem_u32(stB(j));
                {  // [U; O] += [Kwn; Qe] S^T
                    const uint64_t da = dk0(b);
                    const uint32_t d = tmem + kColUO + 64 * (j & 1);
#pragma unroll
                    for (int ks = 0; ks < K / 16; ++ks)
                        ptx::umma_bf16(d, da + koff(128, ks), dS + mnoff(ks), id_uo, 1);
                    ptx::umma_commit(&bars.u_full);
                    ptx::umma_commit(&bars.o_full[j & 1]);
                }
                if (!wait_bar(&bars.u_sm, j & 1, &s_abort, st)) break;
                ptx::tc_fence_after();
                {  // S^T += Kt^T Uh
                    const uint64_t da = dmn0(b + LY::oKt, 8192);
#pragma unroll
                    for (int ks = 0; ks < C / 16; ++ks)
                        ptx::umma_bf16(tmem + kColS, da + mnoff(ks), dU + mnoff(ks), id_s, 1);
                    ptx::umma_commit(&bars.s_full);
                    ptx::umma_commit(&bars.emptyB[j % NB]);
                }
                if (j + 1 < nch) {  // V term of the next chunk, once its buffer is read out
                    const int n = j + 1;
                    if (!wait_bar(&bars.fullA[n % NA], (n / NA) & 1, &s_abort, st)) break;
                    if (n >= 2 && !wait_bar(&bars.acc_free[n & 1], ((n >> 1) - 1) & 1, &s_abort, st)) break;
                    ptx::tc_fence_after();
                    vterm(n);
                }
            }
            // every product issued has completed before TMEM is released
            ptx::umma_commit(&bars.done);
            drain_bar(&bars.done, 0);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ======================================================== O readout
        const int ot = tid - 64;   // row t of the chunk (TMEM lane 64 + t)
        for (int j = 0; j < nch; ++j) {
            if (!vote_all(wait_bar(&bars.o_full[j & 1], (j >> 1) & 1, &s_abort, st), 3, 64)) break;
            ptx::tc_fence_after();
            float o[64];
            tmem_ld64(tmem + lane_off + kColUO + 64 * (j & 1), o);
            ptx::tc_fence_before();
            ptx::named_bar(3, 64);
            if (ot == 0) ptx::mbar_arrive(&bars.acc_free[j & 1]);
            const int t = j * C + ot;
            if (t < T) st_global_bf16(p.o + ((size_t)seq * T + t) * p.V + v0, o, 64);
        }
    } else if (warp < 8) {
        // ======================================================== state
        const int sti = tid - 128;
        // S^T row k: TMEM lane k (M=128) or 32*(k/16) + k%16 (M=64)
        const int krow = (K == 128) ? 32 * q4 + lane : 16 * q4 + lane;
        const bool act = (K == 128) || lane < 16;
        {  // initial state: TMEM S^T = g_C(0) S0^T, bf16 copy = S0^T
            const float g0 = GATED ? p.gc[(size_t)seq * nch] : 1.0f;
#pragma unroll
            for (int c0 = 0; c0 < BV; c0 += 32) {
                float sv[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    sv[e] = (act && p.S0) ? p.S0[((size_t)seq * p.V + v0 + c0 + e) * K + krow] : 0.0f;
                if (act) st_row_sw128(sS, K, krow, c0, sv, 32);
                float lo[16], hi[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    lo[e] = g0 * sv[e];
                    hi[e] = g0 * sv[16 + e];
                }
                ptx::tmem_st16(tmem + lane_off + kColS + c0, lo);
                ptx::tmem_st16(tmem + lane_off + kColS + c0 + 16, hi);
            }
            ptx::tmem_wait_st();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_bar(1, 128);
            if (sti == 0) ptx::mbar_arrive(&bars.s_ready);
        }
        for (int j = 0; j < nch; ++j) {
            const bool last = (j == nch - 1);
            const float gN = (GATED && !last) ? p.gc[(size_t)seq * nch + j + 1] : 1.0f;
            if (!vote_all(wait_bar(&bars.s_full, j & 1, &s_abort, st), 1, 128)) break;
            ptx::tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < BV; c0 += 32) {
                float sv[32];
                tmem_ld32(tmem + lane_off + kColS + c0, sv);
                if (last) {
                    if (act && p.ST) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            p.ST[((size_t)seq * p.V + v0 + c0 + e) * K + krow] = sv[e];
                    }
                } else {
                    if (act) st_row_sw128(sS, K, krow, c0, sv, 32);
                    if (GATED) {  // the next chunk's decay, applied before its update
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
            }
            if (last) break;
            if (GATED) ptx::tmem_wait_st();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_bar(1, 128);
            if (sti == 0) ptx::mbar_arrive(&bars.s_ready);
        }
    } else {
        // ======================================================== U readout
        const int ut = tid - 256;   // row t of the chunk (TMEM lane t)
        for (int j = 0; j < nch; ++j) {
            const float gk = GATED ? p.gk[(size_t)seq * p.Tp + j * C + ut] : 1.0f;
            if (!vote_all(wait_bar(&bars.u_full, j & 1, &s_abort, st), 2, 64)) break;
            ptx::tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < BV; c0 += 32) {
                float u[32];
                tmem_ld32(tmem + lane_off + kColUO + 64 * (j & 1) + c0, u);
                if (GATED) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) u[e] *= gk;
                }
                st_row_sw128(sU, C, ut, c0, u, 32);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_bar(2, 64);
            if (ut == 0) ptx::mbar_arrive(&bars.u_sm);
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
}

template <int K, bool GATED>
cudaError_t chain_launch_t(int BH, int T, int V, const void *kt, const void *v,
                           const __nv_bfloat16 *kwn, const __nv_bfloat16 *qe,
                           const __nv_bfloat16 *xb, const __nv_bfloat16 *ae, const float *gk,
                           const float *gc, const float *S0, void *o, float *ST, int *status,
                           cudaStream_t stream) {
    const int nch = (T + C - 1) / C, Tp = nch * C;
    CUtensorMap mxb, mae, mv, mkwn, mqe, mkt;
    if (!make_map(&mxb, xb, BH, Tp, C) || !make_map(&mae, ae, BH, Tp, C) ||
        !make_map(&mv, v, BH, T, V) || !make_map(&mkwn, kwn, BH, Tp, K) ||
        !make_map(&mqe, qe, BH, Tp, K) || !make_map(&mkt, kt, BH, T, K))
        return cudaErrorInvalidValue;
    constexpr int smem = Lay<K>::kAlloc;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(chunk_chain_kernel<K, GATED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    Params p;
    p.T = T;
    p.V = V;
    p.nch = nch;
    p.Tp = Tp;
    p.S0 = S0;
    p.gk = gk;
    p.gc = gc;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.ST = ST;
    p.status = status;
    dim3 grid(V / BV, BH);
    chunk_chain_kernel<K, GATED><<<grid, kThreads, smem, stream>>>(mxb, mae, mv, mkwn, mqe, mkt, p);
    return cudaGetLastError();
}

// Workspace carve-up of the prepared operands, chunk-padded to Tp rows.
struct Carve {
    __nv_bfloat16 *kwn, *qe, *xb, *ae;
    float *gk, *gc;
    size_t bytes;
};
size_t round256(size_t x) { return (x + 255) / 256 * 256; }
Carve carve(void *base, int BH, int T, int K) {
    const size_t nch = (size_t)(T + C - 1) / C, Tp = nch * C;
    const size_t sz[6] = {round256((size_t)BH * Tp * K * 2), round256((size_t)BH * Tp * K * 2),
                          round256((size_t)BH * Tp * C * 2), round256((size_t)BH * Tp * C * 2),
                          round256((size_t)BH * Tp * 4), round256((size_t)BH * nch * 4)};
    char *b = static_cast<char *>(base);
    Carve c;
    size_t off = 0;
    char *ptrs[6];
    for (int i = 0; i < 6; ++i) {
        ptrs[i] = b ? b + off : nullptr;
        off += sz[i];
    }
    c.kwn = reinterpret_cast<__nv_bfloat16 *>(ptrs[0]);
    c.qe = reinterpret_cast<__nv_bfloat16 *>(ptrs[1]);
    c.xb = reinterpret_cast<__nv_bfloat16 *>(ptrs[2]);
    c.ae = reinterpret_cast<__nv_bfloat16 *>(ptrs[3]);
    c.gk = reinterpret_cast<float *>(ptrs[4]);
    c.gc = reinterpret_cast<float *>(ptrs[5]);
    c.bytes = off;
    return c;
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

size_t delta_tc_scratch_bytes(int BH, int T, int K) {
    return tc::carve(nullptr, BH, T, K).bytes;
}

cudaError_t delta_tc_launch(int BH, int T, int K, int V, const void *q, const void *k,
                            const void *kt, const void *v, const float *beta, const float *alpha,
                            const float *S0, void *o, float *ST, void *scratch, int *status,
                            cudaStream_t stream) {
    if (!tc::tensor_map_encoder_ready()) return cudaErrorNotSupported;
    const tc::Carve w = tc::carve(scratch, BH, T, K);
    cudaError_t e = tc::chunk_prep_launch(BH, T, K, q, k, kt, beta, alpha, w.kwn, w.qe, w.xb, w.ae,
                                          w.gk, w.gc, status, stream);
    if (e != cudaSuccess) return e;
    if (K == 128) {
        if (alpha)
            return tc::chain_launch_t<128, true>(BH, T, V, kt, v, w.kwn, w.qe, w.xb, w.ae, w.gk, w.gc, S0, o, ST, status, stream);
        return tc::chain_launch_t<128, false>(BH, T, V, kt, v, w.kwn, w.qe, w.xb, w.ae, w.gk, w.gc, S0, o, ST, status, stream);
    }
    if (alpha)
        return tc::chain_launch_t<64, true>(BH, T, V, kt, v, w.kwn, w.qe, w.xb, w.ae, w.gk, w.gc, S0, o, ST, status, stream);
    return tc::chain_launch_t<64, false>(BH, T, V, kt, v, w.kwn, w.qe, w.xb, w.ae, w.gk, w.gc, S0, o, ST, status, stream);
}

}  // namespace osdn
