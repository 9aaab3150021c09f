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
// (ktilde_t = d (.) k_t, d <- r_t d + e_t w_t).  The chain from one chunk to
// the next is one K-wide reduction (p), the 16-step substitution and the
// column updates.  G only enters through the small coupling c beta G, so it
// is formed on the tensor cores (mma.sync, tf32 inputs, fp32 accumulation);
// p and n, which enter e directly, are reduced in fp32.
//
// Time segments.  With a retention gate the map d -> d_{t+1} contracts, so a
// segment can start from a state estimated by running the scan over the W
// tokens before it from d = 0 ("warm-up").  Every segment records its
// estimated start and its end state; a second kernel checks each start
// against the predecessor's end (exact by induction from d_0) and recomputes
// any segment whose estimate is off by more than 2^-21 relative, or all
// segments after a token whose one-step map could expand (||A_t||_2 > 1).
// The result is therefore the exact recurrence to fp32 rounding on every
// input; speculation only decides how much runs in parallel.
#include <mutex>

#include "osdn_device.cuh"

namespace osdn {
namespace p1 {

constexpr int C = 16;          // tokens per chunk
constexpr int NSTAGE = 4;      // key chunks in flight
constexpr int kWarm = 128;     // warm-up tokens in front of a speculative segment
constexpr float kRelTol = 4.76837158203125e-07f;  // 2^-21

template <typename io_t, int K>
struct Smem {
    static constexpr int NW = K / 32;
    io_t keys[NSTAGE][C][K];
    alignas(16) float gb[NSTAGE][C];      // beta of the staged chunk
    alignas(16) float gr[NSTAGE][C];      // r of the staged chunk
    float wS[C][K + 4];                   // w = k^2 for the Gram fragments
    float gpart[NW][C][C + 4];            // per-warp partial Gram (16-byte aligned rows)
    float part[NW][2 * C];                // per-warp partial p (0..15) and n (16..31)
    alignas(16) float sE[C];
    alignas(16) float sR[C];
    float red[NW][2];
    int flag;
};

struct Params {
    int BH, T, L, nseg;
    const void *k;
    const float *beta, *r, *d0;
    float eta;
    void *ktilde;
    float *dT;
    float *ws_start, *ws_end;   // [BH][nseg][K]
    int *ws_flag;               // [BH][nseg]
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
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t to_tf32(float x) {
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

// Scan tokens [tb, te) of sequence `seq` starting from the state in `d`
// (this thread's column); ktilde is written for tokens >= te_emit0.  Returns
// the state after te in `d`.  Sets sm.flag if some token's one-step map
// could expand.  All K threads of the CTA call this together.
template <typename io_t, int K>
__device__ void scan_range(const Params &p, Smem<io_t, K> &sm, int seq, int tb, int tseg, int te,
                           float &d) {
    constexpr int NW = K / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const io_t *kseq = static_cast<const io_t *>(p.k) + (size_t)seq * p.T * K;
    io_t *ktseq = static_cast<io_t *>(p.ktilde) + (size_t)seq * p.T * K;
    const float *bseq = p.beta + (size_t)seq * p.T;
    const float *rseq = p.r ? p.r + (size_t)seq * p.T : nullptr;
    const int nc = (te - tb + C - 1) / C;

    auto issue = [&](int j) {
        if (j < nc) {
            const int s = j % NSTAGE, t0 = tb + j * C;
            constexpr int PER_ROW = K * (int)sizeof(io_t) / 16;   // 16-byte pieces per key row
            for (int i = tid; i < C * PER_ROW; i += K) {
                const int t = i / PER_ROW, pc = i % PER_ROW;
                const bool valid = t0 + t < te;
                const io_t *src = valid ? kseq + (size_t)(t0 + t) * K + pc * (16 / sizeof(io_t)) : kseq;
                cp_async16(&sm.keys[s][t][pc * (16 / sizeof(io_t))], src, valid);
            }
            if (tid < C) {
                const bool valid = t0 + tid < te;
                cp_async4(&sm.gb[s][tid], valid ? bseq + t0 + tid : bseq, valid);
            } else if (tid < 2 * C && rseq) {
                const int t = tid - C;
                const bool valid = t0 + t < te;
                cp_async4(&sm.gr[s][t], valid ? rseq + t0 + t : rseq, valid);
            }
        }
        cp_commit();
    };
#pragma unroll
    for (int j = 0; j < NSTAGE - 1; ++j) issue(j);

    for (int j = 0; j < nc; ++j) {
        issue(j + NSTAGE - 1);
        cp_wait<NSTAGE - 1>();
        __syncthreads();
        const int s = j % NSTAGE, t0 = tb + j * C;
        const int nv = min(C, te - t0);

        // ---- 1. this column of the chunk; p and n partials ---------------------
        float kv[C], w[C];
#pragma unroll
        for (int t = 0; t < C; ++t) {
            kv[t] = to_f32(sm.keys[s][t][tid]);
            w[t] = kv[t] * kv[t];
            sm.wS[t][tid] = w[t];
        }
        {
            // transpose-reduce 32 partials across the warp: lane l ends with index l
            float v[2 * C];
#pragma unroll
            for (int t = 0; t < C; ++t) {
                v[t] = d * w[t];
                v[C + t] = w[t];
            }
#pragma unroll
            for (int off = 16, n = 16; off >= 1; off >>= 1, n >>= 1) {
                const bool hi = (lane & off) != 0;
#pragma unroll
                for (int i = 0; i < n; ++i) {
                    const float keep = hi ? v[i + n] : v[i];
                    const float send = hi ? v[i] : v[i + n];
                    v[i] = keep + __shfl_xor_sync(kFullMask, send, off);
                }
            }
            sm.part[warp][lane] = v[0];
        }
        __syncthreads();

        // ---- 2. partial Gram of this warp's 32 key columns (tensor cores) -------
        {
            const int g = lane >> 2, tq = lane & 3;
            float acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const int k0 = warp * 32 + ks * 8;
                uint32_t a[4];
                a[0] = to_tf32(sm.wS[g][k0 + tq]);
                a[1] = to_tf32(sm.wS[g + 8][k0 + tq]);
                a[2] = to_tf32(sm.wS[g][k0 + tq + 4]);
                a[3] = to_tf32(sm.wS[g + 8][k0 + tq + 4]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const uint32_t b0 = to_tf32(sm.wS[8 * nt + g][k0 + tq]);
                    const uint32_t b1 = to_tf32(sm.wS[8 * nt + g][k0 + tq + 4]);
                    mma_tf32(acc[nt], a, b0, b1);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                sm.gpart[warp][g][8 * nt + 2 * tq] = acc[nt][0];
                sm.gpart[warp][g][8 * nt + 2 * tq + 1] = acc[nt][1];
                sm.gpart[warp][g + 8][8 * nt + 2 * tq] = acc[nt][2];
                sm.gpart[warp][g + 8][8 * nt + 2 * tq + 1] = acc[nt][3];
            }
        }
        __syncthreads();

        // ---- 3. the 16 coefficients e_t (warp 0, lane t) -------------------------
        if (warp == 0) {
            const int t = lane & (C - 1);
            float pt = 0.f, nt_ = 0.f;
#pragma unroll
            for (int ww = 0; ww < NW; ++ww) {
                pt += sm.part[ww][t];
                nt_ += sm.part[ww][C + t];
            }
            // row t of the Gram and the chunk's r, all loaded before the chains below
            float g[C], rr[C];
#pragma unroll
            for (int u = 0; u < C; u += 4) {
                float4 acc4 = *reinterpret_cast<const float4 *>(&sm.gpart[0][t][u]);
#pragma unroll
                for (int ww = 1; ww < NW; ++ww) {
                    const float4 x = *reinterpret_cast<const float4 *>(&sm.gpart[ww][t][u]);
                    acc4.x += x.x; acc4.y += x.y; acc4.z += x.z; acc4.w += x.w;
                }
                g[u] = acc4.x; g[u + 1] = acc4.y; g[u + 2] = acc4.z; g[u + 3] = acc4.w;
                if (rseq) {
                    const float4 r4 = *reinterpret_cast<const float4 *>(&sm.gr[s][u]);
                    rr[u] = r4.x; rr[u + 1] = r4.y; rr[u + 2] = r4.z; rr[u + 3] = r4.w;
                } else {
                    rr[u] = rr[u + 1] = rr[u + 2] = rr[u + 3] = 1.0f;
                }
            }
            const float bt = sm.gb[s][t];
            float rt = 1.0f, gtt = 0.0f;
#pragma unroll
            for (int u = 0; u < C; ++u) {
                if (u == t) {
                    rt = rr[u];
                    gtt = g[u];
                }
            }
            const float ct = nt_ > 0.0f ? p.eta * bt / nt_ : 0.0f;
            // coupling row t: coef_u = c_t beta_t pi_ut G_tu (u < t); rho_t
            float coef[C];
            float pi = 1.0f;
#pragma unroll
            for (int u = C - 1; u >= 0; --u) {
                coef[u] = (u < t) ? ct * bt * pi * g[u] : 0.0f;
                if (u < t) pi *= rr[u];
            }
            const float rho = pi;  // prod_{v < t} r_v
            // can this token's one-step map expand?  ||A_t|| = max(|r|, |r - lambda|)
            {
                const float lam = nt_ > 0.0f ? p.eta * bt * bt * gtt / nt_ : 0.0f;
                const float nrm = fmaxf(fabsf(rt), fabsf(rt - lam));
                if (lane < C && t < nv && nrm > 1.0f + 1e-6f) sm.flag = 1;
            }
            float acc = ct * (1.0f - bt * rho * pt);
#pragma unroll
            for (int u = 0; u < C; ++u) {
                const float eu = __shfl_sync(kFullMask, acc, u);
                if (t > u) acc = fmaf(-coef[u], eu, acc);
            }
            if (lane < C) {
                sm.sE[t] = t < nv ? acc : 0.0f;
                sm.sR[t] = rt;
            }
        }
        __syncthreads();

        // ---- 4. this column through the chunk; emit ktilde ----------------------
        const bool emit = t0 >= tseg;
        // the chunk's e and r in registers first: the ktilde stores below go
        // through a generic pointer and would otherwise order every later load
        float eR[C], rR[C];
#pragma unroll
        for (int t = 0; t < C; t += 4) {
            const float4 e4 = *reinterpret_cast<const float4 *>(&sm.sE[t]);
            const float4 r4 = *reinterpret_cast<const float4 *>(&sm.sR[t]);
            eR[t] = e4.x; eR[t + 1] = e4.y; eR[t + 2] = e4.z; eR[t + 3] = e4.w;
            rR[t] = r4.x; rR[t + 1] = r4.y; rR[t + 2] = r4.z; rR[t + 3] = r4.w;
        }
#pragma unroll
        for (int t = 0; t < C; ++t) {
            if (t < nv) {
                if (emit) from_f32(ktseq[(size_t)(t0 + t) * K + tid], d * kv[t]);
                d = fmaf(rR[t], d, eR[t] * w[t]);
            }
        }
    }
    cp_wait<0>();
    __syncthreads();
}

// Grid (nseg, BH): segment `seg` of sequence `seq`.
template <typename io_t, int K>
__global__ void __launch_bounds__(K) precond_segment_kernel(Params p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Smem<io_t, K> &sm = *reinterpret_cast<Smem<io_t, K> *>(smem_raw);
    const int seg = blockIdx.x, seq = blockIdx.y, tid = threadIdx.x;
    if (tid == 0) sm.flag = 0;
    const int tseg = seg * p.L;
    const int te = min(p.T, tseg + p.L);
    float d;
    int tb;
    if (seg == 0) {
        d = p.d0 ? p.d0[(size_t)seq * K + tid] : 1.0f;
        tb = 0;
    } else {
        d = 0.0f;  // speculative: the warm-up forgets this guess
        tb = tseg - kWarm;
    }
    __syncthreads();
    if (seg > 0) {
        scan_range<io_t, K>(p, sm, seq, tb, tseg, tseg, d);  // warm-up, nothing emitted
    }
    if (p.nseg > 1) p.ws_start[((size_t)seq * p.nseg + seg) * K + tid] = d;
    scan_range<io_t, K>(p, sm, seq, tseg, tseg, te, d);
    if (p.nseg > 1) {
        p.ws_end[((size_t)seq * p.nseg + seg) * K + tid] = d;
        if (tid == 0) p.ws_flag[(size_t)seq * p.nseg + seg] = sm.flag;
    } else if (p.dT) {
        p.dT[(size_t)seq * K + tid] = d;
    }
}

// Grid (BH): verify every speculative segment start against its predecessor's
// end; recompute (exactly) the segments that do not match; write d_T.
// Without a repair every boundary check is independent (the predecessor's
// end is then exact), so all boundaries are checked at once first; the
// sequential check-and-repair walk starts at the first boundary that fails.
template <typename io_t, int K>
__global__ void __launch_bounds__(K) precond_verify_kernel(Params p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Smem<io_t, K> &sm = *reinterpret_cast<Smem<io_t, K> *>(smem_raw);
    constexpr int NW = K / 32;
    constexpr int kBatch = 64;   // boundaries checked per pass
    const int seq = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t base = (size_t)seq * p.nseg;
    __shared__ int any_flag, first_bad;
    __shared__ float sDiff[NW][kBatch], sMag[NW][kBatch];
    if (tid == 0) {
        int f = 0;
        for (int i = 0; i < p.nseg; ++i) f |= p.ws_flag[base + i];
        any_flag = f;
        first_bad = f ? 1 : p.nseg;
        sm.flag = 0;
    }
    __syncthreads();
    // ---- all boundaries in parallel: segment i starts where i-1 ended?
    for (int b0 = 1; b0 < p.nseg && !any_flag; b0 += kBatch) {
        const int nb = min(kBatch, p.nseg - b0);
#pragma unroll 4
        for (int q = 0; q < nb; ++q) {
            const int i = b0 + q;
            const float st = p.ws_start[(base + i) * K + tid];
            float diff = fabsf(p.ws_end[(base + i - 1) * K + tid] - st), mag = fabsf(st);
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) {
                diff = fmaxf(diff, __shfl_xor_sync(kFullMask, diff, m));
                mag = fmaxf(mag, __shfl_xor_sync(kFullMask, mag, m));
            }
            if (lane == 0) {
                sDiff[warp][q] = diff;
                sMag[warp][q] = mag;
            }
        }
        __syncthreads();
        if (tid < nb) {
            float dmax = 0.f, mmax = 0.f;
#pragma unroll
            for (int ww = 0; ww < NW; ++ww) {
                dmax = fmaxf(dmax, sDiff[ww][tid]);
                mmax = fmaxf(mmax, sMag[ww][tid]);
            }
            if (!(dmax <= kRelTol * mmax)) atomicMin(&first_bad, b0 + tid);
        }
        __syncthreads();
        if (first_bad < p.nseg) break;
    }
    const bool all_suspect = any_flag != 0;
    const int start = first_bad;
    // ---- sequential walk from the first failing boundary (rare)
    float prev_end = p.ws_end[(base + start - 1) * K + tid];
    for (int i = start; i < p.nseg; ++i) {
        const float st = p.ws_start[(base + i) * K + tid];
        float diff = fabsf(prev_end - st), mag = fabsf(st);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            diff = fmaxf(diff, __shfl_xor_sync(kFullMask, diff, m));
            mag = fmaxf(mag, __shfl_xor_sync(kFullMask, mag, m));
        }
        if (lane == 0) {
            sm.red[warp][0] = diff;
            sm.red[warp][1] = mag;
        }
        __syncthreads();
        float dmax = 0.f, mmax = 0.f;
#pragma unroll
        for (int ww = 0; ww < NW; ++ww) {
            dmax = fmaxf(dmax, sm.red[ww][0]);
            mmax = fmaxf(mmax, sm.red[ww][1]);
        }
        __syncthreads();
        const bool ok = !all_suspect && dmax <= kRelTol * mmax;
        float d = p.ws_end[(base + i) * K + tid];
        if (!ok) {  // recompute segment i from the exact end of segment i-1
            d = prev_end;
            const int tseg = i * p.L, te = min(p.T, tseg + p.L);
            scan_range<io_t, K>(p, sm, seq, tseg, tseg, te, d);
            p.ws_end[(base + i) * K + tid] = d;
        }
        prev_end = d;
    }
    if (p.dT) p.dT[(size_t)seq * K + tid] = prev_end;
}

// T == 0: the final preconditioner is the initial one.
__global__ void copy_or_fill_kernel(size_t n, const float *__restrict__ src, float fill,
                                    float *__restrict__ dst) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src ? src[i] : fill;
}

template <typename io_t, int K>
static cudaError_t launch(const Params &p, cudaStream_t stream) {
    const int smem = (int)sizeof(Smem<io_t, K>);
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(precond_segment_kernel<io_t, K>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(precond_verify_kernel<io_t, K>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    precond_segment_kernel<io_t, K><<<dim3(p.nseg, p.BH), K, smem, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.nseg == 1) return e;
    precond_verify_kernel<io_t, K><<<p.BH, K, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace p1

// Segment length: long enough that the warm-up costs little extra reading,
// short enough to give the GPU a few waves of CTAs.  Only a retention gate
// (r != NULL) makes the warm-up converge, so without one there is a single
// segment per sequence.
int precond_segments(int BH, int T, bool has_r, int *L_out) {
    int L = T;
    if (has_r && T > 2 * p1::kWarm) {
        L = 1024;
        if ((long long)BH * ((T + L - 1) / L) < 4LL * 152) L = 512;
        if (L >= T) L = T;
    }
    if (L < 1) L = 1;
    if (L_out) *L_out = L;
    return (T + L - 1) / L;
}

size_t precond_scratch_bytes(int BH, int T, int K) {
    int L;
    const int nseg = precond_segments(BH, T, true, &L);
    if (nseg <= 1) return 0;
    const size_t n = (size_t)BH * nseg;
    return n * K * 4 * 2 + ((n * 4 + 255) / 256) * 256;
}

cudaError_t precond_scan_launch(int io, int BH, int T, int K, const void *k, const float *beta,
                                const float *r, float eta, const float *d0, void *ktilde,
                                float *dT, void *scratch, int *status, cudaStream_t stream) {
    if (T == 0) {
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
    p.status = status;
    float *f = static_cast<float *>(scratch);
    const size_t n = (size_t)BH * p.nseg;
    p.ws_start = p.nseg > 1 ? f : nullptr;
    p.ws_end = p.nseg > 1 ? f + n * K : nullptr;
    p.ws_flag = p.nseg > 1 ? reinterpret_cast<int *>(f + 2 * n * K) : nullptr;
    if (io == OSDN_BF16)
        return K == 64 ? p1::launch<__nv_bfloat16, 64>(p, stream)
                       : p1::launch<__nv_bfloat16, 128>(p, stream);
    return K == 64 ? p1::launch<float, 64>(p, stream) : p1::launch<float, 128>(p, stream);
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
    return precond_scan_launch(io, BH, T, K, k, beta, r, eta, d0, ktilde, dT, scratch, nullptr,
                               stream);
}

// Bytes of scratch the scan needs for this call (0 without a retention gate).
size_t precond_scratch_bytes_for(int BH, int T, int K, bool has_r) {
    int L;
    const int nseg = precond_segments(BH, T, has_r, &L);
    if (nseg <= 1 || T == 0) return 0;
    const size_t n = (size_t)BH * nseg;
    return n * K * 4 * 2 + ((n * 4 + 255) / 256) * 256;
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
