// phase2_simt.cu -- Phase 2 of OSDN in fp32 FFMA: the delta-rule recurrence
// with preconditioned keys (gist.science summary of arXiv 2605.13473,
// section 2.1), for fp32 I/O, where tensor-core operand rounding would not
// meet fp32 accuracy, and for the per-channel decay (both I/O types).
//
//     S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) ktilde_t^T
//     o_t = S_t q_t
//
// With PCH (a decay per key channel, the Kimi-Delta-Attention-style backbone
// of section 4) alpha_t is a K-vector that scales the key columns of S:
//
//     S_t = S_{t-1} Diag(alpha_t) + beta_t (v_t - S_{t-1} Diag(alpha_t) k_t) ktilde_t^T
//
// The rows of S evolve independently (row i only sees v_t[i]), so the grid is
// one CTA per (sequence, slice of 32 value rows).  Four threads share a row:
// thread p of the group holds the key columns j = p + 4m, so the broadcast
// reads of k, ktilde and q from shared memory are conflict-free and the two
// row dot products per token reduce with two shuffles.  Tokens are staged
// through shared memory 16 at a time with coalesced loads.
#include "osdn_device.cuh"

namespace osdn {

constexpr int kRows = 32;   // value rows per CTA
constexpr int kStage = 16;  // tokens staged per pass (static smem stays < 48 KB)

template <typename io_t, int K, bool PCH>
__global__ void __launch_bounds__(128)
delta_simt_kernel(int BH, int T, int V, const io_t *__restrict__ q, const io_t *__restrict__ k,
                  const io_t *__restrict__ ktilde, const io_t *__restrict__ v,
                  const float *__restrict__ beta, const float *__restrict__ alpha,
                  const float *__restrict__ S0, io_t *__restrict__ o, float *__restrict__ ST) {
    constexpr int KP = K / 4;
    __shared__ __align__(16) float ks[kStage][K];
    __shared__ __align__(16) float kts[kStage][K];
    __shared__ __align__(16) float qs[kStage][K];
    __shared__ __align__(16) float aks[PCH ? kStage : 1][PCH ? K : 4];   // per-channel decay
    __shared__ float vs[kStage][kRows];
    __shared__ float os[kStage][kRows];
    __shared__ float bs[kStage], as[kStage];

    const int tid = threadIdx.x;
    const int row = tid >> 2, p = tid & 3;
    const int row0 = blockIdx.x * kRows;
    const size_t seq = grid_seq();
    if (seq >= (size_t)BH) return;
    const size_t kbase = seq * (size_t)T * K, vbase = seq * (size_t)T * V;

    float S[KP];
    {
        const float *s0 = S0 ? S0 + (seq * V + row0 + row) * (size_t)K : nullptr;
#pragma unroll
        for (int m = 0; m < KP; ++m) S[m] = s0 ? s0[p + 4 * m] : 0.0f;
    }

    // The next group of tokens is loaded into registers while the current one
    // is computed, and written to shared memory at the top of the next pass.
    constexpr int NKV = kStage * K / (128 * 4);      // float4 pieces of each key tile a thread loads
    constexpr int NVV = kStage * kRows / 128;         // values a thread loads
    float rk[NKV][4], rkt[NKV][4], rq[NKV][4], rak[PCH ? NKV : 1][4], rv[NVV];
    float rb = 0.0f, ra = 1.0f;
    auto fetch = [&](int t0) {   // tokens t0 .. t0 + kStage - 1 (zero past T; decay 1)
        const int tn = min(kStage, T - t0);
#pragma unroll
        for (int n = 0; n < NKV; ++n) {
            const int idx = tid * 4 + n * 128 * 4;
            const int tt = idx / K, j = idx % K;
#pragma unroll
            for (int e = 0; e < 4; ++e) rk[n][e] = rkt[n][e] = rq[n][e] = 0.0f;
            if (tt < tn) {
                const size_t g = kbase + (size_t)(t0 + tt) * K + j;
                load4(k + g, rk[n]);
                load4(ktilde + g, rkt[n]);
                load4(q + g, rq[n]);
            }
            if constexpr (PCH) {
#pragma unroll
                for (int e = 0; e < 4; ++e) rak[n][e] = 1.0f;
                if (alpha && tt < tn) load4(alpha + kbase + (size_t)(t0 + tt) * K + j, rak[n]);
            }
        }
#pragma unroll
        for (int n = 0; n < NVV; ++n) {
            const int idx = tid + n * 128;
            const int tt = idx / kRows, i = idx % kRows;
            rv[n] = tt < tn ? to_f32(v[vbase + (size_t)(t0 + tt) * V + row0 + i]) : 0.0f;
        }
        if (tid < kStage) {
            rb = tid < tn ? beta[seq * T + t0 + tid] : 0.0f;
            ra = (!PCH && alpha && tid < tn) ? alpha[seq * T + t0 + tid] : 1.0f;
        }
    };
    fetch(0);
    for (int t0 = 0; t0 < T; t0 += kStage) {
        const int tn = min(kStage, T - t0);
        // stage k, ktilde, q (fp32 in shared memory), the value slice and the gates
#pragma unroll
        for (int n = 0; n < NKV; ++n) {
            const int idx = tid * 4 + n * 128 * 4;
            const int tt = idx / K, j = idx % K;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                ks[tt][j + e] = rk[n][e];
                kts[tt][j + e] = rkt[n][e];
                qs[tt][j + e] = rq[n][e];
            }
            if constexpr (PCH) {
#pragma unroll
                for (int e = 0; e < 4; ++e) aks[tt][j + e] = rak[n][e];
            }
        }
#pragma unroll
        for (int n = 0; n < NVV; ++n) {
            const int idx = tid + n * 128;
            vs[idx / kRows][idx % kRows] = rv[n];
        }
        if (tid < kStage) {
            bs[tid] = rb;
            as[tid] = ra;
        }
        __syncthreads();
        if (t0 + kStage < T) fetch(t0 + kStage);   // in flight during this group's tokens

        for (int tt = 0; tt < tn; ++tt) {
            if constexpr (PCH) {   // decay the key columns first; the scalar gate below is 1
#pragma unroll
                for (int m = 0; m < KP; ++m) S[m] *= aks[tt][p + 4 * m];
            }
            float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
            for (int m = 0; m < KP; m += 4) {
                p0 = fmaf(S[m + 0], ks[tt][p + 4 * (m + 0)], p0);
                p1 = fmaf(S[m + 1], ks[tt][p + 4 * (m + 1)], p1);
                p2 = fmaf(S[m + 2], ks[tt][p + 4 * (m + 2)], p2);
                p3 = fmaf(S[m + 3], ks[tt][p + 4 * (m + 3)], p3);
            }
            float pred = (p0 + p1) + (p2 + p3);
            pred += __shfl_xor_sync(kFullMask, pred, 1);
            pred += __shfl_xor_sync(kFullMask, pred, 2);
            const float at = as[tt];
            const float u = bs[tt] * (vs[tt][row] - at * pred);
            float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
            for (int m = 0; m < KP; m += 4) {
                S[m + 0] = fmaf(at, S[m + 0], u * kts[tt][p + 4 * (m + 0)]);
                S[m + 1] = fmaf(at, S[m + 1], u * kts[tt][p + 4 * (m + 1)]);
                S[m + 2] = fmaf(at, S[m + 2], u * kts[tt][p + 4 * (m + 2)]);
                S[m + 3] = fmaf(at, S[m + 3], u * kts[tt][p + 4 * (m + 3)]);
                o0 = fmaf(S[m + 0], qs[tt][p + 4 * (m + 0)], o0);
                o1 = fmaf(S[m + 1], qs[tt][p + 4 * (m + 1)], o1);
                o2 = fmaf(S[m + 2], qs[tt][p + 4 * (m + 2)], o2);
                o3 = fmaf(S[m + 3], qs[tt][p + 4 * (m + 3)], o3);
            }
            float out = (o0 + o1) + (o2 + o3);
            out += __shfl_xor_sync(kFullMask, out, 1);
            out += __shfl_xor_sync(kFullMask, out, 2);
            if (p == 0) os[tt][row] = out;
        }
        __syncthreads();
        for (int idx = tid; idx < tn * kRows; idx += 128) {
            const int tt = idx / kRows, i = idx % kRows;
            from_f32(o[vbase + (size_t)(t0 + tt) * V + row0 + i], os[tt][i]);
        }
        // the next stage overwrites vs/os only after this barrier
        __syncthreads();
    }
    if (ST) {
        float *st = ST + (seq * V + row0 + row) * (size_t)K;
#pragma unroll
        for (int m = 0; m < KP; ++m) st[p + 4 * m] = S[m];
    }
}

template <typename io_t, int K, bool PCH = false>
static cudaError_t launch_delta_simt(int BH, int T, int V, const void *q, const void *k,
                                     const void *kt, const void *v, const float *beta,
                                     const float *alpha, const float *S0, void *o, float *ST,
                                     cudaStream_t stream) {
    const dim3 grid = seq_grid(V / kRows, BH);
    delta_simt_kernel<io_t, K, PCH><<<grid, 128, 0, stream>>>(
        BH, T, V, static_cast<const io_t *>(q), static_cast<const io_t *>(k),
        static_cast<const io_t *>(kt), static_cast<const io_t *>(v), beta, alpha, S0,
        static_cast<io_t *>(o), ST);
    return cudaGetLastError();
}

cudaError_t delta_simt_launch(int io, int BH, int T, int K, int V, const void *q, const void *k,
                              const void *kt, const void *v, const float *beta,
                              const float *alpha, const float *S0, void *o, float *ST,
                              cudaStream_t stream) {
    if (io == OSDN_BF16) {
        if (K == 64)
            return launch_delta_simt<__nv_bfloat16, 64>(BH, T, V, q, k, kt, v, beta, alpha, S0, o, ST, stream);
        return launch_delta_simt<__nv_bfloat16, 128>(BH, T, V, q, k, kt, v, beta, alpha, S0, o, ST, stream);
    }
    if (K == 64)
        return launch_delta_simt<float, 64>(BH, T, V, q, k, kt, v, beta, alpha, S0, o, ST, stream);
    return launch_delta_simt<float, 128>(BH, T, V, q, k, kt, v, beta, alpha, S0, o, ST, stream);
}

// Phase 2 with a per-channel decay alpha_k [BH][T][K] (NULL: no decay).
cudaError_t delta_simt_kda_launch(int io, int BH, int T, int K, int V, const void *q,
                                  const void *k, const void *kt, const void *v,
                                  const float *beta, const float *alpha_k, const float *S0,
                                  void *o, float *ST, cudaStream_t stream) {
    if (io == OSDN_BF16) {
        if (K == 64)
            return launch_delta_simt<__nv_bfloat16, 64, true>(BH, T, V, q, k, kt, v, beta, alpha_k, S0, o, ST, stream);
        return launch_delta_simt<__nv_bfloat16, 128, true>(BH, T, V, q, k, kt, v, beta, alpha_k, S0, o, ST, stream);
    }
    if (K == 64)
        return launch_delta_simt<float, 64, true>(BH, T, V, q, k, kt, v, beta, alpha_k, S0, o, ST, stream);
    return launch_delta_simt<float, 128, true>(BH, T, V, q, k, kt, v, beta, alpha_k, S0, o, ST, stream);
}

}  // namespace osdn
