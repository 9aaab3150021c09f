// phase1_scan.cu -- Phase 1 of OSDN: the O(K) preconditioner scan over the
// key stream (gist.science summary of arXiv 2605.13473, sections 2.2-2.3).
//
// Per sequence (b,h) and token t, with w_t = k_t (.) k_t, n_t = ||k_t||^2 and
// a_t = <d_t, w_t>:
//     ktilde_t = d_t (.) k_t
//     d_{t+1}  = r_t d_t + e_t w_t,   e_t = eta beta_t (1 - beta_t a_t) / n_t
// (e_t = 0 for a zero key), i.e. a descent step on the closed-form surrogate
// h_t(d) = ((1 - beta_t <d, w_t>)^2 - 1) / (2 n_t) with retention r_t.
//
// Kernel: one warp per sequence.  Lane l owns the K/32 consecutive key
// columns [l*K/32, (l+1)*K/32) of d, k and ktilde, so every token is one
// coalesced K-wide load of k and store of ktilde.  n_t and a_t are reduced
// together by a shuffle butterfly; the serial chain per token is that
// reduction plus two FMAs.  The gates of 32 tokens are fetched with one
// coalesced load and broadcast by shuffle.
#include "osdn_device.cuh"

namespace osdn {

template <int E> struct Vec;
template <> struct Vec<2> {
    template <typename T> __device__ static void ld(const T *p, float (&x)[2]) { load2(p, x); }
    template <typename T> __device__ static void st(T *p, const float (&x)[2]) { store2(p, x); }
};
template <> struct Vec<4> {
    template <typename T> __device__ static void ld(const T *p, float (&x)[4]) { load4(p, x); }
    template <typename T> __device__ static void st(T *p, const float (&x)[4]) { store4(p, x); }
};

template <typename io_t, int K>
__global__ void __launch_bounds__(128)
precond_scan_warp_kernel(int BH, int T, const io_t *__restrict__ k, const float *__restrict__ beta,
                         const float *__restrict__ r, float eta, const float *__restrict__ d0,
                         io_t *__restrict__ ktilde, float *__restrict__ dT) {
    constexpr int E = K / 32;
    const int seq = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (seq >= BH) return;

    const size_t base = (size_t)seq * T * K + (size_t)lane * E;
    const io_t *kp = k + base;
    io_t *ktp = ktilde + base;
    const float *bp = beta + (size_t)seq * T;
    const float *rp = r ? r + (size_t)seq * T : nullptr;

    float d[E];
#pragma unroll
    for (int e = 0; e < E; ++e) d[e] = d0 ? d0[(size_t)seq * K + lane * E + e] : 1.0f;

    for (int t0 = 0; t0 < T; t0 += 32) {
        const int tn = min(32, T - t0);
        const float b_l = lane < tn ? bp[t0 + lane] : 0.0f;
        const float r_l = (rp && lane < tn) ? rp[t0 + lane] : 1.0f;
#pragma unroll 4
        for (int i = 0; i < tn; ++i) {
            const size_t off = (size_t)(t0 + i) * K;
            float kv[E];
            Vec<E>::ld(kp + off, kv);
            const float bt = __shfl_sync(kFullMask, b_l, i);
            const float rt = __shfl_sync(kFullMask, r_l, i);
            float w[E], kt[E], n = 0.0f, a = 0.0f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                w[e] = kv[e] * kv[e];
                n += w[e];
                a = fmaf(d[e], w[e], a);
                kt[e] = d[e] * kv[e];
            }
            Vec<E>::st(ktp + off, kt);
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) {
                n += __shfl_xor_sync(kFullMask, n, m);
                a += __shfl_xor_sync(kFullMask, a, m);
            }
            const float et = n > 0.0f ? eta * bt * (1.0f - bt * a) / n : 0.0f;
#pragma unroll
            for (int e = 0; e < E; ++e) d[e] = fmaf(rt, d[e], et * w[e]);
        }
    }
    if (dT) {
#pragma unroll
        for (int e = 0; e < E; ++e) dT[(size_t)seq * K + lane * E + e] = d[e];
    }
}

// T == 0: the final preconditioner is the initial one.
__global__ void copy_or_fill_kernel(size_t n, const float *__restrict__ src, float fill,
                                    float *__restrict__ dst) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src ? src[i] : fill;
}

template <typename io_t, int K>
static cudaError_t launch_precond_scan_warp(int BH, int T, const void *k, const float *beta,
                                            const float *r, float eta, const float *d0,
                                            void *ktilde, float *dT, cudaStream_t stream) {
    const int threads = 128;
    const int blocks = (BH * 32 + threads - 1) / threads;
    precond_scan_warp_kernel<io_t, K><<<blocks, threads, 0, stream>>>(
        BH, T, static_cast<const io_t *>(k), beta, r, eta, d0, static_cast<io_t *>(ktilde), dT);
    return cudaGetLastError();
}

cudaError_t precond_scan_launch(int io, int BH, int T, int K, const void *k, const float *beta,
                                const float *r, float eta, const float *d0, void *ktilde,
                                float *dT, int *status, cudaStream_t stream) {
    (void)status;
    if (T == 0) {
        if (!dT) return cudaSuccess;
        size_t n = (size_t)BH * K;
        copy_or_fill_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(n, d0, 1.0f, dT);
        return cudaGetLastError();
    }
    if (io == OSDN_BF16) {
        if (K == 64)
            return launch_precond_scan_warp<__nv_bfloat16, 64>(BH, T, k, beta, r, eta, d0, ktilde, dT, stream);
        return launch_precond_scan_warp<__nv_bfloat16, 128>(BH, T, k, beta, r, eta, d0, ktilde, dT, stream);
    }
    if (K == 64)
        return launch_precond_scan_warp<float, 64>(BH, T, k, beta, r, eta, d0, ktilde, dT, stream);
    return launch_precond_scan_warp<float, 128>(BH, T, k, beta, r, eta, d0, ktilde, dT, stream);
}

cudaError_t fill_state_launch(size_t n, const float *src, float fill, float *dst,
                              cudaStream_t stream) {
    if (n == 0 || !dst) return cudaSuccess;
    unsigned blocks = (unsigned)((n + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    copy_or_fill_kernel<<<blocks, 256, 0, stream>>>(n, src, fill, dst);
    return cudaGetLastError();
}

}  // namespace osdn
