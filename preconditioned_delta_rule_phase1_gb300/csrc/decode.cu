// decode.cu -- one recurrent step (T = 1) of both OSDN phases, in place: the
// inference form of the method (gist.science summary of arXiv 2605.13473:
// section 1 on constant-memory recurrent inference, section 2.2 for the
// preconditioner step, section 2.1 for the state update).
//
// Per sequence, with w = k (.) k, n = ||k||^2, a = <d, w>:
//     ktilde = d (.) k                       (d before the step)
//     d     <- r d + eta beta (1 - beta a) w / n      (r = 1 without APF;
//                                                     the step is 0 if n = 0)
//     S     <- alpha S + beta (v - alpha S k) ktilde^T   (alpha = 1 ungated)
//     o      = S q                            (the updated state)
// Row i of S only needs its own values and the sequence's vectors, so one
// pass reads and writes every row once: with sk = <S_i, k>, sq = <S_i, q>,
//     u_i = beta (v_i - alpha sk),   S_i <- alpha S_i + u_i ktilde,
//     o_i = alpha sq + u_i <ktilde, q>.
// The step moves 8 V K bytes of state per sequence and is HBM-bound.
//
// With PCH the decay is per key channel (alpha in R^K, the Kimi Delta
// Attention backbone of section 4 read as GDN's gate made a vector): the
// row is decayed column by column, S_i <- alpha (.) S_i, before the same
// update with a scalar gate of 1.
//
// One CTA of 256 threads per sequence: every warp forms the sequence's
// scalars itself (K/32 elements a lane, warp reductions); after one block
// barrier (all warps have read d) warp 0 writes d and ktilde; the eight
// warps share the V rows, eight rows in flight per warp.
#include "osdn_device.cuh"

namespace osdn {
namespace dec {

constexpr int kThreads = 256;
constexpr int kRowsInFlight = 8;

struct Params {
    int V;
    const void *q, *k, *v;
    const float *beta, *r, *alpha;
    float eta;
    float *d, *S;
    void *o, *ktilde;
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(kFullMask, x, m);
    return x;
}

template <typename io_t, int K, bool PCH>
__global__ void __launch_bounds__(kThreads) decode_kernel(Params p) {
    constexpr int E = K / 32;   // elements of a K-vector per lane
    const int seq = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const io_t *qs = static_cast<const io_t *>(p.q) + (size_t)seq * K;
    const io_t *ks = static_cast<const io_t *>(p.k) + (size_t)seq * K;
    const io_t *vs = static_cast<const io_t *>(p.v) + (size_t)seq * p.V;
    float *ds = p.d + (size_t)seq * K;
    float *Ss = p.S + (size_t)seq * p.V * K;
    // this lane's elements: columns lane*E .. lane*E + E-1
    float kv[E], qv[E], dv[E];
#pragma unroll
    for (int e = 0; e < E; e += 2) {
        float t[2];
        load2(ks + lane * E + e, t);
        kv[e] = t[0];
        kv[e + 1] = t[1];
        load2(qs + lane * E + e, t);
        qv[e] = t[0];
        qv[e + 1] = t[1];
        load2(ds + lane * E + e, t);
        dv[e] = t[0];
        dv[e + 1] = t[1];
    }
    const float beta = p.beta[seq];
    const float r = p.r ? p.r[seq] : 1.0f;
    const float alpha = (!PCH && p.alpha) ? p.alpha[seq] : 1.0f;
    float av[E];   // the per-channel decay of this lane's columns
#pragma unroll
    for (int e = 0; e < E; ++e) av[e] = 1.0f;
    if constexpr (PCH) {
        if (p.alpha) {
#pragma unroll
            for (int e = 0; e < E; e += 2) {
                float t[2];
                load2(p.alpha + (size_t)seq * K + lane * E + e, t);
                av[e] = t[0];
                av[e + 1] = t[1];
            }
        }
    }
    float n = 0.f, a = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float w = kv[e] * kv[e];
        n = fmaf(kv[e], kv[e], n);
        a = fmaf(dv[e], w, a);
    }
    n = warp_sum(n);
    a = warp_sum(a);
    const float coef = n > 0.0f ? p.eta * beta * (1.0f - beta * a) / n : 0.0f;
    float kt[E], kq = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        kt[e] = dv[e] * kv[e];
        kq = fmaf(kt[e], qv[e], kq);
    }
    kq = warp_sum(kq);
    __syncthreads();   // every warp has read d before warp 0 overwrites it
    if (warp == 0) {
        float dn[E];
#pragma unroll
        for (int e = 0; e < E; ++e) dn[e] = fmaf(r, dv[e], coef * (kv[e] * kv[e]));
#pragma unroll
        for (int e = 0; e < E; e += 2) {
            const float x2[2] = {dn[e], dn[e + 1]};
            store2(ds + lane * E + e, x2);
            if (p.ktilde) {
                const float k2[2] = {kt[e], kt[e + 1]};
                store2(static_cast<io_t *>(p.ktilde) + (size_t)seq * K + lane * E + e, k2);
            }
        }
    }
    // rows of S: warp w takes rows w, w + 8, ...; kRowsInFlight at a time
    for (int i0 = warp * kRowsInFlight; i0 < p.V; i0 += (kThreads / 32) * kRowsInFlight) {
        float sv[kRowsInFlight][E];
#pragma unroll
        for (int rr = 0; rr < kRowsInFlight; ++rr) {
            const int i = i0 + rr;
#pragma unroll
            for (int e = 0; e < E; e += 2) {
                float t[2] = {0.f, 0.f};
                if (i < p.V) load2(Ss + (size_t)i * K + lane * E + e, t);
                sv[rr][e] = t[0];
                sv[rr][e + 1] = t[1];
            }
            if constexpr (PCH) {
#pragma unroll
                for (int e = 0; e < E; ++e) sv[rr][e] *= av[e];
            }
        }
#pragma unroll
        for (int rr = 0; rr < kRowsInFlight; ++rr) {
            const int i = i0 + rr;
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                sk = fmaf(sv[rr][e], kv[e], sk);
                sq = fmaf(sv[rr][e], qv[e], sq);
            }
            sk = warp_sum(sk);
            sq = warp_sum(sq);
            if (i < p.V) {
                const float vi = to_f32(vs[i]);
                const float u = beta * (vi - alpha * sk);
#pragma unroll
                for (int e = 0; e < E; e += 2) {
                    const float x2[2] = {fmaf(alpha, sv[rr][e], u * kt[e]),
                                         fmaf(alpha, sv[rr][e + 1], u * kt[e + 1])};
                    store2(Ss + (size_t)i * K + lane * E + e, x2);
                }
                if (lane == 0) {
                    io_t *os = static_cast<io_t *>(p.o) + (size_t)seq * p.V;
                    from_f32(os[i], fmaf(alpha, sq, u * kq));
                }
            }
        }
    }
}

template <typename io_t, int K, bool PCH = false>
cudaError_t launch_t(int BH, const Params &p, cudaStream_t stream) {
    decode_kernel<io_t, K, PCH><<<BH, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dec

cudaError_t decode_step_launch(int io, int BH, int K, int V, const void *q, const void *k,
                               const void *v, const float *beta, const float *r, float eta,
                               const float *alpha, float *d, float *S, void *o, void *ktilde,
                               cudaStream_t stream) {
    dec::Params p;
    p.V = V;
    p.q = q;
    p.k = k;
    p.v = v;
    p.beta = beta;
    p.r = r;
    p.alpha = alpha;
    p.eta = eta;
    p.d = d;
    p.S = S;
    p.o = o;
    p.ktilde = ktilde;
    if (io == OSDN_BF16)
        return K == 64 ? dec::launch_t<__nv_bfloat16, 64>(BH, p, stream)
                       : dec::launch_t<__nv_bfloat16, 128>(BH, p, stream);
    return K == 64 ? dec::launch_t<float, 64>(BH, p, stream) : dec::launch_t<float, 128>(BH, p, stream);
}

// The same step with a decay per key channel, alpha_k [BH][K] (NULL: none).
cudaError_t decode_step_kda_launch(int io, int BH, int K, int V, const void *q, const void *k,
                                   const void *v, const float *beta, const float *r, float eta,
                                   const float *alpha_k, float *d, float *S, void *o,
                                   void *ktilde, cudaStream_t stream) {
    dec::Params p;
    p.V = V;
    p.q = q;
    p.k = k;
    p.v = v;
    p.beta = beta;
    p.r = r;
    p.alpha = alpha_k;
    p.eta = eta;
    p.d = d;
    p.S = S;
    p.o = o;
    p.ktilde = ktilde;
    if (io == OSDN_BF16)
        return K == 64 ? dec::launch_t<__nv_bfloat16, 64, true>(BH, p, stream)
                       : dec::launch_t<__nv_bfloat16, 128, true>(BH, p, stream);
    return K == 64 ? dec::launch_t<float, 64, true>(BH, p, stream)
                   : dec::launch_t<float, 128, true>(BH, p, stream);
}

}  // namespace osdn
