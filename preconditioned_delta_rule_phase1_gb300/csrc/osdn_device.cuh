// osdn_device.cuh -- device-side helpers shared by the OSDN kernels:
// element loads/stores for the two I/O types and the sticky status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "osdn.h"

namespace osdn {

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) for `func`, once per
// device: the attribute belongs to a device's context, so every device the
// process launches on needs its own call.  `done` holds one bit per device
// (devices past 63 set it on every call).
inline cudaError_t smem_attr_once(const void *func, int bytes,
                                  std::atomic<unsigned long long> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

constexpr unsigned kFullMask = 0xffffffffu;

// Sequences are spread over grid y and z (y fastest), so that B*H is not
// bounded by the 65,535 limit of a single grid dimension: seq_grid(x, BH, w)
// covers BH sequences with w extra z-slices per sequence group, grid_seq()
// recovers a CTA's sequence (CTAs past BH leave at once).
constexpr unsigned kGridYMax = 65535;
inline dim3 seq_grid(unsigned x, size_t BH, unsigned zmul = 1) {
    const unsigned y = (unsigned)(BH < kGridYMax ? BH : kGridYMax);
    const unsigned nz = (unsigned)((BH + y - 1) / y);
    return dim3(x, y, nz * zmul);
}
__device__ __forceinline__ size_t grid_seq(unsigned nz = 0) {
    // nz: the sequence groups (gridDim.z without further z-slices when 0)
    const unsigned z = nz ? blockIdx.z % nz : blockIdx.z;
    return blockIdx.y + (size_t)gridDim.y * z;
}

// Record the first problem a kernel meets in the workspace status word and
// keep it: later reports never overwrite an earlier one.
__device__ __forceinline__ void report_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Four consecutive elements at p (16-byte aligned for f32, 8 for bf16).
__device__ __forceinline__ void load4(const float *p, float (&x)[4]) {
    float4 v = *reinterpret_cast<const float4 *>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float (&x)[4]) {
    uint2 u = *reinterpret_cast<const uint2 *>(p);
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&u.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&u.y);
    float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    x[0] = fa.x; x[1] = fa.y; x[2] = fb.x; x[3] = fb.y;
}
__device__ __forceinline__ void store4(float *p, const float (&x)[4]) {
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16 *p, const float (&x)[4]) {
    __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
    __nv_bfloat162 b = __floats2bfloat162_rn(x[2], x[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}
// Two consecutive elements (8-byte aligned for f32, 4 for bf16).
__device__ __forceinline__ void load2(const float *p, float (&x)[2]) {
    float2 v = *reinterpret_cast<const float2 *>(p);
    x[0] = v.x; x[1] = v.y;
}
__device__ __forceinline__ void load2(const __nv_bfloat16 *p, float (&x)[2]) {
    float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
    x[0] = f.x; x[1] = f.y;
}
__device__ __forceinline__ void store2(float *p, const float (&x)[2]) {
    *reinterpret_cast<float2 *>(p) = make_float2(x[0], x[1]);
}
__device__ __forceinline__ void store2(__nv_bfloat16 *p, const float (&x)[2]) {
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(x[0], x[1]);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f32(float &y, float x) { y = x; }
__device__ __forceinline__ void from_f32(__nv_bfloat16 &y, float x) { y = __float2bfloat16_rn(x); }

}  // namespace osdn
