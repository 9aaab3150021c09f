// tc_common.cuh -- pieces shared by the two tensor-core kernels of Phase 2
// (chunk preparation and the state chain): 128-byte-swizzled tile stores,
// TMEM loads, shared-memory matrix descriptors, bounded mbarrier waits and
// the TMA tensor maps.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "osdn_device.cuh"
#include "ptx.cuh"

namespace osdn {
namespace tc {

constexpr int C = 64;                          // tokens per chunk
constexpr uint32_t kWaitLimit = 1u << 15;      // sleeping polls before a wait gives up
constexpr uint32_t kSleepNs = 1u << 16;        // longest sleep per poll (~65 us)

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// n (multiple of 8) consecutive bf16 of row r, columns [c0, c0+n) within one
// 64-column block, into a 128B-swizzled tile whose 64-column blocks hold
// `rows` rows of 128 bytes.  The same bytes serve as a K-major operand
// (rows = M or N) or an MN-major one (rows = the reduction index).
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

// The inverse of st_row_sw128: n bf16 of row r from column c0, as fp32.
__device__ __forceinline__ void ld_row_sw128(const uint8_t *tile, int rows, int r, int c0,
                                             float *vals, int n) {
    const uint8_t *rowp = tile + (c0 >> 6) * rows * 128 + r * 128;
    const int cb = (c0 & 63) >> 3;
#pragma unroll
    for (int i = 0; i < n; i += 8) {
        const int chunk = (cb + (i >> 3)) ^ (r & 7);
        const uint4 pk = *reinterpret_cast<const uint4 *>(rowp + chunk * 16);
        const uint32_t w[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
            vals[i + 2 * e] = f.x;
            vals[i + 2 * e + 1] = f.y;
        }
    }
}

// n (multiple of 8) fp32 values as bf16 to global memory (16-byte aligned).
__device__ __forceinline__ void st_global_bf16(__nv_bfloat16 *dst, const float *vals, int n) {
#pragma unroll
    for (int i = 0; i < n; i += 8) {
        uint4 pk;
        pk.x = pack_bf16x2(vals[i + 0], vals[i + 1]);
        pk.y = pack_bf16x2(vals[i + 2], vals[i + 3]);
        pk.z = pack_bf16x2(vals[i + 4], vals[i + 5]);
        pk.w = pack_bf16x2(vals[i + 6], vals[i + 7]);
        *reinterpret_cast<uint4 *>(dst + i) = pk;
    }
}

// 32 consecutive TMEM columns of this thread's lane.
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
// N (16, 32 or 64) consecutive TMEM columns, all loads in flight before one wait.
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, float (&v)[N]) {
    static_assert(N == 16 || N == 32 || N == 64, "16, 32 or 64 columns");
    float a[4][16];
#pragma unroll
    for (int q = 0; q < N / 16; ++q) ptx::tmem_ld16(taddr + 16 * q, a[q]);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int q = 0; q < N / 16; ++q)
#pragma unroll
        for (int i = 0; i < 16; ++i) v[16 * q + i] = a[q][i];
}
// 64 consecutive TMEM columns, four loads in flight before one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
    float a[16], b[16], c[16], d[16];
    ptx::tmem_ld16(taddr, a);
    ptx::tmem_ld16(taddr + 16, b);
    ptx::tmem_ld16(taddr + 32, c);
    ptx::tmem_ld16(taddr + 48, d);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[i] = a[i];
        v[16 + i] = b[i];
        v[32 + i] = c[i];
        v[48 + i] = d[i];
    }
}
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const float (&v)[64]) {
    float a[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int i = 0; i < 16; ++i) a[i] = v[16 * q + i];
        ptx::tmem_st16(taddr + 16 * q, a);
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

// Bounded wait that also gives up as soon as another thread has aborted
// (at most `limit` sleeping polls).
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         int *status, uint32_t limit = kWaitLimit) {
    for (uint32_t i = 0; i < limit; ++i) {
        if (ptx::mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
        if (*abort_flag) return false;
    }
    report_status(status, OSDN_ERR_TIMEOUT);
    *abort_flag = 1;
    return false;
}
// Bounded poll without a suspend hint, for waits on a critical path, where a
// sleeping thread wakes too late (at most `limit` polls).
__device__ __forceinline__ bool wait_poll(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int *status, uint32_t limit = kWaitLimit << 11) {
    for (uint32_t i = 0; i < limit; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && *abort_flag) return false;
    }
    report_status(status, OSDN_ERR_TIMEOUT);
    *abort_flag = 1;
    return false;
}
// Bounded wait that ignores aborts: used before a CTA exits, so that bulk
// copies and MMAs it started have landed before its shared memory and TMEM
// are released.
__device__ __forceinline__ void drain_bar(uint64_t *bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (ptx::mbar_try_wait_sleep(bar, parity, kSleepNs)) return;
}

// 1024-byte aligned start of dynamic shared memory, by pointer arithmetic so
// accesses stay in the shared state space (an integer round trip would make
// them generic).
__device__ __forceinline__ uint8_t *align1024(uint8_t *raw) {
    return raw + ((1024u - (ptx::smem_u32(raw) & 1023u)) & 1023u);
}

// ----------------------------------------------------------------------- host
bool tensor_map_encoder_ready();
// [BH][rows][width] bf16 in global memory, boxes of 64 columns x 64 rows,
// 128-byte swizzle; rows past `rows` read as zero.
bool make_map(CUtensorMap *m, const void *ptr, int BH, int rows, int width);
// Streaming multiprocessors of the current device (152 if the query fails).
int sm_count();
// Extra inputs of the chunk preparation: the fused forward pass's
// checkpoints, from which it rebuilds Kt (else Kt is read), or a decay per
// key channel (all NULL: the plain or scalar-gated preparation).
struct Fused {
    const float *r = nullptr;       // retention r_t [BH][T], or NULL (r = 1)
    const float *ecoef = nullptr;   // e_t [BH][T]
    const float *dchk = nullptr;    // d entering each 64-token chunk [BH][nch][K]
    const float *alpha_k = nullptr; // a decay per key channel [BH][T][K] instead (not fused)
};

}  // namespace tc
}  // namespace osdn
