// osdn_api.cu -- the extern "C" boundary declared in include/osdn.h:
// argument validation, workspace sizing, kernel dispatch and status.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "osdn.h"

namespace osdn {
cudaError_t precond_scan_launch(int io, int BH, int T, int K, const void *k, const float *beta,
                                const float *r, float eta, const float *d0, void *ktilde,
                                float *dT, float *logratio, void *scratch, int *status,
                                cudaStream_t stream);
size_t precond_scratch_bytes(int BH, int T, int K);
cudaError_t precond_checkpoint_launch(int io, int BH, int T, int K, const void *k,
                                      const float *beta, const float *r, float eta,
                                      const float *d0, float *dT, float *ecoef, float *dchk,
                                      int chk_shift, void *scratch, int *status,
                                      cudaStream_t stream);
cudaError_t delta_tc_fused_launch(int BH, int T, int K, int V, const void *q, const void *k,
                                  const void *v, const float *beta, const float *r,
                                  const float *ecoef, const float *dchk, const float *alpha,
                                  const float *S0, void *o, float *ST, void *scratch, int *status,
                                  cudaStream_t stream);
size_t precond_scratch_bytes_for(int BH, int T, int K, bool has_r);
int precond_segments(int BH, int T, bool has_r, int *L_out);
size_t precond_noalloc_capacity();
cudaError_t precond_scan_noalloc_launch(int io, int BH, int T, int K, const void *k,
                                        const float *beta, const float *r, float eta,
                                        const float *d0, void *ktilde, float *dT,
                                        cudaStream_t stream);
cudaError_t fill_state_launch(size_t n, const float *src, float fill, float *dst,
                              cudaStream_t stream);
cudaError_t delta_simt_launch(int io, int BH, int T, int K, int V, const void *q, const void *k,
                              const void *kt, const void *v, const float *beta,
                              const float *alpha, const float *S0, void *o, float *ST,
                              cudaStream_t stream);
size_t delta_tc_scratch_bytes(int BH, int T, int K, int V);
size_t delta_tc_kda_scratch_bytes(int BH, int T, int K, int V);
cudaError_t delta_tc_kda_launch(int BH, int T, int K, int V, const void *q, const void *k,
                                const void *kt, const void *v, const float *beta,
                                const float *alpha_k, const float *S0, void *o, float *ST,
                                void *scratch, int *status, cudaStream_t stream);
cudaError_t delta_tc_launch(int BH, int T, int K, int V, const void *q, const void *k,
                            const void *kt, const void *v, const float *beta, const float *alpha,
                            const float *S0, void *o, float *ST, void *scratch, int *status,
                            cudaStream_t stream);
size_t backward_scratch_bytes(int BH, int T, int K, int V, bool per_channel);
cudaError_t backward_launch(int io, int BH, int T, int K, int V, const void *q, const void *k,
                            const void *kt, const void *v, const float *beta, const float *r,
                            float eta, const float *d0, const float *alpha, const float *S0,
                            const void *dO, const float *dST, const float *ddT,
                            const void *dkt_ext, void *dq, void *dk, void *dv, float *dbeta,
                            float *dr, float *dalpha, float *dd0, float *dS0, float *deta,
                            bool per_channel, void *scratch, int *status, cudaStream_t stream);
cudaError_t delta_simt_kda_launch(int io, int BH, int T, int K, int V, const void *q,
                                  const void *k, const void *kt, const void *v,
                                  const float *beta, const float *alpha_k, const float *S0,
                                  void *o, float *ST, cudaStream_t stream);
cudaError_t decode_step_kda_launch(int io, int BH, int K, int V, const void *q, const void *k,
                                   const void *v, const float *beta, const float *r, float eta,
                                   const float *alpha_k, float *d, float *S, void *o,
                                   void *ktilde, cudaStream_t stream);
cudaError_t decode_step_launch(int io, int BH, int K, int V, const void *q, const void *k,
                               const void *v, const float *beta, const float *r, float eta,
                               const float *alpha, float *d, float *S, void *o, void *ktilde,
                               cudaStream_t stream);
}  // namespace osdn

namespace {

constexpr size_t kStatusBytes = 256;

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// At most 2^24 sequences: the kernels spread them over two grid dimensions,
// and the Phase 1 scan numbers its speculative segments in a 32-bit index.
constexpr size_t kMaxSeqs = size_t(1) << 24;
bool dims_ok(int B, int H, int T) {
    return B >= 0 && H >= 0 && T >= 0 && (size_t)B * (size_t)H <= kMaxSeqs;
}
bool width_ok(int x) { return x == 64 || x == 128; }
// The tensor-core Phase 2 addresses each chunk's rows of its prepared
// operands (chunk index x K, K <= 128) with 32-bit TMA coordinates and int
// chunk arithmetic: T is capped so that ceil(T/64) * 128 stays below 2^31.
constexpr int kMaxTcTokens = (0x7fffffff / 128) * 64;
size_t io_bytes(int io) { return io == OSDN_BF16 ? 2 : 4; }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// The kernels are built for sm_103a only: refuse other devices up front.
int check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return OSDN_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return OSDN_ERR_CUDA;
    if (major != 10 || minor != 3) return OSDN_ERR_ARCH;
    return OSDN_OK;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// osdn_forward's workspace after the status word: the scan's segment scratch,
// then (bf16) e_t, the 64-token checkpoints of d and Phase 2's workspace, or
// (fp32) ktilde.
struct FwdCarve {
    void *p1;
    float *ecoef, *dchk;
    void *kt, *p2;
    size_t bytes;
};
FwdCarve fwd_carve(void *base, int io, int BH, int T, int K, int V) {
    const size_t nch = ((size_t)T + 63) / 64;
    size_t sz[4];
    sz[0] = round256(osdn::precond_scratch_bytes(BH, T, K));
    if (io == OSDN_BF16) {
        sz[1] = round256((size_t)BH * T * 4);
        sz[2] = round256((size_t)BH * nch * K * 4);
        sz[3] = round256(osdn::delta_tc_scratch_bytes(BH, T, K, V));
    } else {
        sz[1] = round256((size_t)BH * T * K * 4);
        sz[2] = sz[3] = 0;
    }
    char *b = static_cast<char *>(base);
    char *at[4];
    size_t off = 0;
    for (int i = 0; i < 4; ++i) {
        at[i] = b ? b + off : nullptr;
        off += sz[i];
    }
    FwdCarve c;
    c.p1 = at[0];
    c.ecoef = io == OSDN_BF16 ? reinterpret_cast<float *>(at[1]) : nullptr;
    c.dchk = io == OSDN_BF16 ? reinterpret_cast<float *>(at[2]) : nullptr;
    c.kt = io == OSDN_BF16 ? nullptr : at[1];
    c.p2 = io == OSDN_BF16 ? at[3] : nullptr;
    c.bytes = off;
    return c;
}

}  // namespace

extern "C" {

int osdn_version(void) { return 100; }

const char *osdn_status_string(int code) {
    switch (code) {
    case OSDN_OK: return "ok";
    case OSDN_ERR_NULL: return "a required pointer is NULL";
    case OSDN_ERR_DIMS: return "bad dimensions (negative size, B*H over 2^24, or K/V not 64 or 128)";
    case OSDN_ERR_DTYPE: return "unsupported io dtype";
    case OSDN_ERR_ALIGN: return "pointer not 16-byte aligned";
    case OSDN_ERR_WORKSPACE: return "workspace NULL or too small";
    case OSDN_ERR_CUDA: return "CUDA runtime error";
    case OSDN_ERR_TIMEOUT: return "device wait timed out";
    case OSDN_ERR_DEVICE: return "device-side consistency check failed";
    case OSDN_ERR_ALIAS: return "output overlaps an input";
    case OSDN_ERR_ARCH: return "device is not sm_103 (GB300)";
    case OSDN_ERR_SCRATCH: return "problem needs more scratch than the static buffer holds";
    default: return "unknown status";
    }
}

size_t osdn_precond_scan_workspace_bytes(int B, int H, int T, int K) {
    if (B < 0 || H < 0 || T < 0 || !width_ok(K)) return kStatusBytes;
    return kStatusBytes + osdn::precond_scratch_bytes(B * H, T, K);
}

size_t osdn_chunk_fwd_workspace_bytes(int io, int B, int H, int T, int K, int V) {
    if (!dims_ok(B, H, T) || !width_ok(K) || !width_ok(V)) return kStatusBytes;
    if (io != OSDN_BF16 || T == 0 || T > kMaxTcTokens) return kStatusBytes;
    // the tensor-core path keeps each chunk's prepared operands in the workspace
    return kStatusBytes + osdn::delta_tc_scratch_bytes(B * H, T, K, V);
}

size_t osdn_forward_workspace_bytes(int io, int B, int H, int T, int K, int V) {
    if (!dims_ok(B, H, T) || !width_ok(K) || !width_ok(V) || T == 0) return kStatusBytes;
    if (io != OSDN_BF16 && io != OSDN_F32) return kStatusBytes;
    const FwdCarve c = fwd_carve(nullptr, io, B * H, T, K, V);
    return kStatusBytes + c.bytes;
}

size_t osdn_backward_workspace_bytes(int B, int H, int T, int K, int V) {
    if (!dims_ok(B, H, T) || !width_ok(K) || !width_ok(V) || T == 0) return kStatusBytes;
    return kStatusBytes + osdn::backward_scratch_bytes(B * H, T, K, V, false);
}

size_t osdn_backward_kda_workspace_bytes(int B, int H, int T, int K, int V) {
    if (!dims_ok(B, H, T) || !width_ok(K) || !width_ok(V) || T == 0) return kStatusBytes;
    return kStatusBytes + osdn::backward_scratch_bytes(B * H, T, K, V, true);
}

size_t osdn_chunk_fwd_kda_workspace_bytes(int io, int B, int H, int T, int K, int V) {
    if (!dims_ok(B, H, T) || !width_ok(K) || !width_ok(V)) return kStatusBytes;
    // fp32 I/O runs the FFMA recurrence, which needs no scratch; bf16 keeps
    // each chunk's prepared operands and its per-channel decay product
    if (io != OSDN_BF16 || T == 0 || T > kMaxTcTokens) return kStatusBytes;
    return kStatusBytes + osdn::delta_tc_kda_scratch_bytes(B * H, T, K, V);
}

int osdn_workspace_init(void *workspace, size_t workspace_bytes, void *stream) {
    if (!workspace) return OSDN_ERR_NULL;
    if (workspace_bytes < kStatusBytes) return OSDN_ERR_WORKSPACE;
    if (misaligned(workspace)) return OSDN_ERR_ALIGN;
    if (cudaMemsetAsync(workspace, 0, kStatusBytes, (cudaStream_t)stream) != cudaSuccess)
        return OSDN_ERR_CUDA;
    return OSDN_OK;
}

int osdn_check_status(const void *workspace, void *stream) {
    if (!workspace) return OSDN_ERR_NULL;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return OSDN_ERR_CUDA;
    int code = 0;
    if (cudaMemcpy(&code, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return OSDN_ERR_CUDA;
    return code;
}

}  // extern "C"

namespace {

// osdn_precond_scan and osdn_precond_scan_residual: one validation, one launch.
int precond_scan_checked(int io, int B, int H, int T, int K, const void *k, const float *beta,
                         const float *r, float eta, const float *d0, void *ktilde, float *dT,
                         float *log_ratio, void *workspace, size_t workspace_bytes, void *stream) {
    if (io != OSDN_F32 && io != OSDN_BF16) return OSDN_ERR_DTYPE;
    if (!dims_ok(B, H, T) || !width_ok(K)) return OSDN_ERR_DIMS;
    if (!workspace) return OSDN_ERR_WORKSPACE;
    if (workspace_bytes < osdn_precond_scan_workspace_bytes(B, H, T, K)) return OSDN_ERR_WORKSPACE;
    const size_t BH = (size_t)B * H;
    if (BH == 0) return OSDN_OK;
    if (BH * (size_t)osdn::precond_segments((int)BH, T, r != nullptr, nullptr) > 0x7fffffffu)
        return OSDN_ERR_DIMS;   // one warp per segment, numbered in 32 bits
    if (T > 0 && (!k || !beta || !ktilde)) return OSDN_ERR_NULL;
    if (misaligned(k) || misaligned(beta) || misaligned(r) || misaligned(d0) ||
        misaligned(ktilde) || misaligned(dT) || misaligned(log_ratio) || misaligned(workspace))
        return OSDN_ERR_ALIGN;
    const size_t kbytes = BH * (size_t)T * K * io_bytes(io);
    if (overlap(k, kbytes, ktilde, kbytes) || overlap(dT, BH * K * 4, ktilde, kbytes) ||
        overlap(dT, BH * K * 4, k, kbytes) || overlap(log_ratio, BH * 4, k, kbytes) ||
        overlap(log_ratio, BH * 4, ktilde, kbytes) || overlap(log_ratio, BH * 4, dT, BH * K * 4))
        return OSDN_ERR_ALIAS;
    {   // the workspace is written by the call: it may overlap nothing else
        const size_t gb = BH * (size_t)T * 4;
        const void *all[7] = {k, beta, r, d0, ktilde, dT, log_ratio};
        const size_t sz[7] = {kbytes, gb, gb, BH * K * 4, kbytes, BH * K * 4, BH * 4};
        for (int i = 0; i < 7; ++i)
            if (overlap(workspace, workspace_bytes, all[i], sz[i])) return OSDN_ERR_ALIAS;
    }
    int dev = check_device();
    if (dev != OSDN_OK) return dev;
    void *scratch = static_cast<char *>(workspace) + kStatusBytes;
    cudaError_t e = osdn::precond_scan_launch(io, (int)BH, T, K, k, beta, r, eta, d0, ktilde, dT,
                                              log_ratio, scratch, static_cast<int *>(workspace),
                                              (cudaStream_t)stream);
    return e == cudaSuccess ? OSDN_OK : OSDN_ERR_CUDA;
}

}  // namespace

extern "C" {

int osdn_precond_scan(int io, int B, int H, int T, int K, const void *k, const float *beta,
                      const float *r, float eta, const float *d0, void *ktilde, float *dT,
                      void *workspace, size_t workspace_bytes, void *stream) {
    return precond_scan_checked(io, B, H, T, K, k, beta, r, eta, d0, ktilde, dT, nullptr,
                                workspace, workspace_bytes, stream);
}

int osdn_precond_scan_residual(int io, int B, int H, int T, int K, const void *k,
                               const float *beta, const float *r, float eta, const float *d0,
                               void *ktilde, float *dT, float *log_ratio, void *workspace,
                               size_t workspace_bytes, void *stream) {
    if (!log_ratio) return OSDN_ERR_NULL;
    return precond_scan_checked(io, B, H, T, K, k, beta, r, eta, d0, ktilde, dT, log_ratio,
                                workspace, workspace_bytes, stream);
}

int osdn_precond_scan_noalloc(int io, int B, int H, int T, int K, const void *k,
                              const float *beta, const float *r, float eta, const float *d0,
                              void *ktilde, float *dT, void *stream) {
    if (io != OSDN_F32 && io != OSDN_BF16) return OSDN_ERR_DTYPE;
    if (!dims_ok(B, H, T) || !width_ok(K)) return OSDN_ERR_DIMS;
    const size_t BH = (size_t)B * H;
    if (BH == 0) return OSDN_OK;
    if (BH * (size_t)osdn::precond_segments((int)BH, T, r != nullptr, nullptr) > 0x7fffffffu)
        return OSDN_ERR_DIMS;
    if (T > 0 && (!k || !beta || !ktilde)) return OSDN_ERR_NULL;
    if (misaligned(k) || misaligned(beta) || misaligned(r) || misaligned(d0) ||
        misaligned(ktilde) || misaligned(dT))
        return OSDN_ERR_ALIGN;
    const size_t kbytes = BH * (size_t)T * K * io_bytes(io);
    if (overlap(k, kbytes, ktilde, kbytes) || overlap(dT, BH * K * 4, ktilde, kbytes) ||
        overlap(dT, BH * K * 4, k, kbytes))
        return OSDN_ERR_ALIAS;
    if (osdn::precond_scratch_bytes_for((int)BH, T, K, r != nullptr) >
        osdn::precond_noalloc_capacity())
        return OSDN_ERR_SCRATCH;
    int dev = check_device();
    if (dev != OSDN_OK) return dev;
    cudaError_t e = osdn::precond_scan_noalloc_launch(io, (int)BH, T, K, k, beta, r, eta, d0,
                                                      ktilde, dT, (cudaStream_t)stream);
    return e == cudaSuccess ? OSDN_OK : OSDN_ERR_CUDA;
}

int osdn_chunk_fwd(int io, int B, int H, int T, int K, int V, const void *q, const void *k,
                   const void *ktilde, const void *v, const float *beta, const float *alpha,
                   const float *S0, void *o, float *ST, void *workspace, size_t workspace_bytes,
                   void *stream) {
    if (io != OSDN_F32 && io != OSDN_BF16) return OSDN_ERR_DTYPE;
    if (!dims_ok(B, H, T) || !width_ok(K) || !width_ok(V)) return OSDN_ERR_DIMS;
    if (io == OSDN_BF16 && T > kMaxTcTokens) return OSDN_ERR_DIMS;
    if (!workspace) return OSDN_ERR_WORKSPACE;
    if (workspace_bytes < osdn_chunk_fwd_workspace_bytes(io, B, H, T, K, V))
        return OSDN_ERR_WORKSPACE;
    const size_t BH = (size_t)B * H;
    if (BH == 0) return OSDN_OK;
    if (T > 0 && (!q || !k || !ktilde || !v || !beta || !o)) return OSDN_ERR_NULL;
    if (misaligned(q) || misaligned(k) || misaligned(ktilde) || misaligned(v) ||
        misaligned(beta) || misaligned(alpha) || misaligned(S0) || misaligned(o) ||
        misaligned(ST) || misaligned(workspace))
        return OSDN_ERR_ALIGN;
    const size_t es = io_bytes(io);
    const size_t kb = BH * (size_t)T * K * es, vb = BH * (size_t)T * V * es;
    const size_t sb = BH * (size_t)V * K * 4, gb = BH * (size_t)T * 4;
    const void *ins[7] = {q, k, ktilde, v, beta, alpha, S0};
    const size_t insz[7] = {kb, kb, kb, vb, gb, gb, sb};
    for (int i = 0; i < 7; ++i)
        if (overlap(o, vb, ins[i], insz[i]) || overlap(ST, sb, ins[i], insz[i]) ||
            overlap(workspace, workspace_bytes, ins[i], insz[i]))
            return OSDN_ERR_ALIAS;
    if (overlap(o, vb, ST, sb) || overlap(workspace, workspace_bytes, o, vb) ||
        overlap(workspace, workspace_bytes, ST, sb))
        return OSDN_ERR_ALIAS;
    int dev = check_device();
    if (dev != OSDN_OK) return dev;
    cudaError_t e;
    if (T == 0)
        e = osdn::fill_state_launch(ST ? sb / 4 : 0, S0, 0.0f, ST, (cudaStream_t)stream);
    else if (io == OSDN_BF16)  // tensor cores: bf16 operands, fp32 accumulation
        e = osdn::delta_tc_launch((int)BH, T, K, V, q, k, ktilde, v, beta, alpha, S0, o, ST,
                                  static_cast<char *>(workspace) + kStatusBytes,
                                  static_cast<int *>(workspace), (cudaStream_t)stream);
    else  // fp32 I/O: fp32 FFMA (tensor-core operand rounding would not meet fp32 accuracy)
        e = osdn::delta_simt_launch(io, (int)BH, T, K, V, q, k, ktilde, v, beta, alpha, S0, o, ST,
                                    (cudaStream_t)stream);
    return e == cudaSuccess ? OSDN_OK : OSDN_ERR_CUDA;
}

int osdn_forward(int io, int B, int H, int T, int K, int V, const void *q, const void *k,
                 const void *v, const float *beta, const float *r, float eta, const float *d0,
                 const float *alpha, const float *S0, void *o, float *dT, float *ST,
                 void *workspace, size_t workspace_bytes, void *stream) {
    if (io != OSDN_F32 && io != OSDN_BF16) return OSDN_ERR_DTYPE;
    if (!dims_ok(B, H, T) || !width_ok(K) || !width_ok(V)) return OSDN_ERR_DIMS;
    if (io == OSDN_BF16 && T > kMaxTcTokens) return OSDN_ERR_DIMS;
    if (!workspace) return OSDN_ERR_WORKSPACE;
    if (workspace_bytes < osdn_forward_workspace_bytes(io, B, H, T, K, V)) return OSDN_ERR_WORKSPACE;
    const size_t BH = (size_t)B * H;
    if (BH == 0) return OSDN_OK;
    if (BH * (size_t)osdn::precond_segments((int)BH, T, r != nullptr, nullptr) > 0x7fffffffu)
        return OSDN_ERR_DIMS;   // one warp per scan segment, numbered in 32 bits
    if (T > 0 && (!q || !k || !v || !beta || !o)) return OSDN_ERR_NULL;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(beta) || misaligned(r) ||
        misaligned(d0) || misaligned(alpha) || misaligned(S0) || misaligned(o) ||
        misaligned(dT) || misaligned(ST) || misaligned(workspace))
        return OSDN_ERR_ALIGN;
    const size_t es = io_bytes(io);
    const size_t kb = BH * (size_t)T * K * es, vb = BH * (size_t)T * V * es;
    const size_t sb = BH * (size_t)V * K * 4, gb = BH * (size_t)T * 4, db = BH * (size_t)K * 4;
    const void *ins[8] = {q, k, v, beta, r, alpha, d0, S0};
    const size_t insz[8] = {kb, kb, vb, gb, gb, gb, db, sb};
    const void *outs[4] = {o, dT, ST, workspace};
    const size_t outsz[4] = {vb, db, sb, workspace_bytes};
    for (int i = 0; i < 4; ++i) {
        for (int j = 0; j < 8; ++j)
            if (overlap(outs[i], outsz[i], ins[j], insz[j])) return OSDN_ERR_ALIAS;
        for (int j = i + 1; j < 4; ++j)
            if (overlap(outs[i], outsz[i], outs[j], outsz[j])) return OSDN_ERR_ALIAS;
    }
    int dev = check_device();
    if (dev != OSDN_OK) return dev;
    cudaStream_t st = (cudaStream_t)stream;
    int *status = static_cast<int *>(workspace);
    cudaError_t e;
    if (T == 0) {   // d_T = d_0 and S_T = S_0
        e = osdn::precond_scan_launch(io, (int)BH, 0, K, k, beta, r, eta, d0, nullptr, dT, nullptr,
                                      nullptr, status, st);
        if (e == cudaSuccess) e = osdn::fill_state_launch(ST ? sb / 4 : 0, S0, 0.0f, ST, st);
        return e == cudaSuccess ? OSDN_OK : OSDN_ERR_CUDA;
    }
    const FwdCarve c = fwd_carve(static_cast<char *>(workspace) + kStatusBytes, io, (int)BH, T, K, V);
    if (io == OSDN_BF16) {
        e = osdn::precond_checkpoint_launch(io, (int)BH, T, K, k, beta, r, eta, d0, dT, c.ecoef,
                                            c.dchk, 6, c.p1, status, st);
        if (e == cudaSuccess)
            e = osdn::delta_tc_fused_launch((int)BH, T, K, V, q, k, v, beta, r, c.ecoef, c.dchk,
                                            alpha, S0, o, ST, c.p2, status, st);
    } else {
        e = osdn::precond_scan_launch(io, (int)BH, T, K, k, beta, r, eta, d0, c.kt, dT, nullptr,
                                      c.p1, status, st);
        if (e == cudaSuccess)
            e = osdn::delta_simt_launch(io, (int)BH, T, K, V, q, k, c.kt, v, beta, alpha, S0, o, ST,
                                        st);
    }
    return e == cudaSuccess ? OSDN_OK : OSDN_ERR_CUDA;
}

}  // extern "C"

namespace {

// osdn_decode_step and osdn_decode_step_kda: one validation, one launch.
// With a per-channel decay alpha is [B][H][K], else [B][H].
int decode_checked(int io, int B, int H, int K, int V, const void *q, const void *k,
                   const void *v, const float *beta, const float *r, float eta,
                   const float *alpha, float *d, float *S, void *o, void *ktilde,
                   bool per_channel, void *workspace, size_t workspace_bytes, void *stream) {
    if (io != OSDN_F32 && io != OSDN_BF16) return OSDN_ERR_DTYPE;
    if (!dims_ok(B, H, 0) || !width_ok(K) || !width_ok(V)) return OSDN_ERR_DIMS;
    if (!workspace || workspace_bytes < kStatusBytes) return OSDN_ERR_WORKSPACE;
    const size_t BH = (size_t)B * H;
    if (BH == 0) return OSDN_OK;
    if (!q || !k || !v || !beta || !d || !S || !o) return OSDN_ERR_NULL;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(beta) || misaligned(r) ||
        misaligned(alpha) || misaligned(d) || misaligned(S) || misaligned(o) ||
        misaligned(ktilde) || misaligned(workspace))
        return OSDN_ERR_ALIGN;
    const size_t es = io_bytes(io);
    const void *ins[6] = {q, k, v, beta, r, alpha};
    const size_t insz[6] = {BH * K * es, BH * K * es, BH * V * es, BH * 4, BH * 4,
                            per_channel ? BH * K * 4 : BH * 4};
    const void *outs[4] = {d, S, o, ktilde};
    const size_t outsz[4] = {BH * K * 4, BH * V * K * 4, BH * V * es, BH * K * es};
    for (int a = 0; a < 4; ++a) {
        for (int i = 0; i < 6; ++i)
            if (overlap(outs[a], outsz[a], ins[i], insz[i])) return OSDN_ERR_ALIAS;
        for (int b = a + 1; b < 4; ++b)
            if (overlap(outs[a], outsz[a], outs[b], outsz[b])) return OSDN_ERR_ALIAS;
        if (overlap(workspace, workspace_bytes, outs[a], outsz[a])) return OSDN_ERR_ALIAS;
    }
    for (int i = 0; i < 6; ++i)
        if (overlap(workspace, workspace_bytes, ins[i], insz[i])) return OSDN_ERR_ALIAS;
    int dev = check_device();
    if (dev != OSDN_OK) return dev;
    cudaError_t e = per_channel
        ? osdn::decode_step_kda_launch(io, (int)BH, K, V, q, k, v, beta, r, eta, alpha, d, S, o,
                                       ktilde, (cudaStream_t)stream)
        : osdn::decode_step_launch(io, (int)BH, K, V, q, k, v, beta, r, eta, alpha, d, S, o,
                                   ktilde, (cudaStream_t)stream);
    return e == cudaSuccess ? OSDN_OK : OSDN_ERR_CUDA;
}

}  // namespace

extern "C" {

int osdn_decode_step(int io, int B, int H, int K, int V, const void *q, const void *k,
                     const void *v, const float *beta, const float *r, float eta,
                     const float *alpha, float *d, float *S, void *o, void *ktilde,
                     void *workspace, size_t workspace_bytes, void *stream) {
    return decode_checked(io, B, H, K, V, q, k, v, beta, r, eta, alpha, d, S, o, ktilde, false,
                          workspace, workspace_bytes, stream);
}

int osdn_decode_step_kda(int io, int B, int H, int K, int V, const void *q, const void *k,
                         const void *v, const float *beta, const float *r, float eta,
                         const float *alpha_k, float *d, float *S, void *o, void *ktilde,
                         void *workspace, size_t workspace_bytes, void *stream) {
    return decode_checked(io, B, H, K, V, q, k, v, beta, r, eta, alpha_k, d, S, o, ktilde, true,
                          workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

// osdn_backward and osdn_backward_kda: one validation, one launch.  With a
// per-channel decay alpha and dalpha are [B][H][T][K], else [B][H][T].
int backward_checked(int io, int B, int H, int T, int K, int V, const void *q, const void *k,
                     const void *ktilde, const void *v, const float *beta, const float *r,
                     float eta, const float *d0, const float *alpha, const float *S0,
                     const void *d_o, const float *d_ST, const float *d_dT,
                     const void *d_ktilde, void *dq, void *dk, void *dv, float *dbeta, float *dr,
                     float *dalpha, float *dd0, float *dS0, float *deta, bool per_channel,
                     void *workspace, size_t workspace_bytes, void *stream) {
    if (io != OSDN_F32 && io != OSDN_BF16) return OSDN_ERR_DTYPE;
    if (!dims_ok(B, H, T) || !width_ok(K) || !width_ok(V)) return OSDN_ERR_DIMS;
    if (!workspace) return OSDN_ERR_WORKSPACE;
    const size_t need = per_channel ? osdn_backward_kda_workspace_bytes(B, H, T, K, V)
                                    : osdn_backward_workspace_bytes(B, H, T, K, V);
    if (workspace_bytes < need) return OSDN_ERR_WORKSPACE;
    const size_t BH = (size_t)B * H;
    if (BH == 0) return OSDN_OK;
    if (T > 0 && (!q || !k || !ktilde || !v || !beta || !dq || !dk || !dv || !dbeta))
        return OSDN_ERR_NULL;
    const void *ins[13] = {q, k, ktilde, v, beta, r, d0, alpha, S0, d_o, d_ST, d_dT, d_ktilde};
    void *outs[9] = {dq, dk, dv, dbeta, dr, dalpha, dd0, dS0, deta};
    if (misaligned(workspace)) return OSDN_ERR_ALIGN;
    for (const void *p : ins)
        if (misaligned(p)) return OSDN_ERR_ALIGN;
    for (const void *p : outs)
        if (misaligned(p)) return OSDN_ERR_ALIGN;
    const size_t es = io_bytes(io);
    const size_t kb = BH * (size_t)T * K * es, vb = BH * (size_t)T * V * es;
    const size_t gb = BH * (size_t)T * 4, db = BH * (size_t)K * 4, sb = BH * (size_t)V * K * 4;
    const size_t ab = per_channel ? BH * (size_t)T * K * 4 : gb;   // alpha, dalpha
    const size_t insz[13] = {kb, kb, kb, vb, gb, gb, db, ab, sb, vb, sb, db, kb};
    const size_t outsz[9] = {kb, kb, vb, gb, gb, ab, db, sb, BH * 4};
    for (int a = 0; a < 9; ++a) {
        for (int i = 0; i < 13; ++i)
            if (overlap(outs[a], outsz[a], ins[i], insz[i])) return OSDN_ERR_ALIAS;
        for (int b = a + 1; b < 9; ++b)
            if (overlap(outs[a], outsz[a], outs[b], outsz[b])) return OSDN_ERR_ALIAS;
        if (overlap(workspace, workspace_bytes, outs[a], outsz[a])) return OSDN_ERR_ALIAS;
    }
    for (int i = 0; i < 13; ++i)
        if (overlap(workspace, workspace_bytes, ins[i], insz[i])) return OSDN_ERR_ALIAS;
    int dev = check_device();
    if (dev != OSDN_OK) return dev;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e;
    if (T == 0) {
        e = osdn::fill_state_launch(dS0 ? sb / 4 : 0, d_ST, 0.0f, dS0, st);
        if (e == cudaSuccess) e = osdn::fill_state_launch(dd0 ? db / 4 : 0, d_dT, 0.0f, dd0, st);
        if (e == cudaSuccess) e = osdn::fill_state_launch(deta ? BH : 0, nullptr, 0.0f, deta, st);
    } else {
        e = osdn::backward_launch(io, (int)BH, T, K, V, q, k, ktilde, v, beta, r, eta, d0, alpha,
                                  S0, d_o, d_ST, d_dT, d_ktilde, dq, dk, dv, dbeta, dr, dalpha,
                                  dd0, dS0, deta, per_channel,
                                  static_cast<char *>(workspace) + kStatusBytes,
                                  static_cast<int *>(workspace), st);
    }
    return e == cudaSuccess ? OSDN_OK : OSDN_ERR_CUDA;
}

}  // namespace

extern "C" {

int osdn_backward(int io, int B, int H, int T, int K, int V, const void *q, const void *k,
                  const void *ktilde, const void *v, const float *beta, const float *r,
                  float eta, const float *d0, const float *alpha, const float *S0,
                  const void *d_o, const float *d_ST, const float *d_dT, const void *d_ktilde,
                  void *dq, void *dk, void *dv, float *dbeta, float *dr, float *dalpha,
                  float *dd0, float *dS0, float *deta, void *workspace, size_t workspace_bytes,
                  void *stream) {
    return backward_checked(io, B, H, T, K, V, q, k, ktilde, v, beta, r, eta, d0, alpha, S0, d_o,
                            d_ST, d_dT, d_ktilde, dq, dk, dv, dbeta, dr, dalpha, dd0, dS0, deta,
                            false, workspace, workspace_bytes, stream);
}

int osdn_backward_kda(int io, int B, int H, int T, int K, int V, const void *q, const void *k,
                      const void *ktilde, const void *v, const float *beta, const float *r,
                      float eta, const float *d0, const float *alpha_k, const float *S0,
                      const void *d_o, const float *d_ST, const float *d_dT,
                      const void *d_ktilde, void *dq, void *dk, void *dv, float *dbeta,
                      float *dr, float *dalpha_k, float *dd0, float *dS0, float *deta,
                      void *workspace, size_t workspace_bytes, void *stream) {
    return backward_checked(io, B, H, T, K, V, q, k, ktilde, v, beta, r, eta, d0, alpha_k, S0,
                            d_o, d_ST, d_dT, d_ktilde, dq, dk, dv, dbeta, dr, dalpha_k, dd0, dS0,
                            deta, true, workspace, workspace_bytes, stream);
}

int osdn_chunk_fwd_kda(int io, int B, int H, int T, int K, int V, const void *q, const void *k,
                       const void *ktilde, const void *v, const float *beta,
                       const float *alpha_k, const float *S0, void *o, float *ST,
                       void *workspace, size_t workspace_bytes, void *stream) {
    if (io != OSDN_F32 && io != OSDN_BF16) return OSDN_ERR_DTYPE;
    if (!dims_ok(B, H, T) || !width_ok(K) || !width_ok(V)) return OSDN_ERR_DIMS;
    if (io == OSDN_BF16 && T > kMaxTcTokens) return OSDN_ERR_DIMS;
    if (!workspace || workspace_bytes < osdn_chunk_fwd_kda_workspace_bytes(io, B, H, T, K, V))
        return OSDN_ERR_WORKSPACE;
    const size_t BH = (size_t)B * H;
    if (BH == 0) return OSDN_OK;
    if (T > 0 && (!q || !k || !ktilde || !v || !beta || !o)) return OSDN_ERR_NULL;
    if (misaligned(q) || misaligned(k) || misaligned(ktilde) || misaligned(v) ||
        misaligned(beta) || misaligned(alpha_k) || misaligned(S0) || misaligned(o) ||
        misaligned(ST) || misaligned(workspace))
        return OSDN_ERR_ALIGN;
    const size_t es = io_bytes(io);
    const size_t kb = BH * (size_t)T * K * es, vb = BH * (size_t)T * V * es;
    const size_t sb = BH * (size_t)V * K * 4, gb = BH * (size_t)T * 4;
    const size_t ab = BH * (size_t)T * K * 4;
    const void *ins[7] = {q, k, ktilde, v, beta, alpha_k, S0};
    const size_t insz[7] = {kb, kb, kb, vb, gb, ab, sb};
    for (int i = 0; i < 7; ++i)
        if (overlap(o, vb, ins[i], insz[i]) || overlap(ST, sb, ins[i], insz[i]) ||
            overlap(workspace, workspace_bytes, ins[i], insz[i]))
            return OSDN_ERR_ALIAS;
    if (overlap(o, vb, ST, sb) || overlap(workspace, workspace_bytes, o, vb) ||
        overlap(workspace, workspace_bytes, ST, sb))
        return OSDN_ERR_ALIAS;
    int dev = check_device();
    if (dev != OSDN_OK) return dev;
    cudaError_t e;
    if (T == 0)
        e = osdn::fill_state_launch(ST ? sb / 4 : 0, S0, 0.0f, ST, (cudaStream_t)stream);
    else if (io == OSDN_BF16 && alpha_k)  // tensor cores, the decay folded in per channel
        e = osdn::delta_tc_kda_launch((int)BH, T, K, V, q, k, ktilde, v, beta, alpha_k, S0, o, ST,
                                      static_cast<char *>(workspace) + kStatusBytes,
                                      static_cast<int *>(workspace), (cudaStream_t)stream);
    else if (io == OSDN_BF16)  // no decay: the scalar-gate tensor-core path without a gate
        e = osdn::delta_tc_launch((int)BH, T, K, V, q, k, ktilde, v, beta, nullptr, S0, o, ST,
                                  static_cast<char *>(workspace) + kStatusBytes,
                                  static_cast<int *>(workspace), (cudaStream_t)stream);
    else
        e = osdn::delta_simt_kda_launch(io, (int)BH, T, K, V, q, k, ktilde, v, beta, alpha_k, S0,
                                        o, ST, (cudaStream_t)stream);
    return e == cudaSuccess ? OSDN_OK : OSDN_ERR_CUDA;
}

}  // extern "C"
