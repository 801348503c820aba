// common.cuh -- internal declarations shared by the libw4a16 translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "w4a16.h"

namespace w4a16 {

// Device-side status word: kernels with bounded waits receive its address and
// write W4A16_ERR_TIMEOUT there (first writer wins) when a wait gives up;
// w4a16_get_kernel_status swaps it with zero (one atomic exchange on the
// device, after the work queued on `stream`).  The word lives in api.cu (one
// copy per device, shared by every stream); these host helpers are the only
// way to reach it.
cudaError_t kernel_status_address(int **ptr);                             // current device
cudaError_t kernel_status_read_clear(int *value, cudaStream_t stream);    // synchronous

__device__ __forceinline__ void report_status(int *status, int code) {
    atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- launchers
struct GemmArgs {
    const uint16_t *x;
    const uint32_t *packed;
    const uint16_t *scales;
    const uint16_t *zeros;
    uint16_t *out;
    int M, N, K, group;
};

// A grouped launch: E GEMMs of one shape (MoE experts), each with its own
// x, weights and out.  The pointer tables travel in the kernel parameters.
constexpr int kMaxExperts = W4A16_MAX_EXPERTS;
struct GroupedGemmArgs {
    int E;
    const uint16_t *x[kMaxExperts];
    const uint32_t *packed[kMaxExperts];
    const uint16_t *scales[kMaxExperts];
    const uint16_t *zeros[kMaxExperts];
    uint16_t *out[kMaxExperts];
    int M, N, K, group;
};

// One call of the stream decode kernel (decode_stream.cu): E GEMMs of one
// shape (E = 1 for a plain GEMM), natural or repacked weights.  For repacked
// weights w[e] is the block array of w4a16_repack and s, z are unused.
struct StreamCall {
    int E;
    const uint16_t *x[kMaxExperts];
    const uint32_t *w[kMaxExperts];
    const uint16_t *s[kMaxExperts];
    const uint16_t *z[kMaxExperts];
    uint16_t *out[kMaxExperts];
    int M, N, K, group;
    bool permuted;
};

// Each returns cudaSuccess or the launch error; they never synchronize.
cudaError_t launch_quantize_pack(const uint16_t *W, int K, int N, int group, bool symmetric,
                                 uint32_t *packed, uint16_t *scales, uint16_t *zeros,
                                 cudaStream_t stream);
cudaError_t launch_dequantize(const uint32_t *packed, const uint16_t *scales,
                              const uint16_t *zeros, uint16_t *W_out, int K, int N,
                              int group, cudaStream_t stream);
cudaError_t launch_quantize_pack_bf16(const uint16_t *W, int K, int N, int group,
                                      uint32_t *packed, uint16_t *scales, uint16_t *zeros,
                                      cudaStream_t stream);
cudaError_t launch_dequantize_bf16(const uint32_t *packed, const uint16_t *scales,
                                   const uint16_t *zeros, uint16_t *W_out, int K, int N,
                                   int group, cudaStream_t stream);
// The pre-permuted (repacked) weight layout: support check, size, and the
// natural -> repacked transform (quant.cu).
bool repack_supported(int K, int N, int group);
size_t repacked_bytes(int K, int N, int group);
cudaError_t launch_repack(const uint32_t *packed, const uint16_t *scales, const uint16_t *zeros,
                          int K, int N, int group, void *out, cudaStream_t stream);
// Decode path: cfg already fully resolved (split_k, warps_k, warps_n, steps > 0).
// Returns cudaErrorNotSupported for a configuration with no compiled kernel.
cudaError_t launch_decode(const GemmArgs &a, const w4a16_config &cfg, cudaStream_t stream);
// Grouped decode (registers variant, M <= 16): one launch over all E GEMMs.
cudaError_t launch_decode_grouped(const GroupedGemmArgs &a, const w4a16_config &cfg,
                                  cudaStream_t stream);
bool decode_config_supported(const w4a16_config &cfg, int M);
int decode_steps_per_batch(int group);
// Resident CTAs per SM of the decode kernel that `cfg` selects (occupancy
// query on the current device; a fixed estimate when no GPU is present).
int decode_ctas_per_sm(const w4a16_config &cfg, int M, int group);
// Decode path, TMA variant (decode_tma.cu).
bool decode_tma_supported(const w4a16_config &cfg, int group);
int decode_tma_smem_bytes(const w4a16_config &cfg, int M, int group);
cudaError_t launch_decode_tma(const GemmArgs &a, const w4a16_config &cfg, cudaStream_t stream);
// Decode path, stream variant (decode_stream.cu): cfg.warps_n strips per
// tile (1, 2 or 4), cfg.split_k 1 (whole tiles per CTA) or 2 (stream-K
// shares), cfg.ctas CTAs (0: one per SM).
// The warp-stream decode kernel (decode_warp.cu, M <= 4): every warp streams
// its own run of 32-column x 512-k units through a private ring.
bool decode_warp_supported(int M, int N, int K, int group, int ctas);
cudaError_t launch_decode_warp(const GemmArgs &a, const w4a16_config &cfg, cudaStream_t stream);
// The same design on repacked blocks (one bulk copy per unit), for one or up
// to kMaxExperts GEMMs of one shape (M <= 8).
bool decode_warp_perm_supported(int M, int N, int K, int group, int experts, int ctas);
struct StreamCall;
cudaError_t launch_decode_warp_perm(const StreamCall &call, const w4a16_config &cfg,
                                    cudaStream_t stream);
bool decode_stream_supported(int M, int N, int K, int group, int bns, bool perm);
int decode_stream_stage_k(int bns);   // k per stage of a tile of bns strips
cudaError_t launch_decode_stream(const StreamCall &call, const w4a16_config &cfg,
                                 cudaStream_t stream);
// The same kernel with stream-K shares and its scratch in a fixed device array
// of this library (w4a16_gemm_noalloc): nothing is allocated.  `need_*` report
// the scratch a call asked for (cudaErrorInvalidValue when it is too large).
struct NoAllocResult {
    cudaError_t err;
    size_t need_counters, need_partials;
};
NoAllocResult launch_decode_stream_noalloc(const StreamCall &call, int bns, bool pdl,
                                           cudaStream_t stream);
// Prefill path (tcgen05).  Returns cudaErrorNotSupported if unavailable.
cudaError_t launch_prefill(const GemmArgs &a, const w4a16_config &cfg, cudaStream_t stream);
bool prefill_config_supported(const w4a16_config &cfg, int M, int N, int K, int group);

// Measurement aid (read_probe.cu): stream `bytes` into shared memory the way
// the decode kernels stream their weights, with no arithmetic; one word per
// CTA to sink[ctas].
cudaError_t launch_read_probe(const void *src, size_t bytes, uint32_t *sink, int ctas, bool pdl,
                              int *status, cudaStream_t stream);

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per (device, kernel): the attribute belongs to the device's
// context, so a process that drives several GPUs sets it on each.
cudaError_t ensure_dynamic_smem(const void *kernel, int bytes);

// Hardware facts used by the planner (queried once per device, cached).
struct DeviceInfo {
    int sm_count;
    int cc_major, cc_minor;
};
const DeviceInfo &device_info();   // host, current device (queried once per device);
                                   // falls back to GB300 numbers when no GPU
int *device_status_word();         // the status word's device address on the
                                   // current device (looked up once per device)

// ------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t bits) {
    // (a & mask) | bits in one LOP3 (truth table 0xEA)
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(bits));
    return r;
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t hadd2_u32(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// The same three operations on bfloat16 pairs (round to nearest even).
__device__ __forceinline__ uint32_t bsub2_u32(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t badd2_u32(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t bmul2_u32(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// griddepcontrol (programmatic dependent launch); no-ops without the launch
// attribute.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace w4a16
