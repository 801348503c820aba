// read_probe.cu -- a measurement aid, not part of the GEMM: the streaming-read
// ceiling of one launch in a chain of launches.
//
// It moves `bytes` of global memory into shared memory exactly as the decode
// kernels move their weights -- 1-D bulk copies of 16 KB into a ring of
// shared-memory slots guarded by mbarriers, one CTA per SM each taking one
// contiguous share, programmatic dependent launch signalled at the start and
// the wait for the previous kernel taken only before the one store of the
// launch -- and does no arithmetic on what it reads.  Timing a chain of these
// launches over distinct buffers gives the bandwidth a kernel of this shape
// can reach per launch at a given size, the ceiling the decode GEMM's
// weight stream is measured against (page "Triton Kernel Matches
// bitsandbytes: Why Both Lose to Math", section "Roofline First": a kernel that
// only has to read its bytes once is bounded by the copy rate).
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace w4a16 {
namespace {

constexpr int kChunk = 16 * 1024;
constexpr int kSlots = 6;

__global__ void __launch_bounds__(64, 2)
read_probe_kernel(const uint8_t *src, size_t bytes, uint32_t *sink, int *status,
                  unsigned long long timeout_ns)
{
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ uint64_t full[kSlots], empty[kSlots];
    const size_t chunks = (bytes + kChunk - 1) / kChunk;
    const size_t c0 = chunks * blockIdx.x / gridDim.x, c1 = chunks * (blockIdx.x + 1) / gridDim.x;
    const int n = (int)(c1 - c0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            for (int i = 0; i < n; ++i) {
                const int s = i % kSlots;
                if (i >= kSlots && !mbar_wait_bounded(&empty[s], ((i / kSlots) - 1) & 1, timeout_ns))
                    report_status(status, W4A16_ERR_TIMEOUT);
                const size_t off = (c0 + i) * (size_t)kChunk;
                const uint32_t len = (uint32_t)(bytes - off < (size_t)kChunk ? bytes - off : kChunk);
                mbar_arrive_expect_tx(&full[s], len);
                bulk_load(smem_u32(ring + s * kChunk), src + off, len, smem_u32(&full[s]), pol);
            }
        }
        return;
    }
    // one consumer warp: takes each chunk as it lands, folds one word of it
    uint32_t acc = 0;
    for (int i = 0; i < n; ++i) {
        const int s = i % kSlots;
        if (!mbar_wait_bounded(&full[s], (i / kSlots) & 1, timeout_ns))
            report_status(status, W4A16_ERR_TIMEOUT);
        acc ^= reinterpret_cast<const uint32_t *>(ring + s * kChunk)[lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    pdl_wait();   // the store waits for the previous kernel, as a GEMM's output would
    if (lane == 0) sink[blockIdx.x] = acc;
}

}  // namespace

cudaError_t launch_read_probe(const void *src, size_t bytes, uint32_t *sink, int ctas, bool pdl,
                              int *status, cudaStream_t stream) {
    const int smem = kSlots * kChunk;
    cudaError_t e = ensure_dynamic_smem((const void *)read_probe_kernel, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(ctas, 1, 1);
    lc.blockDim = dim3(64, 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = &attr;
    lc.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&lc, read_probe_kernel, static_cast<const uint8_t *>(src), bytes,
                              sink, status, 1000000000ull);
}

}  // namespace w4a16
