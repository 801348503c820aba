// api.cu -- the extern "C" boundary of libw4a16.so: argument validation,
// launch planning (dispatch), error reporting.  Every compute step runs in the
// kernels of quant.cu, decode.cu and prefill.cu.
#include <atomic>
#include <mutex>
#include <set>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>
#include <string>

#include "common.cuh"

namespace w4a16 {

__device__ int g_kernel_status = 0;
__device__ int g_kernel_status_taken = 0;

cudaError_t kernel_status_address(int **ptr) {
    return cudaGetSymbolAddress(reinterpret_cast<void **>(ptr), g_kernel_status);
}

namespace {
// Swaps the status word with zero in one atomic step, so a status set by a
// kernel between a read and a clear can never be lost.
__global__ void status_take_kernel() { g_kernel_status_taken = atomicExch(&g_kernel_status, 0); }
}  // namespace

cudaError_t kernel_status_read_clear(int *value, cudaStream_t stream) {
    static std::mutex mu;   // one taker at a time: the snapshot word is shared
    std::lock_guard<std::mutex> lock(mu);
    status_take_kernel<<<1, 1, 0, stream>>>();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbolAsync(value, g_kernel_status_taken, sizeof(int), 0,
                                  cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

namespace {

thread_local std::string t_last_error;

w4a16_status fail(w4a16_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
w4a16_status fail(w4a16_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

w4a16_status cuda_fail(cudaError_t e, const char *what) {
    return fail(W4A16_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

constexpr long long kMaxElems = (1ll << 31) - 1;

// Shape rules common to all entry points (pointer checks done by callers).
w4a16_status check_shape(int M, int N, int K, int group) {
    if (M < 0 || N < 0 || K < 0)
        return fail(W4A16_ERR_INVALID_ARG, "negative size (M=%d N=%d K=%d)", M, N, K);
    if (group <= 0 || group % 8 != 0)
        return fail(W4A16_ERR_INVALID_ARG, "group must be a positive multiple of 8 (got %d)", group);
    if (group % 32 != 0 || group > 1024)
        return fail(W4A16_ERR_UNSUPPORTED,
                    "group %d: this library implements groups that are multiples of 32 up to 1024",
                    group);
    if (K == 0 || K % group != 0)
        return fail(W4A16_ERR_INVALID_ARG, "K (%d) must be a positive multiple of group (%d)", K,
                    group);
    if (N % 4 != 0)
        return fail(W4A16_ERR_MISALIGNED,
                    "N (%d) must be a multiple of 4 so that packed rows are 16-byte aligned", N);
    if ((long long)M * K > kMaxElems || (long long)K * N > kMaxElems ||
        (long long)M * N > kMaxElems)
        return fail(W4A16_ERR_UNSUPPORTED, "an operand exceeds 2^31-1 elements");
    return W4A16_OK;
}

DeviceInfo query_device() {
    DeviceInfo d{152, 10, 3};   // GB300 when no GPU is visible (host-only planning)
    int dev = 0, n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) {
        cudaGetLastError();
        return d;
    }
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return d;
    }
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) d.sm_count = v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess) d.cc_major = v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess) d.cc_minor = v;
    cudaGetLastError();
    return d;
}

// -------------------------------------------------------------- planning
// Decode path.  A column tile of 32*warps_n columns is covered by
// warps_k * split warps along K, each streaming `steps` 32-row steps.  The
// choice aims at enough CTAs to fill the SMs about twice (so that every SM has
// loads from several warps in flight) with the fewest CTAs per cluster.
void plan_decode(int M, int N, int K, int group, int sm_count, w4a16_config &c) {
    const int U = decode_steps_per_batch(group);
    if (c.warps_n <= 0) c.warps_n = M > 8 ? 2 : 1;
    if (c.warps_k <= 0) c.warps_k = c.warps_n == 1 ? 8 : (c.warps_n == 2 ? 4 : 2);
    const int strips = (N + 32 * c.warps_n - 1) / (32 * c.warps_n);
    const int total_steps = K / 32;
    if (c.split_k <= 0 && c.steps <= 0) {
        // Most CTAs that still fit in one wave; ties go to the smaller cluster.
        const long long capacity = (long long)sm_count * decode_ctas_per_sm(c, M, group);
        int best_split = 0, best_steps = 0;
        long long best_ctas = -1;
        for (int s = 1; s <= 8; ++s) {
            int st = (total_steps + c.warps_k * s - 1) / (c.warps_k * s);
            st = (st + U - 1) / U * U;
            const int s_eff = (total_steps + c.warps_k * st - 1) / (c.warps_k * st);
            const long long ctas = (long long)strips * s_eff;
            const bool fits = ctas <= capacity;
            const bool better = best_ctas < 0 ||
                                (fits && (best_ctas > capacity || ctas > best_ctas)) ||
                                (!fits && best_ctas > capacity && ctas < best_ctas);
            if (better) {
                best_split = s_eff;
                best_steps = st;
                best_ctas = ctas;
            }
        }
        c.split_k = best_split;
        c.steps = best_steps;
    } else if (c.steps <= 0) {
        int st = (total_steps + c.warps_k * c.split_k - 1) / (c.warps_k * c.split_k);
        c.steps = (st + U - 1) / U * U;
    } else if (c.split_k <= 0) {
        c.split_k = (total_steps + c.warps_k * c.steps - 1) / (c.warps_k * c.steps);
    }
}

// Decode path, TMA variant: a CTA covers 32*warps_n columns and `steps`
// 256-row stages of K; split_k CTAs of a cluster cover K.  The choice
// minimizes the stages streamed by the busiest SM, then the cluster size.
void plan_decode_tma(int M, int N, int K, int group, int sm_count, w4a16_config &c) {
    if (c.warps_n <= 0) c.warps_n = 4;
    const int BN = 32 * c.warps_n;
    const int tiles = (N + BN - 1) / BN;
    const int total = (K / 8 + 31) / 32;    // 256-row stages
    if (c.split_k <= 0 && c.steps <= 0) {
        // prefer configurations that leave room for a second CTA per SM
        // (about half of the shared memory), then the smallest busiest-SM load
        long long best_cost = -1;
        for (int s = 1; s <= 8; ++s) {
            const int st = (total + s - 1) / s;
            const int s_eff = (total + st - 1) / st;
            w4a16_config t = c;
            t.split_k = s_eff;
            t.steps = st;
            const bool fits_half = decode_tma_smem_bytes(t, M, group) <= 113 * 1024;
            const long long ctas = (long long)tiles * s_eff;
            const long long cost = ((ctas + sm_count - 1) / sm_count * st) * 2 + (fits_half ? 0 : 1);
            if (best_cost < 0 || cost < best_cost) {
                best_cost = cost;
                c.split_k = s_eff;
                c.steps = st;
            }
        }
    } else if (c.steps <= 0) {
        c.steps = (total + c.split_k - 1) / c.split_k;
    } else if (c.split_k <= 0) {
        c.split_k = (total + c.steps - 1) / c.steps;
    }
}

// Decode path, stream variant: tiles of 32*warps_n columns cut into 16 KB
// stages; split_k = 1 gives every CTA whole tiles (no shared tile, no
// scratch), 2 gives every CTA an equal share of all stages (stream-K).
// Measured on GB300 (repacked weights, CUDA graph + PDL; 4096 x 4096,
// 4096 x 14336 and 2048 x 768 at M = 1..16): the narrowest tiles that fit
// (32 columns up to M = 8, 64 above) and whole tiles per CTA were the fastest
// at every shape and M -- stream-K shares were 1.5-2x slower, even where
// whole tiles leave SMs idle.
void plan_decode_stream(int M, int N, int K, int group, int experts, bool perm, int sm_count,
                        w4a16_config &c) {
    (void)experts;
    (void)sm_count;
    if (c.warps_n <= 0) {
        c.warps_n = M <= 8 ? 1 : 2;
        while (c.warps_n < 4 && !decode_stream_supported(M, N, K, group, c.warps_n, perm))
            c.warps_n *= 2;
    }
    if (c.split_k <= 0) c.split_k = 1;
}

// Measured dispatch table (GB300, group 128, one call per distinct weight copy
// in a CUDA graph with programmatic dependent launch): the fastest decode
// configuration for the projection shapes of the benchmark workloads (the TMA
// variant with the zero-free step at M <= 8).  Interleaved runs in one process
// decided the close rows: 4096 x 4096 takes the TMA variant at M <= 2 (1-2%
// ahead) and the warp-stream variant at M = 3..4 (2% ahead).
struct TableEntry {
    int K, N, m_max;        // shape and the largest M the row covers
    w4a16_config cfg;
};
constexpr TableEntry kDecodeTable[] = {
    // K      N      M<=   path split warps_k warps_n steps tile flags variant
    {4096, 4096, 2, {1, 8, 4, 2, 2, 0, 0, W4A16_DECODE_TMA}},
    {4096, 4096, 4, {1, 0, 0, 0, 0, 0, 0, W4A16_DECODE_WARP}},
    {4096, 4096, 8, {1, 2, 8, 1, 8, 0, 0, W4A16_DECODE_REGISTERS}},
    {4096, 4096, 16, {1, 1, 8, 1, 16, 0, 0, W4A16_DECODE_REGISTERS}},
    {4096, 14336, 16, {1, 2, 4, 2, 8, 0, 0, W4A16_DECODE_TMA}},
    {14336, 4096, 8, {1, 8, 8, 4, 7, 0, 0, W4A16_DECODE_TMA}},
    {14336, 4096, 16, {1, 6, 4, 2, 10, 0, 0, W4A16_DECODE_TMA}},
    {2048, 768, 4, {1, 4, 4, 2, 4, 0, 0, W4A16_DECODE_REGISTERS}},
    {2048, 768, 16, {1, 4, 4, 1, 4, 0, 0, W4A16_DECODE_REGISTERS}},
    {768, 2048, 16, {1, 1, 8, 1, 4, 0, 0, W4A16_DECODE_REGISTERS}},
};

// The same for bfloat16 (registers and TMA variants only; measured the same
// way on bf16 weights and activations).
constexpr TableEntry kDecodeTableBf16[] = {
    // K      N      M<=   path split warps_k warps_n steps tile flags variant
    {4096, 4096, 4, {1, 8, 4, 2, 2, 0, 0, W4A16_DECODE_TMA}},
    {4096, 4096, 8, {1, 4, 16, 4, 4, 0, 0, W4A16_DECODE_TMA}},
    {4096, 4096, 16, {1, 2, 16, 2, 8, 0, 0, W4A16_DECODE_TMA}},
    {4096, 14336, 16, {1, 2, 4, 2, 8, 0, 0, W4A16_DECODE_TMA}},
    {14336, 4096, 8, {1, 8, 8, 4, 7, 0, 0, W4A16_DECODE_TMA}},
    {14336, 4096, 16, {1, 4, 16, 4, 14, 0, 0, W4A16_DECODE_TMA}},
    {2048, 768, 4, {1, 8, 8, 2, 1, 0, 0, W4A16_DECODE_TMA}},
    {2048, 768, 16, {1, 2, 8, 1, 4, 0, 0, W4A16_DECODE_REGISTERS}},
    {768, 2048, 16, {1, 1, 8, 1, 4, 0, 0, W4A16_DECODE_REGISTERS}},
};

// Grouped launches of 64 experts (measured the same way, one grouped launch
// per 64 distinct weight copies): registers variant, no split -- the experts
// already give thousands of CTAs.
constexpr TableEntry kGroupedTable[] = {
    // K      N      M<=   path split warps_k warps_n steps tile flags variant
    {2048, 768, 8, {1, 1, 4, 2, 16, 0, 0, W4A16_DECODE_REGISTERS}},
    {2048, 768, 16, {1, 1, 4, 1, 16, 0, 0, W4A16_DECODE_REGISTERS}},
    {768, 2048, 8, {1, 1, 2, 4, 12, 0, 0, W4A16_DECODE_REGISTERS}},
    {768, 2048, 16, {1, 1, 2, 2, 12, 0, 0, W4A16_DECODE_REGISTERS}},
};

bool grouped_from_table(int M, int N, int K, int group, w4a16_config &c) {
    if (group != 128 || c.split_k || c.warps_k || c.warps_n || c.steps) return false;
    for (const TableEntry &e : kGroupedTable)
        if (e.K == K && e.N == N && M <= e.m_max) {
            const int flags = c.flags;
            c = e.cfg;
            c.flags = flags;
            return true;
        }
    return false;
}

// Fill an all-automatic decode request from the table of its dtype; false if
// no row fits.
bool decode_from_table(int M, int N, int K, int group, w4a16_config &c) {
    if (group != 128 || c.variant != W4A16_DECODE_AUTO || c.split_k || c.warps_k || c.warps_n ||
        c.steps)
        return false;
    const bool bf = c.dtype == W4A16_DTYPE_BF16;
    const TableEntry *rows = bf ? kDecodeTableBf16 : kDecodeTable;
    const size_t n = bf ? sizeof(kDecodeTableBf16) / sizeof(TableEntry)
                        : sizeof(kDecodeTable) / sizeof(TableEntry);
    for (size_t i = 0; i < n; ++i) {
        const TableEntry &e = rows[i];
        if (e.K == K && e.N == N && M <= e.m_max) {
            const int flags = c.flags, dtype = c.dtype;
            c = e.cfg;
            c.flags = flags;
            c.dtype = dtype;
            return true;
        }
    }
    return false;
}

bool tma_variant_possible(int N, int group) {
    return (group == 32 || group == 64 || group == 128 || group == 256) && N % 8 == 0;
}

// Crossover between the decode path and the tcgen05 prefill path, in rows of x
// (measured on GB300: at M = 16 the decode kernels are still ahead).
constexpr int kDecodeMaxM = 16;

// Rows of x per prefill CTA (measured on GB300): 256 from M = 256 up; below,
// all of M in one tile -- except that for M <= 64 with fewer 128-column tiles
// than SMs, a 128-row tile (one CTA per SM) beats narrow tiles two to an SM.
int default_tile_m(int M, int N) {
    if (M >= 256) return 256;
    const int rounded = ((M + 15) / 16) * 16;
    if (rounded <= 64 && (N + 127) / 128 < device_info().sm_count) return 128;
    return rounded;
}

w4a16_status make_plan(int M, int N, int K, int group, const w4a16_config *req,
                       w4a16_config &c) {
    w4a16_status st = check_shape(M, N, K, group);
    if (st != W4A16_OK) return st;
    c = req ? *req : w4a16_config{};
    if (c.dtype != W4A16_DTYPE_F16 && c.dtype != W4A16_DTYPE_BF16)
        return fail(W4A16_ERR_INVALID_ARG, "unknown dtype %d", c.dtype);
    const bool bf = c.dtype == W4A16_DTYPE_BF16;
    if (c.path == W4A16_PATH_AUTO) {
        c.path = W4A16_PATH_DECODE;
        if (M > kDecodeMaxM) {
            w4a16_config pc = c;
            pc.path = W4A16_PATH_PREFILL;
            if (pc.tile_m <= 0) pc.tile_m = default_tile_m(M, N);
            if (prefill_config_supported(pc, M, N, K, group)) c.path = W4A16_PATH_PREFILL;
        }
    }
    if (c.path == W4A16_PATH_DECODE) {
        if (M <= 16) decode_from_table(M, N, K, group, c);
        // bfloat16 runs on the registers and TMA variants; a table row for
        // another variant falls back to the TMA planner
        if (bf && c.variant != W4A16_DECODE_AUTO && c.variant != W4A16_DECODE_REGISTERS &&
            c.variant != W4A16_DECODE_TMA) {
            if (req && req->variant == c.variant)
                return fail(W4A16_ERR_UNSUPPORTED,
                            "bfloat16 decode: registers or TMA variant (variant %d requested)",
                            c.variant);
            const int flags = c.flags;
            c = w4a16_config{};
            c.path = W4A16_PATH_DECODE;
            c.flags = flags;
            c.dtype = W4A16_DTYPE_BF16;
        }
        if (c.variant == W4A16_DECODE_AUTO)
            c.variant = tma_variant_possible(N, group) ? W4A16_DECODE_TMA : W4A16_DECODE_REGISTERS;
        if (c.variant == W4A16_DECODE_TMA) {
            plan_decode_tma(M, N, K, group, device_info().sm_count, c);
            if (!tma_variant_possible(N, group) || !decode_tma_supported(c, group) ||
                (long long)c.steps * 256 * c.split_k < K)
                return fail(W4A16_ERR_UNSUPPORTED,
                            "TMA decode configuration not available (split_k=%d warps_n=%d "
                            "steps=%d, group=%d, N=%d)",
                            c.split_k, c.warps_n, c.steps, group, N);
        } else if (c.variant == W4A16_DECODE_STREAM) {
            plan_decode_stream(M, N, K, group, 1, false, device_info().sm_count, c);
            if (M > 16 || !decode_stream_supported(M, N, K, group, c.warps_n, false) ||
                c.split_k < 1 || c.split_k > 2 || c.ctas < 0)
                return fail(W4A16_ERR_UNSUPPORTED,
                            "stream decode configuration not available (M=%d warps_n=%d "
                            "split_k=%d ctas=%d, group=%d, N=%d)",
                            M, c.warps_n, c.split_k, c.ctas, group, N);
        } else if (c.variant == W4A16_DECODE_WARP) {
            if (!decode_warp_supported(M, N, K, group, c.ctas) || c.ctas < 0)
                return fail(W4A16_ERR_UNSUPPORTED,
                            "warp-stream decode not available (M=%d N=%d K=%d group=%d)", M, N,
                            K, group);
        } else if (c.variant == W4A16_DECODE_REGISTERS) {
            plan_decode(M, N, K, group, device_info().sm_count, c);
            if (!decode_config_supported(c, M) || c.steps % decode_steps_per_batch(group) != 0 ||
                (long long)c.warps_k * c.steps * 4 * c.split_k < K / 8)
                return fail(W4A16_ERR_UNSUPPORTED,
                            "decode configuration not available (split_k=%d warps_k=%d "
                            "warps_n=%d steps=%d)",
                            c.split_k, c.warps_k, c.warps_n, c.steps);
        } else {
            return fail(W4A16_ERR_INVALID_ARG, "unknown decode variant %d", c.variant);
        }
    } else if (c.path == W4A16_PATH_PREFILL) {
        if (c.tile_m <= 0) c.tile_m = default_tile_m(M, N);
        if (c.variant <= 0) c.variant = W4A16_PREFILL_A_TMEM;
        // measured: 4 dequantizing warps, on both kernels -- 1-3% ahead of 8
        // at M = 32..4096 on both prefill shapes; fewer busy warps also draw
        // less power, so the clock sits higher under the power cap
        if (c.warps_k <= 0) c.warps_k = 4;
        if (!prefill_config_supported(c, M, N, K, group))
            return fail(W4A16_ERR_UNSUPPORTED, "prefill path not available for M=%d N=%d K=%d "
                        "group=%d tile_m=%d", M, N, K, group, c.tile_m);
    } else {
        return fail(W4A16_ERR_INVALID_ARG, "unknown path %d", c.path);
    }
    return W4A16_OK;
}

// Thread-private cache of resolved plans.  A decode loop repeats a handful of
// (shape, request) pairs; planning (table lookup, the planners' searches,
// occupancy queries) then runs once per pair instead of once per call.  Only
// successful plans are kept; a plan depends on the device, the shape and the
// request, which together form the key.
struct PlanKey {
    int dev, M, N, K, group, has_req;
    w4a16_config req;
};

w4a16_status cached_plan(int M, int N, int K, int group, const w4a16_config *req,
                         w4a16_config &c) {
    PlanKey key;
    memset(&key, 0, sizeof key);
    if (cudaGetDevice(&key.dev) != cudaSuccess) {
        cudaGetLastError();
        key.dev = -1;
    }
    key.M = M;
    key.N = N;
    key.K = K;
    key.group = group;
    key.has_req = req != nullptr;
    if (req) key.req = *req;
    struct Entry {
        PlanKey key;
        w4a16_config plan;
        bool valid;
    };
    constexpr int kEntries = 64;
    static thread_local Entry cache[kEntries];
    uint64_t h = 0xCBF29CE484222325ull;
    const unsigned char *b = reinterpret_cast<const unsigned char *>(&key);
    for (size_t i = 0; i < sizeof key; ++i) h = (h ^ b[i]) * 0x100000001B3ull;
    Entry &e = cache[(h >> 29) & (kEntries - 1)];
    if (e.valid && memcmp(&e.key, &key, sizeof key) == 0) {
        c = e.plan;
        return W4A16_OK;
    }
    const w4a16_status st = make_plan(M, N, K, group, req, c);
    if (st == W4A16_OK) {
        e.key = key;
        e.plan = c;
        e.valid = true;
    }
    return st;
}

}  // namespace

cudaError_t ensure_dynamic_smem(const void *kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    // thread-private record of the (device, kernel) pairs already set up
    constexpr int kFront = 16;
    static thread_local std::pair<int, const void *> front[kFront];
    static thread_local int front_next = 0;
    for (const auto &f : front)
        if (f.second == kernel && f.first == dev) return cudaSuccess;
    static std::mutex mu;
    static std::set<std::pair<int, const void *>> done;
    std::lock_guard<std::mutex> lock(mu);
    if (!done.count({dev, kernel})) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        done.insert({dev, kernel});
    }
    front[front_next] = {dev, kernel};
    front_next = (front_next + 1) % kFront;
    return cudaSuccess;
}

const DeviceInfo &device_info() {
    constexpr int kMaxDev = 64;
    static DeviceInfo infos[kMaxDev + 1];
    static std::atomic<bool> ready[kMaxDev + 1];
    static std::mutex mu;
    static int ndev = -1;
    static std::once_flag once;
    std::call_once(once, [] {
        if (cudaGetDeviceCount(&ndev) != cudaSuccess) ndev = 0;
        cudaGetLastError();
    });
    int dev = 0;
    // no GPU (host-only planning) uses the last slot
    if (ndev <= 0 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
        cudaGetLastError();
        dev = kMaxDev;
    }
    if (!ready[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(mu);
        if (!ready[dev].load(std::memory_order_relaxed)) {
            infos[dev] = query_device();
            ready[dev].store(true, std::memory_order_release);
        }
    }
    return infos[dev];
}

int *device_status_word() {
    static std::atomic<int *> ptrs[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    int *p = ptrs[dev].load(std::memory_order_acquire);
    if (p) return p;
    if (kernel_status_address(&p) != cudaSuccess) return nullptr;
    ptrs[dev].store(p, std::memory_order_release);
    return p;
}

}  // namespace w4a16

using namespace w4a16;

extern "C" {

w4a16_status w4a16_quantize_pack(const uint16_t *W, int K, int N, int group, uint32_t *packed,
                                 uint16_t *scales, uint16_t *zeros, cudaStream_t stream) {
    return w4a16_quantize_pack_ex(W, K, N, group, W4A16_QUANT_ASYMMETRIC, packed, scales, zeros,
                                  stream);
}

w4a16_status w4a16_quantize_pack_ex(const uint16_t *W, int K, int N, int group, int mode,
                                    uint32_t *packed, uint16_t *scales, uint16_t *zeros,
                                    cudaStream_t stream) {
    if (mode != W4A16_QUANT_ASYMMETRIC && mode != W4A16_QUANT_SYMMETRIC)
        return fail(W4A16_ERR_INVALID_ARG, "unknown quantization mode %d", mode);
    w4a16_status st = check_shape(0, N, K, group);
    if (st != W4A16_OK) return st;
    if (N == 0) return W4A16_OK;
    if (!W || !packed || !scales || !zeros)
        return fail(W4A16_ERR_INVALID_ARG, "null pointer");
    if (((uintptr_t)W & 1) || ((uintptr_t)packed & 3) || ((uintptr_t)scales & 1) ||
        ((uintptr_t)zeros & 1))
        return fail(W4A16_ERR_MISALIGNED, "pointer not aligned to its element size");
    cudaError_t e = launch_quantize_pack(W, K, N, group, mode == W4A16_QUANT_SYMMETRIC, packed,
                                         scales, zeros, stream);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "quantize_pack launch");
}

w4a16_status w4a16_dequantize(const uint32_t *packed, const uint16_t *scales,
                              const uint16_t *zeros, uint16_t *W_out, int K, int N, int group,
                              cudaStream_t stream) {
    w4a16_status st = check_shape(0, N, K, group);
    if (st != W4A16_OK) return st;
    if (N == 0) return W4A16_OK;
    if (!W_out || !packed || !scales || !zeros)
        return fail(W4A16_ERR_INVALID_ARG, "null pointer");
    if (((uintptr_t)W_out & 1) || ((uintptr_t)packed & 3) || ((uintptr_t)scales & 1) ||
        ((uintptr_t)zeros & 1))
        return fail(W4A16_ERR_MISALIGNED, "pointer not aligned to its element size");
    cudaError_t e = launch_dequantize(packed, scales, zeros, W_out, K, N, group, stream);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "dequantize launch");
}

namespace {
// Argument checks shared by the quantize / dequantize entries.
w4a16_status check_quant_args(const void *W, int K, int N, int group, const void *packed,
                              const void *scales, const void *zeros) {
    w4a16_status st = check_shape(0, N, K, group);
    if (st != W4A16_OK) return st;
    if (N == 0) return W4A16_OK;
    if (!W || !packed || !scales || !zeros) return fail(W4A16_ERR_INVALID_ARG, "null pointer");
    if (((uintptr_t)W & 1) || ((uintptr_t)packed & 3) || ((uintptr_t)scales & 1) ||
        ((uintptr_t)zeros & 1))
        return fail(W4A16_ERR_MISALIGNED, "pointer not aligned to its element size");
    return W4A16_OK;
}
}  // namespace

w4a16_status w4a16_quantize_pack_bf16(const uint16_t *W, int K, int N, int group,
                                      uint32_t *packed, uint16_t *scales, uint16_t *zeros,
                                      cudaStream_t stream) {
    w4a16_status st = check_quant_args(W, K, N, group, packed, scales, zeros);
    if (st != W4A16_OK || N == 0) return st;
    cudaError_t e = launch_quantize_pack_bf16(W, K, N, group, packed, scales, zeros, stream);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "quantize_pack_bf16 launch");
}

w4a16_status w4a16_dequantize_bf16(const uint32_t *packed, const uint16_t *scales,
                                   const uint16_t *zeros, uint16_t *W_out, int K, int N,
                                   int group, cudaStream_t stream) {
    w4a16_status st = check_quant_args(W_out, K, N, group, packed, scales, zeros);
    if (st != W4A16_OK || N == 0) return st;
    cudaError_t e = launch_dequantize_bf16(packed, scales, zeros, W_out, K, N, group, stream);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "dequantize_bf16 launch");
}

w4a16_status w4a16_plan(int M, int N, int K, int group, const w4a16_config *request,
                        w4a16_config *plan_out) {
    if (!plan_out) return fail(W4A16_ERR_INVALID_ARG, "plan_out is null");
    w4a16_config c;
    w4a16_status st = make_plan(M, N, K, group, request, c);
    if (st == W4A16_OK) *plan_out = c;
    return st;
}

w4a16_status w4a16_gemm_ex(const uint16_t *x, const uint32_t *packed, const uint16_t *scales,
                           const uint16_t *zeros, uint16_t *out, int M, int N, int K, int group,
                           const w4a16_config *cfg, cudaStream_t stream) {
    w4a16_status st = check_shape(M, N, K, group);
    if (st != W4A16_OK) return st;
    if (M == 0 || N == 0) return W4A16_OK;
    if (!x || !packed || !scales || !zeros || !out)
        return fail(W4A16_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(x) || !aligned16(packed) || !aligned16(scales) || !aligned16(zeros) ||
        !aligned16(out))
        return fail(W4A16_ERR_MISALIGNED, "x, packed, scales, zeros and out must be 16-byte "
                    "aligned");
    w4a16_config c;
    st = cached_plan(M, N, K, group, cfg, c);
    if (st != W4A16_OK) return st;
    GemmArgs a{x, packed, scales, zeros, out, M, N, K, group};
    cudaError_t e;
    if (c.path == W4A16_PATH_DECODE && c.variant == W4A16_DECODE_STREAM) {
        StreamCall sc;
        sc.E = 1;
        sc.x[0] = x;
        sc.w[0] = packed;
        sc.s[0] = scales;
        sc.z[0] = zeros;
        sc.out[0] = out;
        sc.M = M;
        sc.N = N;
        sc.K = K;
        sc.group = group;
        sc.permuted = false;
        e = launch_decode_stream(sc, c, stream);
    } else if (c.path == W4A16_PATH_DECODE && c.variant == W4A16_DECODE_WARP) {
        e = launch_decode_warp(a, c, stream);
    } else if (c.path == W4A16_PATH_DECODE) {
        e = c.variant == W4A16_DECODE_TMA ? launch_decode_tma(a, c, stream)
                                          : launch_decode(a, c, stream);
    } else {
        e = launch_prefill(a, c, stream);
    }
    if (e == cudaErrorNotSupported)
        return fail(W4A16_ERR_UNSUPPORTED, "no kernel for this configuration");
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "gemm launch");
}

w4a16_status w4a16_gemm_call(const w4a16_gemm_args *args, cudaStream_t stream) {
    if (!args) return fail(W4A16_ERR_INVALID_ARG, "args is null");
    return w4a16_gemm_ex(args->x, args->packed, args->scales, args->zeros, args->out, args->M,
                         args->N, args->K, args->group, args->cfg, stream);
}

w4a16_status w4a16_gemm(const uint16_t *x, const uint32_t *packed, const uint16_t *scales,
                        const uint16_t *zeros, uint16_t *out, int M, int N, int K, int group,
                        cudaStream_t stream) {
    return w4a16_gemm_ex(x, packed, scales, zeros, out, M, N, K, group, nullptr, stream);
}

w4a16_status w4a16_gemm_grouped(int E, const uint16_t *const *x, const uint32_t *const *packed,
                                const uint16_t *const *scales, const uint16_t *const *zeros,
                                uint16_t *const *out, int M, int N, int K, int group,
                                const w4a16_config *cfg, cudaStream_t stream) {
    if (E < 1 || E > W4A16_MAX_EXPERTS)
        return fail(W4A16_ERR_INVALID_ARG, "E=%d: 1..%d experts per grouped call", E,
                    W4A16_MAX_EXPERTS);
    if (!x || !packed || !scales || !zeros || !out)
        return fail(W4A16_ERR_INVALID_ARG, "null pointer table");
    w4a16_status st = check_shape(M, N, K, group);
    if (st != W4A16_OK) return st;
    for (int e = 0; e < E; ++e) {
        if (!x[e] || !packed[e] || !scales[e] || !zeros[e] || !out[e])
            return fail(W4A16_ERR_INVALID_ARG, "null pointer (expert %d)", e);
        if (!aligned16(x[e]) || !aligned16(packed[e]) || !aligned16(scales[e]) ||
            !aligned16(zeros[e]) || !aligned16(out[e]))
            return fail(W4A16_ERR_MISALIGNED, "expert %d: x, packed, scales, zeros and out must "
                        "be 16-byte aligned", e);
    }
    if (M == 0 || N == 0) return W4A16_OK;
    if (cfg && cfg->dtype != W4A16_DTYPE_F16 && M <= kDecodeMaxM)
        return fail(W4A16_ERR_UNSUPPORTED, "grouped GEMM at M <= %d: fp16 only", kDecodeMaxM);
    if (M > kDecodeMaxM) {
        // prefill-sized experts: one launch each (the tensor-core path is
        // already compute-bound per expert)
        for (int e = 0; e < E; ++e) {
            st = w4a16_gemm_ex(x[e], packed[e], scales[e], zeros[e], out[e], M, N, K, group, cfg,
                               stream);
            if (st != W4A16_OK) return st;
        }
        return W4A16_OK;
    }
    w4a16_config c = cfg ? *cfg : w4a16_config{};
    if ((c.path != W4A16_PATH_AUTO && c.path != W4A16_PATH_DECODE) ||
        (c.variant != W4A16_DECODE_AUTO && c.variant != W4A16_DECODE_REGISTERS &&
         c.variant != W4A16_DECODE_STREAM))
        return fail(W4A16_ERR_UNSUPPORTED,
                    "grouped GEMM: decode path, registers or stream variant only");
    if (c.variant == W4A16_DECODE_STREAM) {
        c.path = W4A16_PATH_DECODE;
        plan_decode_stream(M, N, K, group, E, false, device_info().sm_count, c);
        if (!decode_stream_supported(M, N, K, group, c.warps_n, false) || c.split_k < 1 ||
            c.split_k > 2 || c.ctas < 0)
            return fail(W4A16_ERR_UNSUPPORTED, "grouped stream configuration not available "
                        "(warps_n=%d split_k=%d, group=%d, N=%d)", c.warps_n, c.split_k, group, N);
        StreamCall sc;
        sc.E = E;
        for (int e = 0; e < E; ++e) {
            sc.x[e] = x[e];
            sc.w[e] = packed[e];
            sc.s[e] = scales[e];
            sc.z[e] = zeros[e];
            sc.out[e] = out[e];
        }
        sc.M = M;
        sc.N = N;
        sc.K = K;
        sc.group = group;
        sc.permuted = false;
        cudaError_t err = launch_decode_stream(sc, c, stream);
        if (err == cudaErrorNotSupported)
            return fail(W4A16_ERR_UNSUPPORTED, "no kernel for this configuration");
        return err == cudaSuccess ? W4A16_OK : cuda_fail(err, "grouped gemm launch");
    }
    c.path = W4A16_PATH_DECODE;
    c.variant = W4A16_DECODE_REGISTERS;
    // measured rows for the expert shapes; otherwise the E experts' column
    // tiles fill the GPU together: plan as one GEMM with E * N columns
    if (E == W4A16_MAX_EXPERTS) grouped_from_table(M, N, K, group, c);
    plan_decode(M, N * E, K, group, device_info().sm_count, c);
    if (!decode_config_supported(c, M) || c.steps % decode_steps_per_batch(group) != 0 ||
        (long long)c.warps_k * c.steps * 4 * c.split_k < K / 8)
        return fail(W4A16_ERR_UNSUPPORTED, "grouped decode configuration not available "
                    "(split_k=%d warps_k=%d warps_n=%d steps=%d)",
                    c.split_k, c.warps_k, c.warps_n, c.steps);
    GroupedGemmArgs a;
    a.E = E;
    for (int e = 0; e < E; ++e) {
        a.x[e] = x[e];
        a.packed[e] = packed[e];
        a.scales[e] = scales[e];
        a.zeros[e] = zeros[e];
        a.out[e] = out[e];
    }
    a.M = M;
    a.N = N;
    a.K = K;
    a.group = group;
    cudaError_t err = launch_decode_grouped(a, c, stream);
    if (err == cudaErrorNotSupported)
        return fail(W4A16_ERR_UNSUPPORTED, "no kernel for this configuration");
    return err == cudaSuccess ? W4A16_OK : cuda_fail(err, "grouped gemm launch");
}

size_t w4a16_repacked_bytes(int K, int N, int group) { return repacked_bytes(K, N, group); }

w4a16_status w4a16_repack(const uint32_t *packed, const uint16_t *scales, const uint16_t *zeros,
                          int K, int N, int group, void *repacked, cudaStream_t stream) {
    w4a16_status st = check_shape(0, N, K, group);
    if (st != W4A16_OK) return st;
    if (N == 0) return W4A16_OK;
    if (!repack_supported(K, N, group))
        return fail(W4A16_ERR_UNSUPPORTED, "repacked layout needs K %% 256 == 0, N %% 32 == 0 and "
                    "a group that divides 256 or is a multiple of it (K=%d N=%d group=%d)",
                    K, N, group);
    if (!packed || !scales || !zeros || !repacked)
        return fail(W4A16_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(packed) || !aligned16(repacked) || ((uintptr_t)scales & 7) ||
        ((uintptr_t)zeros & 7))
        return fail(W4A16_ERR_MISALIGNED, "packed and repacked must be 16-byte aligned, scales "
                    "and zeros 8-byte aligned");
    cudaError_t e = launch_repack(packed, scales, zeros, K, N, group, repacked, stream);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "repack launch");
}

namespace {
// Checks shared by the repacked GEMM entry points; fills the stream plan.
w4a16_status plan_repacked(int M, int N, int K, int group, int experts, const w4a16_config *cfg,
                           w4a16_config &c) {
    w4a16_status st = check_shape(M, N, K, group);
    if (st != W4A16_OK) return st;
    if (!repack_supported(K, N, group))
        return fail(W4A16_ERR_UNSUPPORTED, "repacked layout needs K %% 256 == 0, N %% 32 == 0 and "
                    "a group that divides 256 or is a multiple of it (K=%d N=%d group=%d)",
                    K, N, group);
    c = cfg ? *cfg : w4a16_config{};
    if ((c.path != W4A16_PATH_AUTO && c.path != W4A16_PATH_DECODE) ||
        (c.variant != W4A16_DECODE_AUTO && c.variant != W4A16_DECODE_STREAM &&
         c.variant != W4A16_DECODE_WARP))
        return fail(W4A16_ERR_UNSUPPORTED, "repacked weights: decode path, stream or warp "
                    "variant only");
    if (c.dtype != W4A16_DTYPE_F16)
        return fail(W4A16_ERR_UNSUPPORTED, "repacked weights: fp16 only");
    c.path = W4A16_PATH_DECODE;
    // the warp-stream kernel serves M <= 8 (every row in one launch); the
    // stream kernel the rest.  By default the warp kernel takes calls of at
    // least four 256-k blocks per SM: below that too few warps have work, and
    // the stream kernel (more CTAs per tile) was measured faster
    const bool warp_ok = M <= 8 && decode_warp_perm_supported(M > 0 ? M : 1, N, K, group,
                                                              experts, c.ctas);
    const long long blocks = (long long)experts * (N / 32) * (K / 256);
    if (c.variant == W4A16_DECODE_WARP) {
        if (!warp_ok)
            return fail(W4A16_ERR_UNSUPPORTED, "repacked warp-stream kernel: M <= 8 and at "
                        "most 64 tiles per CTA (M=%d N=%d K=%d group=%d E=%d ctas=%d)",
                        M, N, K, group, experts, c.ctas);
        return W4A16_OK;
    }
    if (c.variant == W4A16_DECODE_AUTO && warp_ok && c.warps_n == 0 && c.split_k == 0 &&
        blocks >= 4LL * device_info().sm_count) {
        c.variant = W4A16_DECODE_WARP;
        return W4A16_OK;
    }
    c.variant = W4A16_DECODE_STREAM;
    const int m = M < 16 ? M : 16;
    plan_decode_stream(m > 0 ? m : 1, N, K, group, experts, true, device_info().sm_count, c);
    if (!decode_stream_supported(m > 0 ? m : 1, N, K, group, c.warps_n, true) || c.split_k < 1 ||
        c.split_k > 2 || c.ctas < 0)
        return fail(W4A16_ERR_UNSUPPORTED, "repacked stream configuration not available "
                    "(warps_n=%d split_k=%d ctas=%d)", c.warps_n, c.split_k, c.ctas);
    return W4A16_OK;
}
}  // namespace

w4a16_status w4a16_gemm_repacked(const uint16_t *x, const void *repacked, uint16_t *out, int M,
                                 int N, int K, int group, const w4a16_config *cfg,
                                 cudaStream_t stream) {
    w4a16_config c;
    w4a16_status st = plan_repacked(M, N, K, group, 1, cfg, c);
    if (st != W4A16_OK) return st;
    if (M == 0 || N == 0) return W4A16_OK;
    if (!x || !repacked || !out) return fail(W4A16_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(x) || !aligned16(repacked) || !aligned16(out))
        return fail(W4A16_ERR_MISALIGNED, "x, repacked and out must be 16-byte aligned");
    StreamCall sc;
    sc.E = 1;
    sc.s[0] = sc.z[0] = nullptr;
    sc.w[0] = static_cast<const uint32_t *>(repacked);
    sc.N = N;
    sc.K = K;
    sc.group = group;
    sc.permuted = true;
    if (c.variant == W4A16_DECODE_WARP) {
        sc.M = M;
        sc.x[0] = x;
        sc.out[0] = out;
        cudaError_t e = launch_decode_warp_perm(sc, c, stream);
        if (e == cudaErrorNotSupported)
            return fail(W4A16_ERR_UNSUPPORTED, "no kernel for this configuration");
        return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "gemm launch");
    }
    // 16 rows of x per launch (the decode kernel's batch); larger M runs
    // several launches in stream order
    for (int m0 = 0; m0 < M; m0 += 16) {
        sc.M = M - m0 < 16 ? M - m0 : 16;
        sc.x[0] = x + (size_t)m0 * K;
        sc.out[0] = out + (size_t)m0 * N;
        w4a16_config cm = c;
        if (sc.M != (M < 16 ? M : 16)) {
            // a ragged last chunk keeps the tile width when its layout fits
            if (!decode_stream_supported(sc.M, N, K, group, cm.warps_n, true)) cm.warps_n = 4;
        }
        cudaError_t e = launch_decode_stream(sc, cm, stream);
        if (e == cudaErrorNotSupported)
            return fail(W4A16_ERR_UNSUPPORTED, "no kernel for this configuration");
        if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
    }
    return W4A16_OK;
}

w4a16_status w4a16_gemm_grouped_repacked(int E, const uint16_t *const *x,
                                         const void *const *repacked, uint16_t *const *out, int M,
                                         int N, int K, int group, const w4a16_config *cfg,
                                         cudaStream_t stream) {
    if (E < 1 || E > W4A16_MAX_EXPERTS)
        return fail(W4A16_ERR_INVALID_ARG, "E=%d: 1..%d experts per grouped call", E,
                    W4A16_MAX_EXPERTS);
    if (!x || !repacked || !out) return fail(W4A16_ERR_INVALID_ARG, "null pointer table");
    if (M > 16)
        return fail(W4A16_ERR_UNSUPPORTED, "grouped repacked GEMM: M <= 16 (got %d)", M);
    w4a16_config c;
    w4a16_status st = plan_repacked(M, N, K, group, E, cfg, c);
    if (st != W4A16_OK) return st;
    for (int e = 0; e < E; ++e) {
        if (!x[e] || !repacked[e] || !out[e])
            return fail(W4A16_ERR_INVALID_ARG, "null pointer (expert %d)", e);
        if (!aligned16(x[e]) || !aligned16(repacked[e]) || !aligned16(out[e]))
            return fail(W4A16_ERR_MISALIGNED, "expert %d: x, repacked and out must be 16-byte "
                        "aligned", e);
    }
    if (M == 0 || N == 0) return W4A16_OK;
    StreamCall sc;
    sc.E = E;
    for (int e = 0; e < E; ++e) {
        sc.x[e] = x[e];
        sc.w[e] = static_cast<const uint32_t *>(repacked[e]);
        sc.s[e] = sc.z[e] = nullptr;
        sc.out[e] = out[e];
    }
    sc.M = M;
    sc.N = N;
    sc.K = K;
    sc.group = group;
    sc.permuted = true;
    cudaError_t err = c.variant == W4A16_DECODE_WARP ? launch_decode_warp_perm(sc, c, stream)
                                                     : launch_decode_stream(sc, c, stream);
    if (err == cudaErrorNotSupported)
        return fail(W4A16_ERR_UNSUPPORTED, "no kernel for this configuration");
    return err == cudaSuccess ? W4A16_OK : cuda_fail(err, "grouped gemm launch");
}

w4a16_status w4a16_gemm_noalloc(const uint16_t *x, const uint32_t *packed,
                                const uint16_t *scales, const uint16_t *zeros, uint16_t *out,
                                int M, int N, int K, int group, cudaStream_t stream) {
    w4a16_status st = check_shape(M, N, K, group);
    if (st != W4A16_OK) return st;
    if (M == 0 || N == 0) return W4A16_OK;
    if (!x || !packed || !scales || !zeros || !out)
        return fail(W4A16_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(x) || !aligned16(packed) || !aligned16(scales) || !aligned16(zeros) ||
        !aligned16(out))
        return fail(W4A16_ERR_MISALIGNED, "x, packed, scales, zeros and out must be 16-byte "
                    "aligned");
    if (M > 16)
        return fail(W4A16_ERR_UNSUPPORTED, "gemm_noalloc: M <= 16 (got %d)", M);
    w4a16_config c = {};
    c.path = W4A16_PATH_DECODE;
    c.variant = W4A16_DECODE_STREAM;
    c.split_k = 2;
    plan_decode_stream(M, N, K, group, 1, false, device_info().sm_count, c);
    if (!decode_stream_supported(M, N, K, group, c.warps_n, false))
        return fail(W4A16_ERR_UNSUPPORTED, "gemm_noalloc: no stream kernel for M=%d N=%d K=%d "
                    "group=%d (N %% 8 == 0 and a power-of-two group are required)", M, N, K, group);
    StreamCall sc;
    sc.E = 1;
    sc.x[0] = x;
    sc.w[0] = packed;
    sc.s[0] = scales;
    sc.z[0] = zeros;
    sc.out[0] = out;
    sc.M = M;
    sc.N = N;
    sc.K = K;
    sc.group = group;
    sc.permuted = false;
    const NoAllocResult r = launch_decode_stream_noalloc(sc, c.warps_n, false, stream);
    if (r.err == cudaErrorInvalidValue)
        return fail(W4A16_ERR_UNSUPPORTED, "gemm_noalloc: the call needs %zu bytes of tile "
                    "counters and %zu bytes of partial sums; the library's fixed scratch holds "
                    "65536 and 4128768", r.need_counters, r.need_partials);
    if (r.err == cudaErrorNotSupported)
        return fail(W4A16_ERR_UNSUPPORTED, "gemm_noalloc: no kernel for this configuration");
    return r.err == cudaSuccess ? W4A16_OK : cuda_fail(r.err, "gemm_noalloc");
}

w4a16_status w4a16_stream_read(const void *src, size_t bytes, uint32_t *sink, int flags,
                               cudaStream_t stream) {
    if (!src || !sink || bytes == 0)
        return fail(W4A16_ERR_INVALID_ARG, "stream_read: null pointer or zero bytes");
    if (!aligned16(src) || bytes % 16 != 0 || ((uintptr_t)sink & 3))
        return fail(W4A16_ERR_MISALIGNED, "stream_read: src 16-byte aligned, bytes a multiple of "
                    "16, sink 4-byte aligned");
    int *status = nullptr;
    cudaError_t e = kernel_status_address(&status);
    if (e != cudaSuccess) return cuda_fail(e, "status word");
    e = launch_read_probe(src, bytes, sink, device_info().sm_count, (flags & W4A16_FLAG_PDL) != 0,
                          status, stream);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "stream_read launch");
}

w4a16_status w4a16_get_kernel_status(cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    int v = 0;
    e = kernel_status_read_clear(&v, stream);
    if (e != cudaSuccess) return cuda_fail(e, "read/clear the device status word");
    if (v != 0)
        return fail((w4a16_status)v, "a kernel reported status %d (bounded wait gave up)", v);
    return W4A16_OK;
}

const char *w4a16_last_error(void) { return t_last_error.c_str(); }

int w4a16_version(void) { return 100; }

}  // extern "C"
