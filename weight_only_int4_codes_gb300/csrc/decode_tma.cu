// decode_tma.cu -- the decode-regime W4A16 GEMM (M <= 16 per pass) with the
// weight stream staged by TMA.
//
// Same arithmetic as decode.cu (decode_math.cuh: LOP3 magic-exponent unpack,
// exact q - z in fp16, register-fed mma.m16n8k16 with swapped roles, one fp32
// scale per group), different data movement:
//   * one producer warp (one elected thread) issues 2-D TMA loads of each
//     stage -- 32 packed rows (256 k) of the CTA's column tile, the matching
//     scale and zero rows, and the 256 x M slice of x -- into a ring of shared
//     memory stages guarded by mbarriers.  The bytes in flight per SM no longer
//     depend on registers: with a 4-deep ring a CTA asks for its whole K slice
//     of a 4096 x 4096 weight at once.
//   * packed words land 128B-swizzled; consumer thread g reads 16-byte chunk
//     perm(g) of its row, which makes every ld.shared.v4 conflict-free (the
//     column permutation is undone when the results are stored).
//   * 8 consumer warps split a stage: 32-column strips x 32-k steps.
//   * split-K across the CTAs of one thread-block cluster, reduced in a fixed
//     order through distributed shared memory (no atomics, no workspace).
//   * the CTA uses under half of an SM (about 100 KB of shared memory, 288
//     threads), and signals programmatic dependent launch at its start, so the
//     next GEMM on the stream can start streaming its weights while this one
//     finishes.  Only x and out wait for the previous kernel (griddepcontrol).
//   * every mbarrier wait is bounded in wall time; a wait that gives up records
//     W4A16_ERR_TIMEOUT in the device status word and the kernel runs to its
//     end without touching memory it does not own.
#include <cooperative_groups.h>
#include <mutex>

#include "common.cuh"
#include "decode_math.cuh"
#include "sm100_ptx.cuh"
#include "tmap.cuh"

namespace cg = cooperative_groups;

namespace w4a16 {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kStageRows = 32;                 // packed rows per stage
constexpr int kStageK = 8 * kStageRows;        // 256 k per stage
constexpr int kRingBudget = 100 * 1024;        // bytes of ring per CTA (<= half an SM)

struct TmaDecodeArgs {
    uint16_t *out;
    int *status;
    int M, N, K, group;
    int rows_per_cta;         // packed rows per CTA (multiple of 32)
    int split;                // CTAs per cluster along K (= gridDim.y)
    int stages;               // ring depth
    int stage_bytes;          // bytes per ring slot (multiple of 1024)
    int s_off, z_off, x_off;  // tile offsets inside a slot
    int tx_bytes;             // bytes the TMA loads of one stage deliver
    unsigned long long timeout_ns;
    int test_skip_last;       // test hook: arm but never load the CTA's last stage
};

// consumer lane group g reads 16-byte chunk perm8(g) of its 128-byte row
__device__ __forceinline__ int perm8(int g) { return (g >> 1) + ((g & 1) << 2); }

template <int NT, int BNS>
__global__ void __launch_bounds__(kThreads, 2)
decode_tma_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
                  const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_x,
                  const TmaDecodeArgs a)
{
    constexpr int BN = 32 * BNS;                 // columns per CTA
    constexpr int WK = kConsumerWarps / BNS;     // consumer warps along a stage's 8 steps
    constexpr int SPW = 8 / WK;                  // steps per warp per stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + a.stages * a.stage_bytes);
    uint64_t *empty = full + a.stages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = a.K >> 3;
    const int cta_row0 = blockIdx.y * a.rows_per_cta;
    const int rows_here = min(a.rows_per_cta, KB - cta_row0);
    const int n_st = rows_here > 0 ? (rows_here + kStageRows - 1) / kStageRows : 0;
    const int col_base = blockIdx.x * BN;
    const int m_base = blockIdx.z * 16;
    const int Mc = min(16, a.M - m_base);

    pdl_launch_dependents();

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    float acc[NT][2][4];
#pragma unroll
    for (int p = 0; p < NT; ++p)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[p][j][r] = 0.f;

    const int g = lane >> 2, t = lane & 3;
    const int wn = warp % BNS, wk = warp / BNS;
    const int cl = 32 * wn + 4 * perm8(g);     // first of the thread's 4 columns in the tile

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tm_w);
            prefetch_tmap(&tm_s);
            prefetch_tmap(&tm_z);
            prefetch_tmap(&tm_x);
            const uint64_t pol_stream = l2_evict_first_policy();
            const uint64_t pol_keep = l2_evict_last_policy();
            const int skip = (a.test_skip_last && n_st > 0) ? n_st - 1 : -1;
            const int first = min(a.stages, n_st);
            // weights, scales and zeros do not depend on the previous kernel:
            // stream the first ring's worth before waiting for it
            for (int st = 0; st < first; ++st) {
                uint8_t *slot = ring + st * a.stage_bytes;
                mbar_arrive_expect_tx(&full[st], a.tx_bytes);
                if (st == skip) continue;
                const int row = cta_row0 + st * kStageRows;
                const int grow = row * 8 / a.group;
#pragma unroll
                for (int s = 0; s < BNS; ++s)
                    tma_load_2d(slot + s * 4096, &tm_w, &full[st], col_base + 32 * s, row, pol_stream);
                tma_load_2d(slot + a.s_off, &tm_s, &full[st], col_base, grow, pol_stream);
                tma_load_2d(slot + a.z_off, &tm_z, &full[st], col_base, grow, pol_stream);
            }
            pdl_wait();   // x may be the previous kernel's output
            for (int st = 0; st < first; ++st) {
                if (st == skip) continue;
                tma_load_2d(ring + st * a.stage_bytes + a.x_off, &tm_x, &full[st],
                            (cta_row0 + st * kStageRows) * 8, m_base, pol_keep);
            }
            for (int st = first; st < n_st; ++st) {
                const int slot = st % a.stages;
                const uint32_t parity = ((st / a.stages) - 1) & 1;
                if (!mbar_wait_bounded(&empty[slot], parity, a.timeout_ns))
                    report_status(a.status, W4A16_ERR_TIMEOUT);
                uint8_t *sl = ring + slot * a.stage_bytes;
                mbar_arrive_expect_tx(&full[slot], a.tx_bytes);
                if (st == skip) continue;
                const int row = cta_row0 + st * kStageRows;
                const int grow = row * 8 / a.group;
#pragma unroll
                for (int s = 0; s < BNS; ++s)
                    tma_load_2d(sl + s * 4096, &tm_w, &full[slot], col_base + 32 * s, row, pol_stream);
                tma_load_2d(sl + a.s_off, &tm_s, &full[slot], col_base, grow, pol_stream);
                tma_load_2d(sl + a.z_off, &tm_z, &full[slot], col_base, grow, pol_stream);
                tma_load_2d(sl + a.x_off, &tm_x, &full[slot], row * 8, m_base, pol_keep);
            }
            // no copy of this CTA may still be landing when it exits
            for (int st = max(0, n_st - a.stages); st < n_st; ++st) {
                if (st == skip) continue;
                if (!mbar_wait_bounded(&full[st % a.stages], (st / a.stages) & 1, a.timeout_ns))
                    report_status(a.status, W4A16_ERR_TIMEOUT);
            }
        }
    } else {
        // ------------------------------------------------------ consumers
        const int spg = a.group >> 5;              // 32-k steps per group
        const int spf = min(SPW, spg);             // steps between scale flushes
        const bool x0_ok = g < Mc, x1_ok = g + 8 < Mc;
        float gacc[NT][2][4];
#pragma unroll
        for (int p = 0; p < NT; ++p)
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int r = 0; r < 4; ++r) gacc[p][j][r] = 0.f;

        for (int st = 0; st < n_st; ++st) {
            const int slot = st % a.stages;
            if (!mbar_wait_bounded(&full[slot], (st / a.stages) & 1, a.timeout_ns))
                report_status(a.status, W4A16_ERR_TIMEOUT);
            const uint8_t *base = ring + slot * a.stage_bytes;
            const uint8_t *wtile = base + wn * 4096;
            GroupConsts k;
#pragma unroll
            for (int u = 0; u < SPW; ++u) {
                const int r = wk * 4 * SPW + 4 * u + t;        // row within the stage
                if (u % spf == 0) {
                    const int gi = (r * 8) / a.group;           // group within the stage
                    const uint2 sraw = *reinterpret_cast<const uint2 *>(base + a.s_off + (gi * BN + cl) * 2);
                    const uint2 zraw = *reinterpret_cast<const uint2 *>(base + a.z_off + (gi * BN + cl) * 2);
                    k = make_group_consts(zraw, sraw);
                }
                const uint4 w = *reinterpret_cast<const uint4 *>(
                    wtile + r * 128 + ((perm8(g) ^ (r & 7)) << 4));
                uint32_t bx[NT][4];
                {
                    const uint4 v = x0_ok ? *reinterpret_cast<const uint4 *>(
                                                base + a.x_off + (g * kStageK + 8 * r) * 2)
                                          : make_uint4(0, 0, 0, 0);
                    x_fragments(v, bx[0]);
                }
                if (NT > 1) {
                    const uint4 v = x1_ok ? *reinterpret_cast<const uint4 *>(
                                                base + a.x_off + ((g + 8) * kStageK + 8 * r) * 2)
                                          : make_uint4(0, 0, 0, 0);
                    x_fragments(v, bx[NT - 1]);
                }
                step_mma<NT>(gacc, w, k, bx);
                if ((u + 1) % spf == 0) flush_group<NT>(acc, gacc, k);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }

    // ---------------------------------------------------------- epilogue
    __syncthreads();   // ring drained: reuse it for the reduction
    pdl_wait();        // out may still be in use by the previous kernel
    float *red = reinterpret_cast<float *>(ring);        // [WK][16][BN]
    float *part = red + WK * 16 * BN;                     // [16][BN]
    if (warp < kConsumerWarps) {
#pragma unroll
        for (int p = 0; p < NT; ++p)
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int m = 8 * p + 2 * t + (r & 1);
                    const int c = cl + 2 * j + (r >> 1);
                    if (m < Mc) red[(wk * 16 + m) * BN + c] = acc[p][j][r];
                }
    }
    __syncthreads();
    const int E = Mc * BN;
    for (int e = threadIdx.x; e < E; e += kThreads) {
        const int m = e / BN, c = e - m * BN;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < WK; ++w) v += red[(w * 16 + m) * BN + c];
        if (a.split == 1) {
            const int col = col_base + c;
            if (col < a.N)
                a.out[(size_t)(m_base + m) * a.N + col] = __half_as_ushort(__float2half_rn(v));
        } else {
            part[e] = v;
        }
    }
    if (a.split == 1) return;

    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int rank = (int)cluster.block_rank();
    const int per = (E + a.split - 1) / a.split;
    const int e_end = min(E, (rank + 1) * per);
    for (int e = rank * per + threadIdx.x; e < e_end; e += kThreads) {
        float v = 0.f;
        for (int q = 0; q < a.split; ++q) v += cluster.map_shared_rank(part, q)[e];
        const int m = e / BN, c = e - m * BN;
        const int col = col_base + c;
        if (col < a.N)
            a.out[(size_t)(m_base + m) * a.N + col] = __half_as_ushort(__float2half_rn(v));
    }
    cluster.sync();    // peers may still be reading this CTA's partials
}

int round_up(int v, int m) { return (v + m - 1) / m * m; }

struct Layout {
    int gps, s_off, z_off, x_off, stage_bytes, tx_bytes, stages, smem_bytes;
};

Layout layout_for(int group, int bns, int nt, int n_st) {
    Layout L;
    const int BN = 32 * bns;
    const int mb = 8 * nt;
    L.gps = kStageK / group;
    const int sz = L.gps * BN * 2;
    L.s_off = bns * 4096;
    L.z_off = L.s_off + round_up(sz, 128);
    L.x_off = L.z_off + round_up(sz, 128);
    L.stage_bytes = round_up(L.x_off + kStageK * mb * 2, 1024);
    L.tx_bytes = bns * 4096 + 2 * sz + kStageK * mb * 2;
    int ns = kRingBudget / L.stage_bytes;
    ns = ns < 2 ? 2 : (ns > 6 ? 6 : ns);
    if (n_st > 0 && ns > n_st) ns = n_st < 2 ? 2 : n_st;
    // the epilogue reuses the ring for WK + 1 partial tiles
    const int red_bytes = (kConsumerWarps / bns + 1) * 16 * BN * 4;
    while (ns * L.stage_bytes < red_bytes) ++ns;
    L.stages = ns;
    L.smem_bytes = ns * L.stage_bytes + 2 * ns * 8 + 1024;
    return L;
}

template <int NT, int BNS>
cudaError_t launch_tma(const CUtensorMap &w, const CUtensorMap &s, const CUtensorMap &z,
                       const CUtensorMap &x, const TmaDecodeArgs &da, int tiles, int mchunks,
                       int smem, bool pdl, cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(decode_tma_kernel<NT, BNS>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, 116 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(tiles, da.split, mchunks);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (da.split > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = 1;
        attrs[na].val.clusterDim.y = da.split;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    lc.attrs = attrs;
    lc.numAttrs = na;
    return cudaLaunchKernelEx(&lc, decode_tma_kernel<NT, BNS>, w, s, z, x, da);
}

int *status_word() {
    static int *ptrs[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        int *p = nullptr;
        if (kernel_status_address(&p) != cudaSuccess) return nullptr;
        ptrs[dev] = p;
    }
    return ptrs[dev];
}

}  // namespace

bool decode_tma_supported(const w4a16_config &cfg, int group) {
    const bool g_ok = group == 32 || group == 64 || group == 128 || group == 256;
    return g_ok && (cfg.warps_n == 2 || cfg.warps_n == 4) && cfg.split_k >= 1 &&
           cfg.split_k <= 8 && cfg.steps >= 1;
}

// cfg: warps_n = 32-column strips per CTA (2 or 4), split_k = CTAs per cluster
// along K, steps = 256-k stages per CTA.
cudaError_t launch_decode_tma(const GemmArgs &a, const w4a16_config &cfg, cudaStream_t stream) {
    if (!decode_tma_supported(cfg, a.group)) return cudaErrorNotSupported;
    const int bns = cfg.warps_n;
    const int nt = a.M > 8 ? 2 : 1;
    const int KB = a.K / 8;
    const int rows_per_cta = cfg.steps * kStageRows;
    if ((long long)rows_per_cta * cfg.split_k < KB) return cudaErrorInvalidValue;
    const Layout L = layout_for(a.group, bns, nt, cfg.steps);
    const int BN = 32 * bns;
    const int mb = 8 * nt;
    CUtensorMap tw, ts, tz, tx;
    if (!make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.packed, a.N, KB, (uint64_t)a.N * 4,
                      32, kStageRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.scales, a.N, a.K / a.group,
                      (uint64_t)a.N * 2, BN, L.gps, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.zeros, a.N, a.K / a.group,
                      (uint64_t)a.N * 2, BN, L.gps, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.x, a.K, a.M, (uint64_t)a.K * 2,
                      kStageK, mb, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    TmaDecodeArgs da;
    da.out = a.out;
    da.status = status_word();
    if (!da.status) return cudaErrorInvalidDevice;
    da.M = a.M;
    da.N = a.N;
    da.K = a.K;
    da.group = a.group;
    da.rows_per_cta = rows_per_cta;
    da.split = cfg.split_k;
    da.stages = L.stages;
    da.stage_bytes = L.stage_bytes;
    da.s_off = L.s_off;
    da.z_off = L.z_off;
    da.x_off = L.x_off;
    da.tx_bytes = L.tx_bytes;
    const bool test_timeout = (cfg.flags & W4A16_FLAG_TEST_TIMEOUT) != 0;
    da.timeout_ns = test_timeout ? 5000000ull : 1000000000ull;   // 5 ms in the test mode, else 1 s
    da.test_skip_last = test_timeout ? 1 : 0;
    const int tiles = (a.N + BN - 1) / BN;
    const int mchunks = (a.M + 15) / 16;
    if (mchunks > 65535) return cudaErrorInvalidValue;
    const bool pdl = (cfg.flags & W4A16_FLAG_PDL) != 0;
    if (nt == 1)
        return bns == 4 ? launch_tma<1, 4>(tw, ts, tz, tx, da, tiles, mchunks, L.smem_bytes, pdl, stream)
                        : launch_tma<1, 2>(tw, ts, tz, tx, da, tiles, mchunks, L.smem_bytes, pdl, stream);
    return bns == 4 ? launch_tma<2, 4>(tw, ts, tz, tx, da, tiles, mchunks, L.smem_bytes, pdl, stream)
                    : launch_tma<2, 2>(tw, ts, tz, tx, da, tiles, mchunks, L.smem_bytes, pdl, stream);
}

}  // namespace w4a16
