// prefill_pair.cu -- the tcgen05 prefill GEMM on CTA pairs (cta_group::2).
//
// Same product as prefill.cu (out[m,n] = sum_k x[m,k] * Wdq[k,n], fp32
// accumulation, fp16 output; page "Beating FP16 with 4-bit Weights", section
// "The design"), with the MMA spread over the two SMs of a cluster pair:
//   D[n, m] (256 weight columns x tile_m rows of x)
//     += A[n, k] (dequantized W^T: CTA r holds columns 128 r .. 128 r + 127
//                 in its own tensor memory)
//      * B[k, m] (x tile: CTA r holds rows r * tile_m/2 .. of the pair's rows
//                 in its own shared memory).
//   UMMA shape M = 256, N = tile_m, K = 16, issued by the even CTA only.
// Each SM stages half of the x tile that a one-CTA tile of the same shape
// would need, and one MMA instruction does twice the work: the single issuing
// thread and the shared-memory traffic (TMA writes plus MMA reads of x), which
// bound the one-CTA kernel at large M, both halve per unit of work.
//
// Per stage (128 k) and CTA: TMA brings the CTA's x half (3-D box, both 64-k
// chunks), its 16 x 128 packed words and scale/zero rows and completes the
// CTA's own `full` barrier; the CTA's dequantizing warps turn the words into
// its A slot in tensor memory and then arrive on the even CTA's `aready`
// barrier (remote arrive, release at cluster scope), which therefore also
// certifies that the odd CTA's x half has landed.  The even CTA's issuer waits
// on `aready` only, issues 8 MMAs and commits them with a multicast arrive on
// `empty` of both CTAs, which frees the slot for both producers.  A final
// multicast commit on `accum` starts both epilogues; each CTA stores its 128
// columns for all tile_m rows.  Every mbarrier wait is bounded; the two
// cluster barriers (after setup, before freeing tensor memory) are reached
// unconditionally by every thread of both CTAs.
#include <mutex>

#include "common.cuh"
#include "prefill_tile.cuh"
#include "sm100_ptx.cuh"
#include "tcgen05.cuh"
#include "tmap.cuh"

namespace w4a16 {
namespace {

// Tensor-memory columns each CTA of a pair allocates.
constexpr int kPairTmemCols = 512;

struct PairArgs {
    uint16_t *out;
    int *status;
    int M, N, K, group;
    int tile_m;            // rows of x per pair (multiple of 16, <= 256) = UMMA N
    int half_m;            // rows of x per CTA
    int stages;
    int stage_bytes;
    int p_off, s_off, z_off;   // offsets in a stage (x half at 0)
    int b_chunk_bytes;     // one 64-k chunk of the CTA's x half (half_m rows x 128 bytes)
    int tx_bytes;
    int tmem_cols;
    int a_col0;            // first column of the A stage ring (D uses [0, tile_m))
    unsigned long long timeout_ns;
};

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t cluster_addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
    return v;
}

template <int NDQ>
__global__ void __launch_bounds__(32 * (NDQ + 2), 1)
prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                    const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_z,
                    const PairArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + a.stages * a.stage_bytes);
    uint64_t *aready = full + a.stages;      // even CTA: both CTAs' A slots (and x halves) ready
    uint64_t *empty = aready + a.stages;     // MMAs of the stage completed (multicast commit)
    uint64_t *accum = empty + a.stages;      // all MMAs of the tile completed (multicast commit)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();            // 0: issues the MMAs
    const int n0 = (blockIdx.x >> 1) * (2 * kTileN) + (int)rank * kTileN;
    const int mp0 = blockIdx.y * a.tile_m;               // first row of x of the pair
    const int mx0 = mp0 + (int)rank * a.half_m;          // first row of this CTA's x half
    const int KT = (a.K + kStageK - 1) / kStageK;

    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_s);
        prefetch_tmap(&tm_z);
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&aready[i], 2 * NDQ);
            mbar_init(&empty[i], 1);
        }
        mbar_init(accum, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc<2>(smem_u32(tmem_slot), a.tmem_cols);
        tmem_relinquish<2>();
    }
    tc_fence_before();
    // every barrier of both CTAs exists and tensor memory is allocated before
    // either CTA signals the other
    cluster_arrive();
    cluster_wait();
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot;
    // the MMA addresses one tensor-memory offset in both CTAs
    const bool tmem_ok = ld_cluster_u32(map_to_rank(smem_u32(tmem_slot), rank ^ 1u)) == tmem_d;
    if (!tmem_ok && threadIdx.x == 0) report_status(a.status, W4A16_ERR_CUDA);

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer (both CTAs)
        const uint64_t pol_w = l2_evict_first_policy();
        const uint64_t pol_x = l2_evict_last_policy();
        int s = 0, r = 0, grow = 0, gnext = a.group;
        for (int kt = 0; kt < KT; ++kt) {
            const int k0 = kt * kStageK;
            while (k0 >= gnext) { ++grow; gnext += a.group; }
            if (r > 0 && !mbar_wait_cluster_bounded(&empty[s], (r - 1) & 1, a.timeout_ns))
                report_status(a.status, W4A16_ERR_TIMEOUT);
            if (lane == 0) {
                uint8_t *st = ring + s * a.stage_bytes;
                mbar_arrive_expect_tx(&full[s], a.tx_bytes);
                tma_load_3d(st, &tm_x, &full[s], 0, mx0, k0 / kChunkK, pol_x);
                tma_load_2d(st + a.p_off, &tm_w, &full[s], n0, k0 / 8, pol_w);
                tma_load_2d(st + a.s_off, &tm_s, &full[s], n0, grow, pol_w);
                tma_load_2d(st + a.z_off, &tm_z, &full[s], n0, grow, pol_w);
            }
            __syncwarp();
            if (++s == a.stages) { s = 0; ++r; }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer (even CTA)
        if (rank == 0) {
            const uint32_t idesc = idesc_f16(2 * kTileN, a.tile_m);
            const uint32_t tmem_u = __shfl_sync(0xffffffffu, tmem_d, 0);
            const uint32_t b_chunk16 = (uint32_t)a.b_chunk_bytes >> 4;
            const uint32_t ring_u = smem_u32(ring);
            int s = 0, r = 0;
            for (int kt = 0; kt < KT; ++kt) {
                if (!mbar_wait_cluster_bounded(&aready[s], r & 1, a.timeout_ns))
                    report_status(a.status, W4A16_ERR_TIMEOUT);
                tc_fence_after();
                const uint64_t b_desc = smem_desc_sw128(ring_u + (uint32_t)(s * a.stage_bytes));
                const uint32_t a_tmem = tmem_u + (uint32_t)(a.a_col0 + s * (kStageK / 2));
                if (lane == 0) {
                    if (tmem_ok) {
#pragma unroll
                        for (int kk = 0; kk < kStageK / 16; ++kk) {
                            const uint32_t c = kk / 4, w = kk % 4;
                            umma_f16_ts<2>(tmem_u, a_tmem + kk * 8, b_desc + c * b_chunk16 + w * 2,
                                           idesc, (kt | kk) != 0);
                        }
                    }
                    umma_commit_multicast2(&empty[s], 0x3);
                }
                __syncwarp();
                if (++s == a.stages) { s = 0; ++r; }
            }
            if (lane == 0) umma_commit_multicast2(accum, 0x3);
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------ dequant (both CTAs)
        constexpr int kParts = NDQ / 4;                   // warps per lane quarter
        static_assert(kPackedRows % kParts == 0, "packed rows must split evenly");
        constexpr int kRowsPer = kPackedRows / kParts;    // packed rows per thread
        constexpr int kBlk = kRowsPer >= 8 ? 8 : 4;       // words per TMEM store
        // a warp may only reach its lane quarter (warp % 4): the column a thread
        // dequantizes is the TMEM lane of that quarter
        const int n = (warp & 3) * 32 + lane;
        const int part = (warp - kDeqWarp0) / 4;          // which packed rows
        const uint32_t lane_base = tmem_d + ((uint32_t)((warp & 3) * 32) << 16);
        int s = 0, r = 0;
        for (int kt = 0; kt < KT; ++kt) {
            if (!mbar_wait_bounded(&full[s], r & 1, a.timeout_ns))
                report_status(a.status, W4A16_ERR_TIMEOUT);
            const uint32_t st = smem_u32(ring + s * a.stage_bytes);
            const int k0 = kt * kStageK;
#pragma unroll
            for (int b0 = 0; b0 < kRowsPer; b0 += kBlk) {
                const int c0 = part * kRowsPer + b0;
                uint32_t h[kBlk * 4];
                dequant_words<kBlk>(st, a.p_off, a.s_off, a.z_off, c0, stage_zrow(k0, a.group, c0),
                                    n, h);
                // A stage s: lane n, 32-bit columns a_col0 + 64 s + 4 c .. +3 (k = 8c .. 8c+7)
                tmem_st_32x32b<kBlk * 4>(lane_base + (uint32_t)(a.a_col0 + s * (kStageK / 2) + c0 * 4),
                                         h);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0)
                    mbar_arrive(&aready[s]);
                else
                    mbar_arrive_remote(map_to_rank(smem_u32(&aready[s]), 0));
            }
            if (++s == a.stages) { s = 0; ++r; }
        }
        // ------------------------------------------------------ epilogue (both CTAs)
        if (!mbar_wait_cluster_bounded(accum, 0, a.timeout_ns))
            report_status(a.status, W4A16_ERR_TIMEOUT);
        tc_fence_after();
        const int q = warp & 3;
        store_accumulator(lane_base, n0 + q * 32 + lane, mp0, a.tile_m, 32 * part, 32 * kParts,
                          a.M, a.N, a.out);
    }
    tc_fence_before();
    // neither CTA frees its tensor memory (or exits) while the other may
    // still signal it or read through the pair's MMAs
    cluster_arrive();
    cluster_wait();
    if (warp == 1) tmem_dealloc<2>(tmem_d, a.tmem_cols);
}

int round_up(int v, int m) { return (v + m - 1) / m * m; }

template <int NDQ>
cudaError_t launch_pair_kernel(dim3 grid, size_t smem, cudaStream_t stream, const CUtensorMap &tx,
                               const CUtensorMap &tw, const CUtensorMap &ts, const CUtensorMap &tz,
                               const PairArgs &pa) {
    const cudaError_t attr =
        ensure_dynamic_smem((const void *)prefill_pair_kernel<NDQ>, 227 * 1024);
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = dim3(32 * (NDQ + 2), 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = 2;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    lc.attrs = attrs;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, prefill_pair_kernel<NDQ>, tx, tw, ts, tz, pa);
}

int *status_word() {
    int *p = nullptr;
    return kernel_status_address(&p) == cudaSuccess ? p : nullptr;
}

}  // namespace

bool prefill_pair_supported(const w4a16_config &cfg, int M, int N, int K, int group) {
    (void)M;
    const bool warps_ok = cfg.warps_k == 0 || cfg.warps_k == 4 || cfg.warps_k == 8;
    return warps_ok && cfg.tile_m >= 16 && cfg.tile_m <= 256 && cfg.tile_m % 16 == 0 &&
           group % kChunkK == 0 && K % kChunkK == 0 && N % 8 == 0 && (K / group) >= 1;
}

cudaError_t launch_prefill_pair(const GemmArgs &a, const w4a16_config &cfg, cudaStream_t stream) {
    if (!prefill_pair_supported(cfg, a.M, a.N, a.K, a.group)) return cudaErrorNotSupported;
    PairArgs pa;
    pa.out = a.out;
    pa.status = status_word();
    if (!pa.status) return cudaErrorInvalidDevice;
    pa.M = a.M;
    pa.N = a.N;
    pa.K = a.K;
    pa.group = a.group;
    pa.tile_m = cfg.tile_m;
    pa.half_m = cfg.tile_m / 2;
    const int ndq = cfg.warps_k > 0 ? cfg.warps_k : 8;
    // stage (128 k): x half (two half_m x 64 fp16 chunks) | packed words
    // (16 x 128) | scale rows | zero rows (1, or 2 when group % 128 != 0)
    const int sz_rows = a.group % kStageK == 0 ? 1 : 2;
    pa.b_chunk_bytes = pa.half_m * kChunkK * 2;               // half_m % 8 == 0: 1024-aligned
    pa.p_off = kChunks * pa.b_chunk_bytes;
    pa.s_off = pa.p_off + kPackedRows * kTileN * 4;
    pa.z_off = pa.s_off + sz_rows * kTileN * 2;
    pa.stage_bytes = round_up(pa.z_off + sz_rows * kTileN * 2, 1024);
    pa.tx_bytes = kChunks * pa.b_chunk_bytes + kPackedRows * kTileN * 4 + 2 * sz_rows * kTileN * 2;
    int stages = (224 * 1024) / pa.stage_bytes;
    stages = stages > 8 ? 8 : stages;
    // tensor memory: the accumulator (tile_m fp32 columns, all rows of the
    // pair) and one 64-column A slot per stage
    pa.tmem_cols = kPairTmemCols;
    pa.a_col0 = round_up(pa.tile_m, 32);
    const int max_stages = (pa.tmem_cols - pa.a_col0) / (kStageK / 2);
    stages = stages > max_stages ? max_stages : stages;
    if (stages < 2) return cudaErrorNotSupported;
    pa.stages = stages;
    pa.timeout_ns = 1000000000ull;
    const size_t smem = (size_t)stages * pa.stage_bytes + (3 * stages + 1) * 8 + 16 + 1024;

    const uint64_t x_dims[3] = {(uint64_t)kChunkK, (uint64_t)a.M, (uint64_t)(a.K / kChunkK)};
    const uint64_t x_strides[2] = {(uint64_t)a.K * 2, (uint64_t)kChunkK * 2};
    const uint32_t x_box[3] = {(uint32_t)kChunkK, (uint32_t)pa.half_m, (uint32_t)kChunks};
    CUtensorMap tx, tw, ts, tz;
    if (!make_tmap(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, a.x, x_dims, x_strides, x_box,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.packed, a.N, a.K / 8,
                      (uint64_t)a.N * 4, kTileN, kPackedRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.scales, a.N, a.K / a.group,
                      (uint64_t)a.N * 2, kTileN, sz_rows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.zeros, a.N, a.K / a.group,
                      (uint64_t)a.N * 2, kTileN, sz_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;

    const int mtiles = (a.M + pa.tile_m - 1) / pa.tile_m;
    if (mtiles > 65535) return cudaErrorInvalidValue;
    dim3 grid(2 * ((a.N + 2 * kTileN - 1) / (2 * kTileN)), mtiles, 1);
    return ndq == 4 ? launch_pair_kernel<4>(grid, smem, stream, tx, tw, ts, tz, pa)
                    : launch_pair_kernel<8>(grid, smem, stream, tx, tw, ts, tz, pa);
}

}  // namespace w4a16
