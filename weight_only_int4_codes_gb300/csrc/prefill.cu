// prefill.cu -- W4A16 GEMM for larger M on the 5th-generation tensor cores
// (tcgen05.mma, accumulator in tensor memory).
//
// What it computes: out[m,n] = sum_k x[m,k] * Wdq[k,n], Wdq = fp16((q - z) * s),
// fp32 accumulation, fp16 output -- or, with bfloat16 data, Wdq = bf16((q - z)
// * s), bf16 x bf16 MMAs and a bfloat16 output (page "Beating FP16 with 4-bit Weights",
// section "The design": the packed tile is loaded, unpacked in registers,
// dequantized and fed to a tensor-core dot product with fp32 accumulation;
// section "Results": once M grows into prefill the unpack must hide under the
// MMA).
//
// Roles are swapped so that one kernel family serves every M from 16 up:
//   D[n, m] (TMEM: 128 lanes = weight columns n, tile_m columns = rows m of x)
//     += A[n, k] (dequantized W^T, in tensor memory -- or, variant 2, in
//                 128B-swizzled shared memory)
//      * B[k, m] (x tile, K-major = x row-major, TMA-loaded 128B-swizzled).
//   UMMA shape M = 128 (weight columns), N = tile_m (16..256, rows of x), K = 16.
// Each weight is dequantized once per tile_m rows of x; with A in tensor
// memory the dequantized weight never touches shared memory, which would
// otherwise become the bottleneck (the MMA re-reads its shared operands).
//
// Two kernels, chosen by tile width (launch_prefill):
//   * prefill_split_kernel (tiles of 192+ rows): persistent, one CTA per SM;
//     a stage slot holds the x tile and the dequantized A stage, freed by one
//     commit, while the weights travel on a ring of their own (see its
//     comment); the epilogue drains the accumulator into registers and stores
//     from there while the next tile's MMAs run;
//   * prefill_tcgen05_kernel (narrower tiles, and the A-in-shared-memory
//     variant): one CTA per tile, one ring of 128-k stages carrying the x
//     chunks, the packed words and the scale/zero rows -- one wait and one
//     commit per stage, cheaper when a stage holds few MMA cycles.  Tiles of
//     up to 64 rows use half an SM, so two CTAs (two issuers) share it; at the
//     end the accumulator is staged as an fp16 tile in the drained ring and
//     stored with one TMA copy.
// In both, the 4, 8 or 16 dequantizing warps own one weight column (one TMEM
// lane) per thread and split the stage's 16 packed rows, and run the
// epilogue.  Every wait is bounded in wall time; a wait that gives up records
// W4A16_ERR_TIMEOUT and the kernel still frees its tensor memory before it
// exits.
#include <mutex>

#include "common.cuh"
#include "sm100_ptx.cuh"
#include "prefill_tile.cuh"
#include "tcgen05.cuh"
#include "tmap.cuh"

namespace w4a16 {
namespace {


struct PrefillArgs {
    uint16_t *out;
    int *status;
    int M, N, K, group;
    int tile_m;            // rows of x per CTA (multiple of 16, <= 256) = UMMA N
    int stages;
    int stage_bytes;
    int b_off, p_off, s_off, z_off;   // offsets in a stage (A tile at 0)
    int b_chunk_bytes;     // one 64-k chunk of the x tile (tile_m rows x 128 bytes)
    int sz_rows;           // scale/zero rows per stage: 1, or 2 when a group boundary may fall mid-stage
    int tx_bytes;
    int tmem_cols;         // allocated columns
    int a_col0;            // A-in-TMEM: first column of the A stage ring (D uses [0, tile_m))
    int split;             // CTAs per cluster along K (gridDim.z); 1 = no split
    int kt_per;            // 128-k stages per CTA of a split cluster
    int red_off;           // leader: fp32 partial slots [split - 1][tile_m][128] (after the ring)
    int bar_off;           // mbarriers
    unsigned long long timeout_ns;
};

// NDQ: dequantizing warps (4, 8 or 16); they split the stage's 16 packed rows
// of each column (NDQ/4 warps per column group) and, in the epilogue, the
// accumulator's columns.
// ATMEM: the dequantized A operand lives in tensor memory (written with
// tcgen05.st, read by the MMA as [a_tmem]) instead of shared memory; the
// stage then carries only x, the packed words and the scale/zero rows.
// SPLIT: split-K across a cluster along z (a separate instantiation, so that
// the kernel without it carries none of its code).
// BF: x, scales, zeros and out are bfloat16 (MMA operands bf16 x bf16).
template <int NDQ, bool ATMEM, bool SPLIT, bool BF>
__global__ void __launch_bounds__(32 * (NDQ + 2), 1)
prefill_tcgen05_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_z,
                       const __grid_constant__ CUtensorMap tm_o, const PrefillArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + a.bar_off);
    uint64_t *aready = full + a.stages;      // dequantized A tile written
    uint64_t *empty = aready + a.stages;     // MMAs of the stage completed
    uint64_t *accum = empty + a.stages;      // all MMAs of the tile completed
    uint64_t *cl_done = accum + 1;           // split leader: the other CTAs' partials landed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(cl_done + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kTileN;
    const int m0 = blockIdx.y * a.tile_m;
    const int KT = (a.K + kStageK - 1) / kStageK;      // a last half stage reads zero x
    // split-K: this CTA's stages [kt0, kt1) (the host makes every range non-empty)
    const int kt0 = SPLIT ? (int)blockIdx.z * a.kt_per : 0;
    const int kt1 = SPLIT ? (kt0 + a.kt_per < KT ? kt0 + a.kt_per : KT) : KT;
    const int rank = SPLIT ? (int)cluster_ctarank() : 0;

    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_s);
        prefetch_tmap(&tm_z);
        prefetch_tmap(&tm_o);
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&aready[i], NDQ);
            mbar_init(&empty[i], 1);
        }
        mbar_init(accum, 1);
        mbar_init(cl_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot;
    if constexpr (SPLIT) {
        // the leader expects the other CTAs' partials as bulk-copy bytes; the
        // first half of a split cluster barrier then publishes every CTA's
        // barriers before any CTA signals another
        if (rank == 0 && threadIdx.x == 0)
            mbar_arrive_expect_tx(cl_done, (uint32_t)((a.split - 1) * a.tile_m * kTileN * 4));
        cluster_arrive();
    }

    // The producer and the MMA issuer are single threads whose loop bodies sit
    // on the critical path of every stage: their ring position is kept
    // incrementally (no division in the loop) and a stage is 128 k deep, so
    // each loop trip feeds the tensor core for 8 MMAs.
    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        // The whole warp runs the loop (its control values stay warp-uniform);
        // lane 0 issues.
        const uint64_t pol_w = l2_evict_first_policy();
        const uint64_t pol_x = l2_evict_last_policy();
        int s = 0, r = 0, grow = 0, gnext = a.group;
        for (int kt = kt0; kt < kt1; ++kt) {
            const int k0 = kt * kStageK;
            while (k0 >= gnext) { ++grow; gnext += a.group; }
            if (r > 0 && !mbar_wait_bounded(&empty[s], (r - 1) & 1, a.timeout_ns))
                report_status(a.status, W4A16_ERR_TIMEOUT);
            if (lane == 0) {
                uint8_t *st = ring + s * a.stage_bytes;
                mbar_arrive_expect_tx(&full[s], a.tx_bytes);
                // x: both 64-k chunks of the tile in one 3-D box (chunk index outermost)
                tma_load_3d(st + a.b_off, &tm_x, &full[s], 0, m0, k0 / kChunkK, pol_x);
                tma_load_2d(st + a.p_off, &tm_w, &full[s], n0, k0 / 8, pol_w);
                tma_load_2d(st + a.s_off, &tm_s, &full[s], n0, grow, pol_w);
                tma_load_2d(st + a.z_off, &tm_z, &full[s], n0, grow, pol_w);
            }
            __syncwarp();
            if (++s == a.stages) { s = 0; ++r; }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        // Warp-wide loop, lane 0 issues the MMAs and the commits (a commit
        // tracks the MMAs of the thread that issues it).
        const uint32_t idesc = idesc_f16(128, a.tile_m, BF);
        const uint32_t tmem_u = __shfl_sync(0xffffffffu, tmem_d, 0);
        const uint32_t b_chunk16 = (uint32_t)a.b_chunk_bytes >> 4;
        const uint32_t ring_u = smem_u32(ring);
        int s = 0, r = 0;
        for (int kt = kt0; kt < kt1; ++kt) {
            // the dequant warps arrive on `aready` only after they saw the
            // stage's copies land (`full`): one wait covers both
            if (!mbar_spin_bounded(&aready[s], r & 1, a.timeout_ns))
                report_status(a.status, W4A16_ERR_TIMEOUT);
            tc_fence_after();
            const uint32_t a_addr = ring_u + (uint32_t)(s * a.stage_bytes);
            const uint64_t b_desc = smem_desc_sw128(a_addr + a.b_off);
            const uint64_t a_desc = smem_desc_sw128(a_addr);
            const uint32_t a_tmem = tmem_u + (uint32_t)(a.a_col0 + s * (kStageK / 2));
            if (lane == 0) {
                // descriptors advance in 16-byte units: 32 bytes per k16 step
                // inside a chunk, a whole chunk between chunks
#pragma unroll
                for (int kk = 0; kk < kStageK / 16; ++kk) {
                    const uint32_t c = kk / 4, w = kk % 4;
                    const uint64_t bd = b_desc + c * b_chunk16 + w * 2;
                    const uint32_t acc = (kt != kt0) || (kk != 0);
                    if (ATMEM)
                        umma_f16_ts(tmem_u, a_tmem + kk * 8, bd, idesc, acc);
                    else
                        umma_f16_ss(tmem_u, a_desc + c * (kTileN * kChunkK * 2 / 16) + w * 2, bd,
                                 idesc, acc);
                }
                umma_commit(&empty[s]);
            }
            __syncwarp();
            if (++s == a.stages) { s = 0; ++r; }
        }
        if (lane == 0) umma_commit(accum);
        __syncwarp();
    } else {
        // ------------------------------------------------------ dequant
        constexpr int kParts = NDQ / 4;                   // warps per column group
        static_assert(kPackedRows % kParts == 0, "packed rows must split evenly");
        constexpr int kRowsPer = kPackedRows / kParts;    // packed rows per thread
        constexpr int kBlk = kRowsPer >= 8 ? 8 : 4;       // words per TMEM store
        // A-in-TMEM: a warp may only reach its lane quarter (warp % 4), so the
        // column a thread dequantizes is the TMEM lane of that quarter
        const int n = ATMEM ? ((warp & 3) * 32 + lane)
                            : (((warp - kDeqWarp0) * 32 + lane) & (kTileN - 1));
        const int part = (warp - kDeqWarp0) / 4;          // which packed rows
        int s = 0, r = 0;
        for (int kt = kt0; kt < kt1; ++kt) {
            if (!mbar_wait_bounded(&full[s], r & 1, a.timeout_ns))
                report_status(a.status, W4A16_ERR_TIMEOUT);
            const uint32_t st = smem_u32(ring + s * a.stage_bytes);
            // the stage's scale/zero rows start at group k0 / group
            const int k0 = kt * kStageK;
#pragma unroll
            for (int b0 = 0; b0 < kRowsPer; b0 += kBlk) {
                const int c0 = part * kRowsPer + b0;              // first packed row of the block
                uint32_t h[kBlk * 4];
                dequant_words<kBlk, BF>(st, a.p_off, a.s_off, a.z_off, c0, stage_zrow(k0, a.group, c0),
                                    n, h);
                if (ATMEM) {
                    // A stage s: lane n, 32-bit columns a_col0 + 64 s + 4 c .. +3 (k = 8c .. 8c+7)
                    const uint32_t ta = tmem_d + ((uint32_t)((warp & 3) * 32) << 16) +
                                        (uint32_t)(a.a_col0 + s * (kStageK / 2) + c0 * 4);
                    tmem_st_32x32b<kBlk * 4>(ta, h);
                } else {
#pragma unroll
                    for (int cc = 0; cc < kBlk; ++cc) {
                        const int c = c0 + cc;
                        const uint32_t off = (c / 8) * (kTileN * kChunkK * 2) + sw128_offset(n, c % 8);
                        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(st + off),
                                     "r"(h[cc * 4]), "r"(h[cc * 4 + 1]), "r"(h[cc * 4 + 2]),
                                     "r"(h[cc * 4 + 3])
                                     : "memory");
                    }
                }
            }
            if (ATMEM) {
                tmem_st_wait();
                tc_fence_before();
            } else {
                fence_proxy_async_smem();      // the tensor cores read these stores
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&aready[s]);
            if (++s == a.stages) { s = 0; ++r; }
        }
        // ------------------------------------------------------ epilogue
        if (!mbar_wait_bounded(accum, 0, a.timeout_ns))
            report_status(a.status, W4A16_ERR_TIMEOUT);
        tc_fence_after();
        const int q = warp & 3;                          // TMEM lane quarter of this warp
        const uint32_t taddr = tmem_d + ((uint32_t)(q * 32) << 16);
        const int epart = (warp - kDeqWarp0) / 4;        // warps of one quarter split the m chunks
        if (SPLIT && rank != 0) {
            // split-K, not the leader: the fp32 partial tile [tile_m][128]
            // goes into the drained ring, then with one bulk copy into slot
            // rank - 1 of the leader's shared memory (completing bytes on the
            // leader's cl_done); the CTA exits once the copy has read it
            stage_partial_f32(taddr, smem_u32(ring), q * 32 + lane, a.tile_m, 32 * epart,
                              32 * kParts);
            fence_proxy_async_smem();                    // the bulk copy reads these writes
            named_bar_sync(1, NDQ * 32);
            if (warp == kDeqWarp0 && lane == 0) {
                cluster_wait();                          // the leader's barrier is initialized
                const uint32_t bytes = (uint32_t)(a.tile_m * kTileN * 4);
                bulk_copy_to_cluster(
                    map_to_rank(smem_u32(ring + a.red_off) + (uint32_t)(rank - 1) * bytes, 0), ring,
                    bytes, map_to_rank(smem_u32(cl_done), 0));
                bulk_commit();
                bulk_wait_read();
            }
        } else {
            if (SPLIT && !mbar_wait_cluster_bounded(cl_done, 0, a.timeout_ns))
                report_status(a.status, W4A16_ERR_TIMEOUT);
            // every copy has landed and every MMA has read its operands: the
            // ring holds the fp16 output tile [tile_m][128] -- this CTA's
            // accumulator plus the other CTAs' partials in rank order -- stored
            // by one TMA copy (rows past M and columns past N are clipped by
            // the tensor map)
            if constexpr (SPLIT)
                stage_accumulator<BF>(taddr, smem_u32(ring), q * 32 + lane, a.tile_m, 32 * epart,
                                      32 * kParts, smem_u32(ring + a.red_off), a.split - 1);
            else
                stage_accumulator<BF>(taddr, smem_u32(ring), q * 32 + lane, a.tile_m, 32 * epart,
                                  32 * kParts);
            fence_proxy_async_smem();
            named_bar_sync(1, NDQ * 32);
            if (warp == kDeqWarp0 && lane == 0) {
                tma_store_2d(&tm_o, ring, n0, m0);
                bulk_commit();
                bulk_wait_all();
            }
        }
    }
    // every thread completes the split cluster barrier once (the non-leader's
    // copying thread already has)
    if (SPLIT && !(rank != 0 && warp == kDeqWarp0 && lane == 0)) cluster_wait();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem_d, a.tmem_cols);
}

// ---------------------------------------------------------------------------
// Split-ring kernel (the default for wide tiles, A in tensor memory).  It is
// persistent: one CTA per SM walks the output tiles t = blockIdx.x, +gridDim.x,
// ... (in the grouped order of split_tile below), and its rings run on across
// tile boundaries, so the next tile's copies and dequantization overlap the
// current tile's last MMAs and epilogue.  The weights travel on their own
// ring, apart from the x tile:
//   stage slots  xs slots, each holding one 128-k x tile (two 64-k chunks,
//                128B-swizzled, one 3-D TMA box) in shared memory AND one
//                dequantized 128-k A stage (64 columns) in tensor memory;
//                filled by warp 0 (x) and the dequantizing warps (A), freed
//                by ONE commit of the stage's MMAs;
//   weight ring  ws slots of one 128-k stage (16 x 128 packed words, scale
//                and zero rows); filled by warp 2, freed by the dequantizing
//                warps as soon as they have the words in registers.
// The single issuing thread is the pace-setter at tile_m = 256 (a
// tcgen05.mma issue costs tens of cycles, a commit about a hundred): per
// stage it waits on two barriers, issues 8 MMAs and one commit.
// The accumulator (tile_m fp32 columns) has one buffer: at the end of a tile
// the dequantizing warps drain it into registers (fp16 pairs), free it for
// the next tile's MMAs, and then write the fp16 tile to global memory with
// 4-byte stores while the next tile's first stages, already dequantized,
// run on the tensor cores.
// Warps: 0 x producer, 1 tensor-memory owner and MMA issuer, 2 weight
// producer, 3.. dequantization and epilogue.
constexpr int kSplitDeq0 = 3;
constexpr int kTwoPerSmMaxTileM = 64;   // one-ring kernel: two CTAs per SM up to this tile
constexpr int kSplitMinTileM = 192;     // measured crossover (128: one ring is faster)
constexpr int kMaxPrefillSplit = 8;     // one-ring kernel: split-K cluster size (portable limit)
constexpr int kMaxWeightSlots = 16;     // split-ring kernel: weight ring depth cap

struct SplitArgs {
    int *status;
    uint16_t *out;
    int M, N, K, group;
    int tile_m;
    int n_tiles, tiles;        // weight-column tiles, all output tiles
    int m_tiles, gm;           // x row tiles; row tiles per group of the tile order
    int xs, ws;                // stage slots (x in shared + A in tensor memory), weight slots
    int x_stage_bytes;         // two 64-k chunks of the x tile: tile_m * 256
    int x_chunk_bytes;         // tile_m * 128
    int w_off;                 // offset of the weight ring (after the x slots)
    int w_stage_bytes;
    int s_off, z_off;          // scale / zero rows inside a weight stage (packed at 0)
    int sz_rows;
    int w_tx;                  // bytes one weight stage's copies deliver
    int tmem_cols, a_col0;
    unsigned long long timeout_ns;
};

// Output tile t of the persistent walk.  Tiles go in groups of `gm` x row
// tiles: within a group the row tile runs fastest and the weight-column tile
// slowest, so the CTAs resident at one time share a few weight tiles (read
// from DRAM once, then from L2 by the group's other row tiles) and the group's
// x rows stay in L2 while the group sweeps every weight column.  Without the
// grouping the whole weight matrix would pass through L2 once per x row tile.
__device__ __forceinline__ void split_tile(const SplitArgs &a, int t, int &m0, int &n0) {
    const int per_group = a.gm * a.n_tiles;
    const int g = t / per_group;
    const int r = t - g * per_group;
    const int left = a.m_tiles - g * a.gm;
    const int gm = left < a.gm ? left : a.gm;
    const int n = r / gm;
    m0 = (g * a.gm + (r - n * gm)) * a.tile_m;
    n0 = n * kTileN;
}

// Write 16 fp16 pairs of one thread -- column n (its TMEM lane), rows
// r0 + 2j and r0 + 2j + 1 -- as 4-byte words: even and odd lanes swap halves
// so that each holds two adjacent columns of one row.
__device__ __forceinline__ void store_pairs(const uint32_t (&hc)[16], int r0, int lane, int col,
                                            bool col_ok, int m0, int tile_m, int M, int N,
                                            uint16_t *out) {
    const bool odd = lane & 1;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint32_t mine = hc[j];
        const uint32_t other = __shfl_xor_sync(0xffffffffu, mine, 1);
        const uint32_t w = odd ? __byte_perm(other, mine, 0x7632) : __byte_perm(mine, other, 0x5410);
        const int r = r0 + 2 * j + (odd ? 1 : 0);
        if (col_ok && r < tile_m && m0 + r < M)
            *reinterpret_cast<uint32_t *>(out + (size_t)(m0 + r) * N + col) = w;
    }
}

template <bool BF>
__device__ __forceinline__ void pack_chunk(const uint32_t (&v)[32], uint32_t (&hc)[16]) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if constexpr (BF) {
            const __nv_bfloat162 p =
                __floats2bfloat162_rn(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            hc[j] = *reinterpret_cast<const uint32_t *>(&p);
        } else {
            const __half2 p =
                __floats2half2_rn(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            hc[j] = *reinterpret_cast<const uint32_t *>(&p);
        }
    }
}

// Epilogue of one dequantizing warp for the tile at (m0, n0): its lane quarter
// of the accumulator, columns 32 * part, + 32 * (NDQ / 4), ...  With 8 or 16
// warps the thread's share (at most 64 pairs) is held in registers and the
// accumulator is freed before any store; with 4 warps it is written chunk by
// chunk and freed after.
template <int NDQ, bool BF>
__device__ __forceinline__ void split_epilogue(uint32_t lane_base, int lane, int n, int part,
                                               int m0, int n0, uint64_t *accum_full,
                                               uint64_t *accum_empty, uint32_t parity,
                                               const SplitArgs &a) {
    constexpr int kStep = 32 * (NDQ / 4);
    constexpr int kCh = 256 / kStep;          // chunks of 32 columns per thread (tile_m <= 256)
    if (!mbar_wait_bounded(accum_full, parity, a.timeout_ns))
        report_status(a.status, W4A16_ERR_TIMEOUT);
    tc_fence_after();
    const int col = n0 + (n & ~1);
    const bool col_ok = col < a.N;
    const int first = 32 * part;
    if constexpr (kCh <= 4) {
        uint32_t h[kCh][16];
#pragma unroll
        for (int c = 0; c < kCh; ++c) {
            // columns first + c * kStep < 256: inside the allocation even
            // where they lie past tile_m (those rows are never stored)
            uint32_t v[32];
            tmem_ld_32x32b_x32(lane_base + (uint32_t)(first + c * kStep), v);
            tmem_ld_wait();
            pack_chunk<BF>(v, h[c]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(accum_empty);
#pragma unroll
        for (int c = 0; c < kCh; ++c)
            store_pairs(h[c], first + c * kStep, lane, col, col_ok, m0, a.tile_m, a.M, a.N, a.out);
    } else {
        for (int c = 0; c < kCh; ++c) {
            uint32_t v[32], hc[16];
            tmem_ld_32x32b_x32(lane_base + (uint32_t)(first + c * kStep), v);
            tmem_ld_wait();
            pack_chunk<BF>(v, hc);
            store_pairs(hc, first + c * kStep, lane, col, col_ok, m0, a.tile_m, a.M, a.N, a.out);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(accum_empty);
    }
}

template <int NDQ, bool BF>
__global__ void __launch_bounds__(32 * (NDQ + 3), 1)
prefill_split_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_z,
                     const SplitArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *wring = ring + a.w_off;
    uint64_t *xfull = reinterpret_cast<uint64_t *>(wring + a.ws * a.w_stage_bytes);
    uint64_t *aready = xfull + a.xs;      // the stage's A slot is written
    uint64_t *sempty = aready + a.xs;     // the stage's MMAs completed: x slot and A slot free
    uint64_t *wfull = sempty + a.xs;
    uint64_t *wempty = wfull + a.ws;
    uint64_t *accum_full = wempty + a.ws;
    uint64_t *accum_empty = accum_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum_empty + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KT = (a.K + kStageK - 1) / kStageK;      // 128-k stages (a last half stage reads zeros)

    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_s);
        prefetch_tmap(&tm_z);
        for (int i = 0; i < a.xs; ++i) {
            mbar_init(&xfull[i], 1);
            mbar_init(&aready[i], NDQ);
            mbar_init(&sempty[i], 1);
        }
        for (int i = 0; i < a.ws; ++i) {
            mbar_init(&wfull[i], 1);
            mbar_init(&wempty[i], NDQ);
        }
        mbar_init(accum_full, 1);
        mbar_init(accum_empty, NDQ);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ x producer (lane 0 issues)
        const uint64_t pol_x = l2_evict_last_policy();
        int s = 0, r = 0;
        for (int t = blockIdx.x; t < a.tiles; t += gridDim.x) {
            int m0, n0;
            split_tile(a, t, m0, n0);
            for (int kt = 0; kt < KT; ++kt) {
                if (r > 0 && !mbar_spin_bounded(&sempty[s], (r - 1) & 1, a.timeout_ns))
                    report_status(a.status, W4A16_ERR_TIMEOUT);
                if (lane == 0) {
                    mbar_arrive_expect_tx(&xfull[s], (uint32_t)a.x_stage_bytes);
                    // both 64-k chunks in one 3-D box (chunk index outermost)
                    tma_load_3d(ring + s * a.x_stage_bytes, &tm_x, &xfull[s], 0, m0, kt * kChunks,
                                pol_x);
                }
                __syncwarp();
                if (++s == a.xs) { s = 0; ++r; }
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------ weight producer
        const uint64_t pol_w = l2_evict_first_policy();
        int s = 0, r = 0;
        for (int t = blockIdx.x; t < a.tiles; t += gridDim.x) {
            int m0, n0;
            split_tile(a, t, m0, n0);
            int grow = 0, gnext = a.group;
            for (int kt = 0; kt < KT; ++kt) {
                const int k0 = kt * kStageK;
                while (k0 >= gnext) { ++grow; gnext += a.group; }
                if (r > 0 && !mbar_wait_bounded(&wempty[s], (r - 1) & 1, a.timeout_ns))
                    report_status(a.status, W4A16_ERR_TIMEOUT);
                if (lane == 0) {
                    uint8_t *st = wring + s * a.w_stage_bytes;
                    mbar_arrive_expect_tx(&wfull[s], (uint32_t)a.w_tx);
                    tma_load_2d(st, &tm_w, &wfull[s], n0, k0 / 8, pol_w);
                    tma_load_2d(st + a.s_off, &tm_s, &wfull[s], n0, grow, pol_w);
                    tma_load_2d(st + a.z_off, &tm_z, &wfull[s], n0, grow, pol_w);
                }
                __syncwarp();
                if (++s == a.ws) { s = 0; ++r; }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (lane 0 issues)
        const uint32_t idesc = idesc_f16(128, a.tile_m, BF);
        const uint32_t tmem_u = __shfl_sync(0xffffffffu, tmem_d, 0);
        const uint32_t ring_u = smem_u32(ring);
        const uint32_t chunk16 = (uint32_t)a.x_chunk_bytes >> 4;
        int s = 0, r = 0, it = 0;
        for (int t = blockIdx.x; t < a.tiles; t += gridDim.x, ++it) {
            // the epilogue of the previous tile has read the accumulator out
            if (it > 0 && !mbar_spin_bounded(accum_empty, (it - 1) & 1, a.timeout_ns))
                report_status(a.status, W4A16_ERR_TIMEOUT);
            for (int kt = 0; kt < KT; ++kt) {
                if (!mbar_spin_bounded(&aready[s], r & 1, a.timeout_ns))
                    report_status(a.status, W4A16_ERR_TIMEOUT);
                if (!mbar_spin_bounded(&xfull[s], r & 1, a.timeout_ns))
                    report_status(a.status, W4A16_ERR_TIMEOUT);
                tc_fence_after();
                const uint64_t b_desc = smem_desc_sw128(ring_u + (uint32_t)(s * a.x_stage_bytes));
                const uint32_t a_tmem = tmem_u + (uint32_t)(a.a_col0 + s * (kStageK / 2));
                if (lane == 0) {
                    // descriptors advance in 16-byte units: 32 bytes per k16
                    // step inside a chunk, a whole chunk between chunks
#pragma unroll
                    for (int kk = 0; kk < kStageK / 16; ++kk)
                        umma_f16_ts(tmem_u, a_tmem + kk * 8,
                                       b_desc + (kk / 4) * chunk16 + (kk % 4) * 2, idesc,
                                       (kt | kk) != 0);
                    umma_commit(&sempty[s]);
                }
                __syncwarp();
                if (++s == a.xs) { s = 0; ++r; }
            }
            if (lane == 0) umma_commit(accum_full);
            __syncwarp();
        }
    } else {
        // ------------------------------------------------ dequant + epilogue
        constexpr int kParts = NDQ / 4;                   // warps per lane quarter
        static_assert(kPackedRows % kParts == 0, "packed rows must split evenly");
        constexpr int kRowsPer = kPackedRows / kParts;    // packed rows per thread
        constexpr int kBlk = kRowsPer >= 8 ? 8 : 4;       // words per TMEM store
        // a warp may only reach its lane quarter (warp % 4): the column a
        // thread dequantizes is the TMEM lane of that quarter
        const int n = (warp & 3) * 32 + lane;
        const int part = (warp - kSplitDeq0) / 4;
        const uint32_t lane_base = tmem_d + ((uint32_t)((warp & 3) * 32) << 16);
        // the previous tile's epilogue comes before the dequantization of
        // this tile's stage `ep_at`: the first one whose A slot is freed by
        // the previous tile's last MMAs (earlier stages overlap those MMAs)
        const int ep_at = (a.xs - 1 < KT - 1) ? a.xs - 1 : KT - 1;
        int sw = 0, rw = 0, s = 0, r = 0, it = 0, pm0 = 0, pn0 = 0;
        auto stage = [&](int kt) {
            if (!mbar_wait_bounded(&wfull[sw], rw & 1, a.timeout_ns))
                report_status(a.status, W4A16_ERR_TIMEOUT);
            // the A slot is free once the MMAs that read it last have completed
            if (r > 0 && !mbar_wait_bounded(&sempty[s], (r - 1) & 1, a.timeout_ns))
                report_status(a.status, W4A16_ERR_TIMEOUT);
            tc_fence_after();
            const uint32_t st = smem_u32(wring + sw * a.w_stage_bytes);
            const int k0 = kt * kStageK;
#pragma unroll
            for (int b0 = 0; b0 < kRowsPer; b0 += kBlk) {
                const int c0 = part * kRowsPer + b0;
                uint32_t h[kBlk * 4];
                dequant_words<kBlk, BF>(st, 0, a.s_off, a.z_off, c0, stage_zrow(k0, a.group, c0), n, h);
                tmem_st_32x32b<kBlk * 4>(
                    lane_base + (uint32_t)(a.a_col0 + s * (kStageK / 2) + c0 * 4), h);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&wempty[sw]);     // the words are in registers (and stored)
                mbar_arrive(&aready[s]);
            }
            if (++sw == a.ws) { sw = 0; ++rw; }
            if (++s == a.xs) { s = 0; ++r; }
        };
        for (int t = blockIdx.x; t < a.tiles; t += gridDim.x, ++it) {
            int kt = 0;
            if (it > 0) {
                for (; kt < ep_at; ++kt) stage(kt);
                split_epilogue<NDQ, BF>(lane_base, lane, n, part, pm0, pn0, accum_full, accum_empty,
                                    (uint32_t)((it - 1) & 1), a);
            }
            for (; kt < KT; ++kt) stage(kt);
            split_tile(a, t, pm0, pn0);
        }
        if (it > 0)
            split_epilogue<NDQ, BF>(lane_base, lane, n, part, pm0, pn0, accum_full, accum_empty,
                                (uint32_t)((it - 1) & 1), a);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem_d, a.tmem_cols);
}

int round_up(int v, int m) { return (v + m - 1) / m * m; }

template <int NDQ, bool ATMEM, bool BF>
cudaError_t launch_prefill_kernel(dim3 grid, size_t smem, cudaStream_t stream,
                                  const CUtensorMap &tx, const CUtensorMap &tw,
                                  const CUtensorMap &ts, const CUtensorMap &tz,
                                  const CUtensorMap &to, const PrefillArgs &pa) {
    if (pa.split <= 1) {
        const cudaError_t attr = ensure_dynamic_smem(
            (const void *)prefill_tcgen05_kernel<NDQ, ATMEM, false, BF>, 227 * 1024);
        if (attr != cudaSuccess) return attr;
        prefill_tcgen05_kernel<NDQ, ATMEM, false, BF><<<grid, 32 * (NDQ + 2), smem, stream>>>(
            tx, tw, ts, tz, to, pa);
        return cudaGetLastError();
    }
    if constexpr (!ATMEM) {
        return cudaErrorNotSupported;     // split-K is built for A in tensor memory only
    } else {
    const cudaError_t attr =
        ensure_dynamic_smem((const void *)prefill_tcgen05_kernel<NDQ, ATMEM, true, BF>, 227 * 1024);
    if (attr != cudaSuccess) return attr;
    // split-K: the CTAs of one output tile form a cluster along z
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = dim3(32 * (NDQ + 2), 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attr1[1];
    attr1[0].id = cudaLaunchAttributeClusterDimension;
    attr1[0].val.clusterDim.x = 1;
    attr1[0].val.clusterDim.y = 1;
    attr1[0].val.clusterDim.z = (unsigned)pa.split;
    lc.attrs = attr1;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, prefill_tcgen05_kernel<NDQ, ATMEM, true, BF>, tx, tw, ts, tz, to, pa);
    }
}

template <int NDQ, bool BF>
cudaError_t launch_split_kernel(dim3 grid, size_t smem, cudaStream_t stream,
                                const CUtensorMap &tx, const CUtensorMap &tw,
                                const CUtensorMap &ts, const CUtensorMap &tz, const SplitArgs &sa) {
    const cudaError_t attr =
        ensure_dynamic_smem((const void *)prefill_split_kernel<NDQ, BF>, 227 * 1024);
    if (attr != cudaSuccess) return attr;
    prefill_split_kernel<NDQ, BF><<<grid, 32 * (NDQ + 3), smem, stream>>>(tx, tw, ts, tz, sa);
    return cudaGetLastError();
}


// Shared-memory and tensor-memory layout of the one-ring kernel for `cfg`
// (tile_m, variant, split_k) and K; false when it does not fit.
bool ring_layout(const w4a16_config &cfg, int K, int group, PrefillArgs &pa) {
    pa.tile_m = cfg.tile_m;
    // A operand in tensor memory unless the caller asks for shared memory
    const bool atmem = cfg.variant != W4A16_PREFILL_A_SMEM;
    // stage (128 k): [A (dequantized W^T, two 128 x 64 fp16 chunks) when in
    // shared memory] | B (x tile: two tile_m x 64 fp16 chunks) | packed words
    // (16 x 128) | scale rows | zero rows (1, or 2 when group % 128 != 0)
    const int a_bytes = atmem ? 0 : kTileN * kStageK * 2;
    pa.b_chunk_bytes = pa.tile_m * kChunkK * 2;              // tile_m % 16 == 0: 1024-aligned
    pa.sz_rows = group % kStageK == 0 ? 1 : 2;
    pa.b_off = a_bytes;
    pa.p_off = pa.b_off + kChunks * pa.b_chunk_bytes;
    pa.s_off = pa.p_off + kPackedRows * kTileN * 4;
    pa.z_off = pa.s_off + pa.sz_rows * kTileN * 2;
    pa.stage_bytes = round_up(pa.z_off + pa.sz_rows * kTileN * 2, 1024);
    pa.tx_bytes = kChunks * pa.b_chunk_bytes + kPackedRows * kTileN * 4 + 2 * pa.sz_rows * kTileN * 2;
    // split-K across a cluster of `split` CTAs along z, each with kt_per of
    // the 128-k stages (every CTA gets at least one); the leader keeps the
    // others' fp32 partials [split - 1][tile_m][128] after its ring
    const int KT = (K + kStageK - 1) / kStageK;
    int split = cfg.split_k > 1 ? cfg.split_k : 1;
    if (split > kMaxPrefillSplit) return false;
    pa.kt_per = (KT + split - 1) / split;
    split = (KT + pa.kt_per - 1) / pa.kt_per;
    pa.split = split;
    const int red_bytes = (split - 1) * pa.tile_m * kTileN * 4;
    pa.a_col0 = round_up(pa.tile_m, 32);
    // Narrow tiles (up to 64 rows of x) are bound by the per-stage control
    // path, not by the tensor core: two CTAs share an SM (half of its shared
    // memory and of its tensor memory each), which doubles the stages in
    // flight per SM -- unless a split leader's partial slots leave that half
    // room for fewer than two stages.  Wider tiles take the whole SM.
    auto ring_stages = [&](bool two_per_sm) {
        const int budget = two_per_sm ? 104 * 1024 : 224 * 1024;
        const int tmem_max = two_per_sm ? 256 : 512;
        int st = (budget - red_bytes) / pa.stage_bytes;
        st = st > 8 ? 8 : st;
        // tensor memory: the accumulator (tile_m fp32 columns) and, with A in
        // tensor memory, one 64-column A slot per stage
        if (atmem) {
            const int max_stages = (tmem_max - pa.a_col0) / (kStageK / 2);
            st = st > max_stages ? max_stages : st;
        }
        return st;
    };
    int stages = ring_stages(atmem && pa.tile_m <= kTwoPerSmMaxTileM);
    if (stages < 2) stages = ring_stages(false);
    if (stages < 2) return false;
    pa.stages = stages;
    const int need = atmem ? pa.a_col0 + stages * (kStageK / 2) : pa.tile_m;
    int cols = 32;
    while (cols < need) cols *= 2;
    pa.tmem_cols = cols;
    // a split partner stages its fp32 partial in its drained ring
    if (split > 1 && stages * pa.stage_bytes < pa.tile_m * kTileN * 4) return false;
    pa.red_off = stages * pa.stage_bytes;
    pa.bar_off = pa.red_off + red_bytes;
    return true;
}

}  // namespace

bool prefill_config_supported(const w4a16_config &cfg, int M, int N, int K, int group) {
    if (cfg.split_k < 0 || cfg.split_k > kMaxPrefillSplit) return false;
    if (cfg.split_k > 1 && cfg.variant == W4A16_PREFILL_A_SMEM) return false;
    if (cfg.dtype != W4A16_DTYPE_F16 && cfg.dtype != W4A16_DTYPE_BF16) return false;
    if (cfg.dtype == W4A16_DTYPE_BF16 && cfg.variant == W4A16_PREFILL_A_SMEM) return false;
    if (cfg.variant != 0 && cfg.variant != W4A16_PREFILL_A_TMEM &&
        cfg.variant != W4A16_PREFILL_A_SMEM)
        return false;
    const bool warps_ok = cfg.warps_k == 0 || cfg.warps_k == 4 || cfg.warps_k == 8 ||
                          cfg.warps_k == 16;
    if (!(warps_ok && cfg.tile_m >= 16 && cfg.tile_m <= 256 && cfg.tile_m % 16 == 0 &&
          group % kChunkK == 0 && K % kChunkK == 0 && N % 8 == 0 && (K / group) >= 1))
        return false;
    // the one-ring kernel (narrow tiles, A in shared memory, or split-K) must
    // fit its ring and a split leader's partial slots
    const bool one_ring = cfg.variant == W4A16_PREFILL_A_SMEM || cfg.split_k > 1 ||
                          cfg.tile_m < kSplitMinTileM;
    PrefillArgs pa;
    return !one_ring || ring_layout(cfg, K, group, pa);
}

// Default variant (A in tensor memory) for wide tiles: the split-ring kernel.
cudaError_t launch_prefill_split(const GemmArgs &a, const w4a16_config &cfg, cudaStream_t stream) {
    SplitArgs sa;
    sa.status = device_status_word();
    if (!sa.status) return cudaErrorInvalidDevice;
    sa.M = a.M;
    sa.N = a.N;
    sa.K = a.K;
    sa.group = a.group;
    sa.tile_m = cfg.tile_m;
    sa.out = a.out;
    sa.n_tiles = (a.N + kTileN - 1) / kTileN;
    const int ndq = cfg.warps_k > 0 ? cfg.warps_k : 8;
    sa.sz_rows = a.group % kStageK == 0 ? 1 : 2;
    sa.x_chunk_bytes = sa.tile_m * kChunkK * 2;                // tile_m % 16 == 0: 1024-aligned
    sa.x_stage_bytes = kChunks * sa.x_chunk_bytes;
    sa.s_off = kPackedRows * kTileN * 4;
    sa.z_off = sa.s_off + sa.sz_rows * kTileN * 2;
    sa.w_stage_bytes = round_up(sa.z_off + sa.sz_rows * kTileN * 2, 1024);
    sa.w_tx = kPackedRows * kTileN * 4 + 2 * sa.sz_rows * kTileN * 2;
    // stage slots: as many x tiles as shared memory holds next to a weight
    // ring of three, and no more A stages than tensor memory holds next to
    // the accumulator (tile_m fp32 columns); then the weight ring takes what
    // shared memory is left (deep for narrow tiles, whose small x slots leave
    // room to keep more weight bytes in flight)
    const int budget = 224 * 1024;
    int xs = (budget - 3 * sa.w_stage_bytes) / sa.x_stage_bytes;
    sa.a_col0 = round_up(sa.tile_m, 32);
    const int a_max = (512 - sa.a_col0) / (kStageK / 2);
    xs = xs > a_max ? a_max : xs;
    sa.xs = xs > 8 ? 8 : xs;
    if (sa.xs < 2) return cudaErrorNotSupported;
    int ws = (budget - sa.xs * sa.x_stage_bytes) / sa.w_stage_bytes;
    sa.ws = ws > kMaxWeightSlots ? kMaxWeightSlots : ws;
    int cols = 32;
    while (cols < sa.a_col0 + sa.xs * (kStageK / 2)) cols *= 2;
    sa.tmem_cols = cols;
    sa.w_off = sa.xs * sa.x_stage_bytes;
    sa.timeout_ns = 1000000000ull;
    const size_t smem = (size_t)sa.w_off + (size_t)sa.ws * sa.w_stage_bytes +
                        (3 * sa.xs + 2 * sa.ws + 2) * 8 + 16 + 1024;

    const uint64_t x_dims[3] = {(uint64_t)kChunkK, (uint64_t)a.M, (uint64_t)(a.K / kChunkK)};
    const uint64_t x_strides[2] = {(uint64_t)a.K * 2, (uint64_t)kChunkK * 2};
    const uint32_t x_box[3] = {(uint32_t)kChunkK, (uint32_t)sa.tile_m, (uint32_t)kChunks};
    const bool bf = cfg.dtype == W4A16_DTYPE_BF16;
    const CUtensorMapDataType et = bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tx, tw, ts, tz;
    if (!make_tmap(&tx, et, 3, a.x, x_dims, x_strides, x_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.packed, a.N, a.K / 8,
                      (uint64_t)a.N * 4, kTileN, kPackedRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&ts, et, a.scales, a.N, a.K / a.group, (uint64_t)a.N * 2, kTileN,
                      sa.sz_rows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&tz, et, a.zeros, a.N, a.K / a.group, (uint64_t)a.N * 2, kTileN,
                      sa.sz_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    // persistent: one CTA per SM (at most one per tile)
    sa.m_tiles = (a.M + sa.tile_m - 1) / sa.tile_m;
    // row tiles per group of the tile order: as many as keep the group's x
    // rows (tile_m x K fp16 each) within 32 MB, a quarter of the L2
    const long long x_tile_bytes = (long long)sa.tile_m * a.K * 2;
    long long gm = (32ll << 20) / x_tile_bytes;
    gm = gm < 1 ? 1 : (gm > sa.m_tiles ? sa.m_tiles : gm);
    sa.gm = (int)gm;
    const long long tiles = (long long)sa.n_tiles * sa.m_tiles;
    if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
    sa.tiles = (int)tiles;
    const int sms = device_info().sm_count;
    dim3 grid(sa.tiles < sms ? sa.tiles : sms, 1, 1);
#define W4A16_SPLIT(NDQ_)                                                          \
    (bf ? launch_split_kernel<NDQ_, true>(grid, smem, stream, tx, tw, ts, tz, sa) \
        : launch_split_kernel<NDQ_, false>(grid, smem, stream, tx, tw, ts, tz, sa))
    switch (ndq) {
    case 4: return W4A16_SPLIT(4);
    case 16: return W4A16_SPLIT(16);
    default: return W4A16_SPLIT(8);
    }
#undef W4A16_SPLIT
}

cudaError_t launch_prefill(const GemmArgs &a, const w4a16_config &cfg, cudaStream_t stream) {
    if (!prefill_config_supported(cfg, a.M, a.N, a.K, a.group)) return cudaErrorNotSupported;
    // Wide tiles: the split-ring kernel (its x ring runs far enough ahead to
    // cover the copy latency at 1024+ MMA cycles per stage).  Narrower tiles
    // are bound by the per-stage control path instead, where one ring (one
    // wait and one commit per stage) is cheaper (measured: 11-13% faster at
    // M = 32..128, K=4096 N=14336, than the split-ring kernel with a deep
    // weight ring); split-K runs on the one-ring kernel too.
    if (cfg.variant != W4A16_PREFILL_A_SMEM && cfg.split_k <= 1 && cfg.tile_m >= kSplitMinTileM)
        return launch_prefill_split(a, cfg, stream);
    PrefillArgs pa;
    if (!ring_layout(cfg, a.K, a.group, pa)) return cudaErrorNotSupported;
    pa.out = a.out;
    pa.status = device_status_word();
    if (!pa.status) return cudaErrorInvalidDevice;
    pa.M = a.M;
    pa.N = a.N;
    pa.K = a.K;
    pa.group = a.group;
    pa.timeout_ns = 1000000000ull;
    const bool atmem = cfg.variant != W4A16_PREFILL_A_SMEM;
    const int ndq = cfg.warps_k > 0 ? cfg.warps_k : 8;
    const size_t smem = (size_t)pa.bar_off + (3 * pa.stages + 2) * 8 + 16 + 1024;
    const int split = pa.split;

    // x as a 3-D view {64 k, M rows, K/64 chunks}: one box brings both 64-k
    // chunks of a stage, each a 128B-swizzled K-major tile
    const uint64_t x_dims[3] = {(uint64_t)kChunkK, (uint64_t)a.M, (uint64_t)(a.K / kChunkK)};
    const uint64_t x_strides[2] = {(uint64_t)a.K * 2, (uint64_t)kChunkK * 2};
    const uint32_t x_box[3] = {(uint32_t)kChunkK, (uint32_t)pa.tile_m, (uint32_t)kChunks};
    const bool bf = cfg.dtype == W4A16_DTYPE_BF16;
    if (bf && !atmem) return cudaErrorNotSupported;   // bfloat16: A in tensor memory only
    const CUtensorMapDataType et = bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tx, tw, ts, tz, to;
    if (!make_tmap(&tx, et, 3, a.x, x_dims, x_strides, x_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&to, et, a.out, a.N, a.M, (uint64_t)a.N * 2, kTileN, pa.tile_m,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.packed, a.N, a.K / 8,
                      (uint64_t)a.N * 4, kTileN, kPackedRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&ts, et, a.scales, a.N, a.K / a.group, (uint64_t)a.N * 2, kTileN,
                      pa.sz_rows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&tz, et, a.zeros, a.N, a.K / a.group, (uint64_t)a.N * 2, kTileN,
                      pa.sz_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;

    const int mtiles = (a.M + pa.tile_m - 1) / pa.tile_m;
    if (mtiles > 65535) return cudaErrorInvalidValue;
    dim3 grid((a.N + kTileN - 1) / kTileN, mtiles, split);
#define W4A16_PF(NDQ_, AT_) \
    launch_prefill_kernel<NDQ_, AT_, false>(grid, smem, stream, tx, tw, ts, tz, to, pa)
#define W4A16_PF_BF(NDQ_) \
    launch_prefill_kernel<NDQ_, true, true>(grid, smem, stream, tx, tw, ts, tz, to, pa)
    if (bf) {
        switch (ndq) {
        case 4: return W4A16_PF_BF(4);
        case 16: return W4A16_PF_BF(16);
        default: return W4A16_PF_BF(8);
        }
    }
    if (atmem) {
        switch (ndq) {
        case 4: return W4A16_PF(4, true);
        case 16: return W4A16_PF(16, true);
        default: return W4A16_PF(8, true);
        }
    }
    switch (ndq) {
    case 4: return W4A16_PF(4, false);
    case 16: return W4A16_PF(16, false);
    default: return W4A16_PF(8, false);
    }
#undef W4A16_PF
#undef W4A16_PF_BF
}

}  // namespace w4a16
