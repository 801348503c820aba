// decode_stream.cu -- the decode-regime W4A16 GEMM (M <= 16) as one persistent
// weight stream per SM.
//
// What it computes: out[m,n] = sum_k x[m,k] * (q[k,n] - z[g(k),n]) * s[g(k),n],
// fp32 accumulation, fp16 result (page "Beating FP16 with 4-bit Weights: A
// Portable W4A16 GEMM in Triton", sections "The design" and "What's next";
// page "Triton Kernel Matches bitsandbytes: Why Both Lose to Math", sections
// "Roofline First" and "Why Marlin Is Still Faster").  Same per-step arithmetic
// as the other decode kernels (decode_math.cuh: magic-exponent unpack, exact
// q - z in fp16, register-fed mma.m16n8k16 with swapped roles, one fp32 scale
// per group); what differs is how the work and the bytes move:
//
//   * Work units.  The weight is cut into column tiles of 32*BNS columns and
//     each tile into stages of 16 KB of packed words (128/BNS packed rows).
//     The grid is at most one CTA per SM and every CTA takes one contiguous
//     run of (tile, stage) units: either whole tiles (no tile is shared, the
//     CTA writes its outputs directly) or an equal share of all units
//     ("stream-K": a tile may be shared by two or more CTAs, whose fp32
//     partials meet in a scratch buffer and are summed in CTA order by the
//     last of them to arrive -- a fixed order, so the result is bitwise
//     reproducible).  A grid of one wave means the next call's CTAs can be
//     resident at the same time (each CTA takes under half an SM).
//   * Data movement.  One producer warp issues 1-D bulk copies (cp.async.bulk,
//     one per packed row with the natural layout, one per 32-column strip with
//     the repacked layout) into a ring of shared-memory stages guarded by
//     mbarriers.  No tensor maps: the host encodes nothing per call, and the
//     operands of up to 64 experts fit in the kernel parameters.  With
//     programmatic dependent launch the weights of the first ring's worth of
//     stages are requested before the wait for the previous kernel; x (and
//     out) wait for it.
//   * Layouts.  Natural: packed [K/8, N] row-major; rows land in shared memory
//     with a 32-byte pad so that the consumers' 128-bit reads are free of bank
//     conflicts.  Repacked (the pre-permuted layout of w4a16_repack): each
//     lane's 128-bit read is its MMA fragment, the nibbles are ordered so that
//     x enters the MMA as it sits in memory (no byte permutes), and a stage is
//     one contiguous block per strip with the scales and zeros inside.
//   * Every mbarrier wait is bounded in wall time (counted from after the wait
//     for the previous kernel); a wait that gives up records W4A16_ERR_TIMEOUT
//     in the device status word and the kernel runs to its end without
//     touching memory it does not own.  There is no spin on another CTA: the
//     cross-CTA sum uses an atomic arrival count, and only the last arrival
//     (which needs nobody else) reads the partials.
#include <mutex>
#include <string.h>

#include "common.cuh"
#include "decode_math.cuh"
#include "sm100_ptx.cuh"
#include "tmap.cuh"

namespace w4a16 {
namespace {

constexpr int kCW = 8;                      // consumer warps per CTA
constexpr int kThreads = 32 * (kCW + 1);    // + one producer warp
constexpr int kSPW = 4;                     // 32-k steps per consumer warp per stage
constexpr int kBudget = 110 * 1024;         // shared memory per CTA: two CTAs per SM
constexpr int kMaxStages = 8;
constexpr int kMaxGrid = 512;               // CTAs per launch (scratch is sized for it)
constexpr int kPermBlockWordBytes = 4096;   // repacked block: 1024 words, then scales/zeros

// Where the weights come from and how they land in shared memory.
enum Layout : int {
    kRows = 0,    // natural [K/8, N]: one bulk copy per packed row, rows padded by 32 bytes
    kTma = 1,     // natural [K/8, N]: one TMA box per stage, 128-byte swizzled 32-column strips
    kPerm = 2,    // repacked blocks: one bulk copy per strip and stage
};

// consumer lane group g reads 16-byte chunk perm8(g) of a 128-byte swizzled
// row (with the row's swizzle this keeps every 128-bit read conflict-free)
__device__ __forceinline__ int perm8(int g) { return (g >> 1) + ((g & 1) << 2); }

struct StreamArgs {
    int M, N, K, group;
    int T, KS;            // column tiles per expert, stages per tile
    int U;                // units = experts * T * KS
    int align;            // 1: every CTA takes whole tiles
    int stages, stage_bytes;
    int w_pitch;          // natural: bytes per packed row in a slot
    int sz_off, sz_rows;  // natural: sz_rows scale rows of the stage at sz_off,
    int z_delta;          //   its zero rows z_delta bytes further (a multiple of 128)
    int x_off, x_pitch;   // x rows of a stage
    int blk_bytes;        // repacked: bytes per 32-column x 256-k block
    int red_off, bar_off;
    float *scratch;       // shared tiles: [2 * gridDim.x][M][BN] fp32 partials
    int *counters;        // shared tiles: arrivals per tile (back to 0 after the last)
    int *status;
    unsigned long long timeout_ns;
    int test_skip_last;   // test hook: arm but never load the CTA's last stage
};

struct StreamOperands {
    const uint16_t *x;
    const uint32_t *w;        // natural: packed [K/8, N]; repacked: the block array
    const uint16_t *s, *z;    // natural layout only
    uint16_t *out;
};

template <int MAXE>
struct StreamTable {
    StreamOperands e[MAXE];
};

// Position of a unit: expert, column tile, stage.  Units are numbered
// expert-major, then tile, then stage.
struct UnitPos {
    int e, tile, ks;
};

__device__ __forceinline__ UnitPos unit_pos(long long u, int T, int KS) {
    const int tg = (int)(u / KS);
    UnitPos p;
    p.ks = (int)(u - (long long)tg * KS);
    p.e = tg / T;
    p.tile = tg - p.e * T;
    return p;
}

__device__ __forceinline__ void advance(UnitPos &p, int T, int KS) {
    if (++p.ks == KS) {
        p.ks = 0;
        if (++p.tile == T) {
            p.tile = 0;
            ++p.e;
        }
    }
}

// First unit of CTA c of G.
__device__ __forceinline__ long long range_begin(int c, int G, const StreamArgs &a) {
    if (a.align) {
        const long long tiles = a.U / a.KS;
        return (long long)c * tiles / G * a.KS;
    }
    return (long long)c * a.U / G;
}

// The CTA whose (stream-K) range holds unit u: the largest c with
// floor(c * U / G) <= u.
__device__ __forceinline__ int cta_of(long long u, int G, int U) {
    return (int)(((u + 1) * G + U - 1) / U - 1);
}

// One 32-k step (decode_math.cuh's fragment mapping): the thread's four words
// become the A operands of two MMA tiles x two k halves; KH = 2 keeps the k
// halves in separate accumulators, KH = 1 adds them into one.
template <bool FIRST, int NT, int KH>
__device__ __forceinline__ void stream_step(float (&gacc)[NT][2][KH][4], uint4 w,
                                            const GroupConsts &k, const uint32_t (&bx)[NT][4]) {
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t c0 = wv[2 * j], c1 = wv[2 * j + 1];
        const uint32_t d0 = c0 >> 8, d1 = c1 >> 8;
        const uint32_t a0 = hsub2_u32(lop3_and_or(c0, kMaskLo, kMagicLo), k.zA[2 * j]);
        const uint32_t a1 = hsub2_u32(lop3_and_or(c1, kMaskLo, kMagicLo), k.zA[2 * j + 1]);
        const uint32_t a2 = hsub2_u32(lop3_and_or(c0, kMaskHi, kMagicHi), k.zB[2 * j]);
        const uint32_t a3 = hsub2_u32(lop3_and_or(c1, kMaskHi, kMagicHi), k.zB[2 * j + 1]);
        const uint32_t e0 = hsub2_u32(lop3_and_or(d0, kMaskLo, kMagicLo), k.zA[2 * j]);
        const uint32_t e1 = hsub2_u32(lop3_and_or(d1, kMaskLo, kMagicLo), k.zA[2 * j + 1]);
        const uint32_t e2 = hsub2_u32(lop3_and_or(d0, kMaskHi, kMagicHi), k.zB[2 * j]);
        const uint32_t e3 = hsub2_u32(lop3_and_or(d1, kMaskHi, kMagicHi), k.zB[2 * j + 1]);
#pragma unroll
        for (int p = 0; p < NT; ++p) {
            mma_acc<FIRST>(gacc[p][j][0], a0, a1, a2, a3, bx[p][0], bx[p][1]);
            if (KH == 2)
                mma_acc<FIRST>(gacc[p][j][KH - 1], e0, e1, e2, e3, bx[p][2], bx[p][3]);
            else
                mma_16816(gacc[p][j][0], e0, e1, e2, e3, bx[p][2], bx[p][3]);
        }
    }
}
template <int NT, int KH>
__device__ __forceinline__ void step_first(float (&g)[NT][2][KH][4], uint4 w, const GroupConsts &k,
                                           const uint32_t (&bx)[NT][4]) {
    stream_step<true, NT, KH>(g, w, k, bx);
}
template <int NT, int KH>
__device__ __forceinline__ void step(float (&g)[NT][2][KH][4], uint4 w, const GroupConsts &k,
                                     const uint32_t (&bx)[NT][4]) {
    stream_step<false, NT, KH>(g, w, k, bx);
}
// acc += s * (sum of the k halves): the group scale, once per group, in fp32.
template <int NT, int KH>
__device__ __forceinline__ void flush(float (&acc)[NT][2][4], const float (&g)[NT][2][KH][4],
                                      const GroupConsts &k) {
#pragma unroll
    for (int p = 0; p < NT; ++p)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r)
                acc[p][j][r] = fmaf(k.sc[2 * j + (r >> 1)],
                                    KH == 2 ? g[p][j][0][r] + g[p][j][KH - 1][r] : g[p][j][0][r],
                                    acc[p][j][r]);
}

constexpr bool kZeroFree = true;   // M <= 8: the zero-free step of decode_math.cuh

template <int NT, int BNS, int LAY, bool OG, int MAXE>
__global__ void __launch_bounds__(kThreads, 2)
decode_stream_kernel(const __grid_constant__ StreamArgs a,
                     const __grid_constant__ StreamTable<MAXE> tab,
                     const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_s,
                     const __grid_constant__ CUtensorMap tm_z)
{
    constexpr bool PERM = LAY == kPerm;
    constexpr bool TMAW = LAY == kTma;
    constexpr int BN = 32 * BNS;           // columns per tile
    constexpr int WK = kCW / BNS;          // consumer warps along a stage's steps
    constexpr int RS = 4 * kSPW * WK;      // packed rows per stage (128 / BNS)
    constexpr int SK = 8 * RS;             // k per stage
    constexpr int R = RS / 32;             // repacked 256-k blocks per stage
    constexpr int WP = BN * 4 + 32;        // natural: bytes per packed row in a slot
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // slots start on a 1024-byte boundary (the span of the 128-byte swizzle)
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.bar_off);
    uint64_t *empty = full + a.stages;
    int *last_flag = reinterpret_cast<int *>(empty + a.stages);
    float *red = reinterpret_cast<float *>(smem + a.red_off);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const long long ub = range_begin(cta, G, a), ue = range_begin(cta + 1, G, a);
    const int n_units = (int)(ue - ub);

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kCW);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kCW) {
        // ---------------------------------------------------------- producer
        // The whole warp runs the loop; lane 0 arms each stage's barrier, then
        // the lanes issue the stage's copies in parallel.
        if (TMAW && lane == 0) {
            prefetch_tmap(&tm_w);
            prefetch_tmap(&tm_s);
            prefetch_tmap(&tm_z);
        }
        const uint64_t pol_w = l2_evict_first_policy();
        const uint64_t pol_x = l2_evict_last_policy();
        const uint32_t ring = smem_u32(smem);
        const int skip = (a.test_skip_last && n_units > 0) ? n_units - 1 : -1;
        const int first = n_units < a.stages ? n_units : a.stages;

        auto shape_of = [&](const UnitPos &p, int &ncols, int &nrows, int &k0, int &klen) {
            const int col0 = p.tile * BN;
            ncols = a.N - col0 < BN ? a.N - col0 : BN;
            k0 = p.ks * SK;
            klen = a.K - k0 < SK ? a.K - k0 : SK;
            nrows = klen >> 3;
        };
        auto stage_bytes = [&](const UnitPos &p) -> uint32_t {
            int ncols, nrows, k0, klen;
            shape_of(p, ncols, nrows, k0, klen);
            uint32_t b = (uint32_t)(a.M * klen * 2);
            if (PERM) {
                const int strips = ncols >> 5;
                b += (uint32_t)(strips * (klen >> 8) * a.blk_bytes);
            } else if (TMAW) {
                // whole boxes count, including rows or strips past the tensor
                b += (uint32_t)(BNS * RS * 128 + 2 * a.sz_rows * BN * 2);
            } else {
                const int ngr = (k0 + klen - 1) / a.group - k0 / a.group + 1;
                b += (uint32_t)(nrows * ncols * 4 + 2 * ngr * ncols * 2);
            }
            return b;
        };
        auto issue_weights = [&](uint32_t slot, const UnitPos &p, uint64_t *bar) {
            const StreamOperands &op = tab.e[p.e];
            int ncols, nrows, k0, klen;
            shape_of(p, ncols, nrows, k0, klen);
            const uint32_t mb = smem_u32(bar);
            if (TMAW) {
                if (lane == 0) {
                    uint8_t *dst = smem + (slot - ring);
                    tma_load_3d(dst, &tm_w, bar, 0, p.ks * RS, p.tile * BNS, pol_w);
                    const int gr0 = k0 / a.group;
                    tma_load_2d(dst + a.sz_off, &tm_s, bar, p.tile * BN, gr0, pol_w);
                    tma_load_2d(dst + a.sz_off + a.z_delta, &tm_z, bar, p.tile * BN, gr0, pol_w);
                }
            } else if (PERM) {
                const int strips = ncols >> 5, nr = klen >> 8;
                const int ks256 = a.K >> 8;
                for (int s = lane; s < strips; s += 32) {
                    const uint8_t *src = reinterpret_cast<const uint8_t *>(op.w) +
                                         ((size_t)(p.tile * BNS + s) * ks256 + (size_t)p.ks * R) *
                                             a.blk_bytes;
                    bulk_load(slot + s * R * a.blk_bytes, src, (uint32_t)(nr * a.blk_bytes), mb,
                              pol_w);
                }
            } else {
                const int col0 = p.tile * BN;
                const uint32_t *wsrc = op.w + (size_t)(p.ks * RS) * a.N + col0;
                for (int r = lane; r < nrows; r += 32)
                    bulk_load(slot + r * a.w_pitch, wsrc + (size_t)r * a.N, (uint32_t)ncols * 4, mb,
                              pol_w);
                const int gr0 = k0 / a.group;
                const int ngr = (k0 + klen - 1) / a.group - gr0 + 1;
                for (int i = lane; i < 2 * ngr; i += 32) {
                    const bool zr = i >= ngr;
                    const int gi = zr ? i - ngr : i;
                    const uint16_t *src = (zr ? op.z : op.s) + (size_t)(gr0 + gi) * a.N + col0;
                    bulk_load(slot + a.sz_off + (zr ? a.z_delta : 0) + gi * BN * 2, src,
                              (uint32_t)ncols * 2, mb, pol_w);
                }
            }
        };
        auto issue_x = [&](uint32_t slot, const UnitPos &p, uint64_t *bar) {
            const StreamOperands &op = tab.e[p.e];
            const int k0 = p.ks * SK;
            const int klen = a.K - k0 < SK ? a.K - k0 : SK;
            for (int m = lane; m < a.M; m += 32)
                bulk_load(slot + a.x_off + m * a.x_pitch, op.x + (size_t)m * a.K + k0,
                          (uint32_t)klen * 2, smem_u32(bar), pol_x);
        };

        const UnitPos p0 = unit_pos(ub, a.T, a.KS);
        // weights, scales and zeros do not depend on the previous kernel:
        // request the first ring's worth before waiting for it
        UnitPos p = p0;
        for (int i = 0; i < first; ++i) {
            if (lane == 0) mbar_arrive_expect_tx(&full[i], stage_bytes(p));
            __syncwarp();
            if (i != skip) issue_weights(ring + i * a.stage_bytes, p, &full[i]);
            advance(p, a.T, a.KS);
        }
        pdl_wait();   // x may be the previous kernel's output
        p = p0;
        for (int i = 0; i < first; ++i) {
            if (i != skip) issue_x(ring + i * a.stage_bytes, p, &full[i]);
            advance(p, a.T, a.KS);
        }
        int slot = first < a.stages ? first : 0;
        int round = first < a.stages ? 0 : 1;
        for (int i = first; i < n_units; ++i) {
            if (!mbar_wait_bounded(&empty[slot], (round - 1) & 1, a.timeout_ns))
                report_status(a.status, W4A16_ERR_TIMEOUT);
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], stage_bytes(p));
            __syncwarp();
            if (i != skip) {
                const uint32_t sl = ring + slot * a.stage_bytes;
                issue_weights(sl, p, &full[slot]);
                issue_x(sl, p, &full[slot]);
            }
            advance(p, a.T, a.KS);
            if (++slot == a.stages) {
                slot = 0;
                ++round;
            }
        }
        // no copy of this CTA may still be landing when it exits (normally the
        // consumers have long seen every stage complete; after a timed-out
        // wait this bounds the rest)
        for (int i = n_units - first; i < n_units; ++i) {
            if (i == skip) continue;
            if (!mbar_wait_bounded(&full[i % a.stages], (i / a.stages) & 1, a.timeout_ns))
                report_status(a.status, W4A16_ERR_TIMEOUT);
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    // Under programmatic dependent launch this CTA may start while the
    // previous kernel still runs: the consumers sleep in griddepcontrol.wait
    // (no stage can complete before its x arrives, which follows that wait)
    // instead of spinning on the stage barriers.
    pdl_wait();
    const int g = lane >> 2, t = lane & 3;
    const int wn = warp % BNS, wk = warp / BNS;
    const int tid = threadIdx.x;                        // < 32 * kCW here
    const int j0 = wk * kSPW;                           // this warp's first 32-k step of a stage
    const int x0_row = g < a.M ? g : 0;                 // rows past M read row 0
    const int x1_row = g + 8 < a.M ? g + 8 : 0;         // (their MMA columns are dropped)
    const int gshift = 31 - __clz(a.group);             // the group is a power of two
    const uint32_t ring = smem_u32(smem);
    // Byte offsets, inside a slot, of this thread's operands of step 0; step u
    // adds a compile-time stride, so the stage loop does no address arithmetic
    // beyond the slot base.
    constexpr uint32_t kWStep = PERM || TMAW ? 512u : 4u * WP;  // packed words, per step
    // first of the thread's four columns in the tile
    const int cl = 32 * wn + 4 * (TMAW ? perm8(g) : g);
    uint32_t w_off, w_off_odd = 0, sz_off[kSPW];
    if (TMAW) {
        // strip wn at wn * RS * 128; row r at r * 128 with its 16-byte chunks
        // swizzled by r % 8 = 4 (u % 2) + t for step u
        const uint32_t row0 = (uint32_t)(wn * RS * 128 + (4 * j0 + t) * 128);
        w_off = row0 + (uint32_t)((perm8(g) ^ t) << 4);
        w_off_odd = row0 + (uint32_t)((perm8(g) ^ (4 + t)) << 4);
#pragma unroll
        for (int u = 0; u < kSPW; ++u) {
            const int gi = ((j0 + u) << 5) >> gshift;
            sz_off[u] = (uint32_t)(a.sz_off + (gi * BN + cl) * 2);
        }
    } else if (PERM) {
        const uint32_t blk = (uint32_t)((wn * R + (j0 >> 3)) * a.blk_bytes);
        w_off = blk + (uint32_t)((((j0 & 7) << 5) + lane) << 4);
#pragma unroll
        for (int u = 0; u < kSPW; ++u) {
            const int gi = a.group < 256 ? (((j0 & 7) + u) << 5) >> gshift : 0;
            sz_off[u] = blk + kPermBlockWordBytes + (uint32_t)((gi * 8 + g) << 4);
        }
    } else {
        w_off = (uint32_t)((4 * j0 + t) * WP + ((32 * wn + 4 * g) << 2));
#pragma unroll
        for (int u = 0; u < kSPW; ++u) {
            const int gi = ((j0 + u) << 5) >> gshift;
            sz_off[u] = (uint32_t)(a.sz_off + (gi * BN + 32 * wn + 4 * g) * 2);
        }
    }
    const uint32_t z_rows = (uint32_t)a.z_delta;             // natural: zero rows after scale rows
    const uint32_t x0_off = (uint32_t)(a.x_off + x0_row * a.x_pitch + ((4 * j0 + t) << 4));
    const uint32_t x1_off = (uint32_t)(a.x_off + x1_row * a.x_pitch + ((4 * j0 + t) << 4));

    float acc[NT][2][4];
#pragma unroll
    for (int p = 0; p < NT; ++p)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[p][j][r] = 0.f;

    UnitPos p = unit_pos(ub, a.T, a.KS);
    long long seg_begin = ub;                           // first unit of the current tile segment
    int slot = 0;
    uint32_t phase = 0;
    for (int i = 0; i < n_units; ++i) {
        if (!mbar_wait_bounded(&full[slot], phase, a.timeout_ns))
            report_status(a.status, W4A16_ERR_TIMEOUT);
        const uint32_t base = ring + slot * a.stage_bytes;
        const int kleft = a.K - p.ks * SK;
        const int steps_here = (kleft < SK ? kleft : SK) >> 5;   // valid 32-k steps of the stage
        auto load_sz = [&](int u, uint2 &sr, uint2 &zr) {
            if (PERM) {
                const uint4 v = lds128(base + sz_off[u]);
                sr = make_uint2(v.x, v.y);
                zr = make_uint2(v.z, v.w);
            } else {
                sr = lds64(base + sz_off[u]);
                zr = lds64(base + sz_off[u] + z_rows);
            }
        };
        auto fragments = [&](const uint4 (&xq)[NT], uint32_t (&bx)[NT][4]) {
#pragma unroll
            for (int q = 0; q < NT; ++q) {
                if (PERM) {
                    // repacked nibble order: x pairs (k0,k1), (k2,k3), (k4,k5),
                    // (k6,k7) feed the MMA as they sit in memory
                    bx[q][0] = xq[q].x;
                    bx[q][1] = xq[q].y;
                    bx[q][2] = xq[q].z;
                    bx[q][3] = xq[q].w;
                } else {
                    x_fragments(xq[q], bx[q]);
                }
            }
        };
        auto release = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (++slot == a.stages) {
                slot = 0;
                phase ^= 1;
            }
        };
        // group partials: M <= 8 keeps the two k halves apart (four
        // independent MMA chains per step); M > 8 joins them (its two batch
        // tiles already give four chains) to stay within the registers.  The
        // first step of a group starts from zero in the MMA itself.
        constexpr int KH = NT == 1 ? 2 : 1;
        float gs[NT][2][KH][4];
        GroupConsts k;
        if constexpr (NT == 1 && kZeroFree) {
            uint4 wv[kSPW], xv[kSPW];
            uint2 sraw[OG ? 1 : kSPW], zraw[OG ? 1 : kSPW];
#pragma unroll
            for (int u = 0; u < kSPW; ++u) {
                wv[u] = lds128(base + ((TMAW && (u & 1)) ? w_off_odd : w_off) + u * kWStep);
                xv[u] = lds128(base + x0_off + u * 64);
                if (!OG || u == 0) load_sz(u, sraw[OG ? 0 : u], zraw[OG ? 0 : u]);
            }
            release();
            ZfConsts zk = make_zf_consts(zraw[0], sraw[0]);
            float dlo[2][4], dhi[2][4], dx[4];
#pragma unroll
            for (int u = 0; u < kSPW; ++u) {
                if (j0 + u < steps_here) {                    // warp-uniform
                    if (!OG && u > 0) zk = make_zf_consts(zraw[u], sraw[u]);
                    uint32_t blo[2], bhi[2];
                    if (PERM) {
                        // repacked: nibbles (0,4) / (2,6) hold k (0,1) / (4,5);
                        // (1,5) / (3,7) hold k (2,3) / (6,7)
                        blo[0] = xv[u].x;
                        blo[1] = xv[u].z;
                        bhi[0] = xv[u].y;
                        bhi[1] = xv[u].w;
                    } else {
                        // natural: nibble p holds k = p
                        blo[0] = __byte_perm(xv[u].x, xv[u].z, 0x5410);   // (x0, x4)
                        blo[1] = __byte_perm(xv[u].y, xv[u].w, 0x5410);   // (x2, x6)
                        bhi[0] = __byte_perm(xv[u].x, xv[u].z, 0x7632);   // (x1, x5)
                        bhi[1] = __byte_perm(xv[u].y, xv[u].w, 0x7632);   // (x3, x7)
                    }
                    if (!OG || u == 0)
                        zf_step<true>(dlo, dhi, dx, wv[u], blo, bhi);
                    else
                        zf_step<false>(dlo, dhi, dx, wv[u], blo, bhi);
                    if (!OG)
                        zf_flush(reinterpret_cast<float (&)[1][2][4]>(acc), dlo, dhi, dx, zk);
                }
            }
            if (OG && steps_here > j0)
                zf_flush(reinterpret_cast<float (&)[1][2][4]>(acc), dlo, dhi, dx, zk);
        } else if constexpr (NT == 1) {
            // all of the warp's operands of the stage first, then the slot is
            // released and the steps' MMAs overlap
            uint4 wv[kSPW], xv[kSPW][1];
            uint2 sraw[OG ? 1 : kSPW], zraw[OG ? 1 : kSPW];
#pragma unroll
            for (int u = 0; u < kSPW; ++u) {
                wv[u] = lds128(base + ((TMAW && (u & 1)) ? w_off_odd : w_off) + u * kWStep);
                xv[u][0] = lds128(base + x0_off + u * 64);
                if (!OG || u == 0) load_sz(u, sraw[OG ? 0 : u], zraw[OG ? 0 : u]);
            }
            release();
            k = make_group_consts(zraw[0], sraw[0]);
#pragma unroll
            for (int u = 0; u < kSPW; ++u) {
                if (j0 + u < steps_here) {                    // warp-uniform
                    if (!OG && u > 0) k = make_group_consts(zraw[u], sraw[u]);
                    uint32_t bx[NT][4];
                    fragments(xv[u], bx);
                    if (!OG || u == 0)
                        step_first(gs, wv[u], k, bx);
                    else
                        step(gs, wv[u], k, bx);
                    if (!OG) flush(acc, gs, k);
                }
            }
        } else {
            // two batch tiles: twice the x registers, so each step loads its
            // operands just before its MMAs and the slot is released after the
            // stage
#pragma unroll
            for (int u = 0; u < kSPW; ++u) {
                if (j0 + u < steps_here) {                    // warp-uniform
                    if (!OG || u == 0) {
                        uint2 sr, zr;
                        load_sz(u, sr, zr);
                        k = make_group_consts(zr, sr);
                    }
                    const uint4 w =
                        lds128(base + ((TMAW && (u & 1)) ? w_off_odd : w_off) + u * kWStep);
                    uint4 xq[NT];
                    xq[0] = lds128(base + x0_off + u * 64);
                    xq[NT - 1] = lds128(base + x1_off + u * 64);
                    uint32_t bx[NT][4];
                    fragments(xq, bx);
                    if (!OG || u == 0)
                        step_first(gs, w, k, bx);
                    else
                        step(gs, w, k, bx);
                    if (!OG) flush(acc, gs, k);
                }
            }
            release();
        }
        if (!(NT == 1 && kZeroFree) && OG && steps_here > j0) flush(acc, gs, k);

        // ------------------------------------------------ end of a tile segment
        const long long u_glob = ub + i;
        const bool seg_end = (i + 1 == n_units) || (p.ks + 1 == a.KS);
        if (seg_end) {
            const int tg = p.e * a.T + p.tile;            // tile index over all experts
            const long long t_first = (long long)tg * a.KS, t_last = t_first + a.KS - 1;
            const bool whole = seg_begin == t_first && u_glob == t_last;
            const int col0 = p.tile * BN;
            const int E = a.M * BN;
            uint16_t *out = tab.e[p.e].out;
            // the consumer warps' partials, summed in warp order
#pragma unroll
            for (int q = 0; q < NT; ++q)
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int m = 8 * q + 2 * t + (r & 1);
                        const int c = cl + 2 * j + (r >> 1);
                        if (m < a.M) red[(wk * a.M + m) * BN + c] = acc[q][j][r];
                        acc[q][j][r] = 0.f;
                    }
            named_bar_sync(1, 32 * kCW);
            const int sel = (tg == (int)(ub / a.KS)) ? 0 : 1;   // this CTA's partial slot
            float *mine = whole ? nullptr : a.scratch + (size_t)(2 * cta + sel) * E;
            for (int e = tid; e < E; e += 32 * kCW) {
                const int m = e / BN, c = e - m * BN;
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < WK; ++w) v += red[(w * a.M + m) * BN + c];
                if (whole) {
                    if (col0 + c < a.N)
                        out[(size_t)m * a.N + col0 + c] = __half_as_ushort(__float2half_rn(v));
                } else {
                    mine[e] = v;
                }
            }
            if (!whole) __threadfence();                  // publish the partial
            named_bar_sync(1, 32 * kCW);
            if (!whole) {
                // shared tile: count the arrival; the last CTA to arrive adds
                // every partial in CTA order and writes the tile
                const int c_lo = cta_of(t_first, G, a.U), c_hi = cta_of(t_last, G, a.U);
                if (tid == 0) {
                    __threadfence();
                    const int before = atomicAdd(&a.counters[tg], 1);
                    *last_flag = before == c_hi - c_lo;
                }
                named_bar_sync(1, 32 * kCW);
                if (*last_flag) {
                    __threadfence();
                    for (int e = tid; e < E; e += 32 * kCW) {
                        const int m = e / BN, c = e - m * BN;
                        float v = 0.f;
                        for (int cc = c_lo; cc <= c_hi; ++cc) {
                            const int s2 = (tg == (int)(range_begin(cc, G, a) / a.KS)) ? 0 : 1;
                            v += __ldcg(a.scratch + (size_t)(2 * cc + s2) * E + e);
                        }
                        if (col0 + c < a.N)
                            out[(size_t)m * a.N + col0 + c] = __half_as_ushort(__float2half_rn(v));
                    }
                    if (tid == 0) a.counters[tg] = 0;     // ready for the next call
                }
            }
            seg_begin = u_glob + 1;
        }
        advance(p, a.T, a.KS);
    }
}

// ------------------------------------------------------------------- host side
// Scratch for shared tiles, one per (device, stream): calls on one stream run
// in order, so they may reuse it; calls on different streams get their own.
struct ScratchEntry {
    int dev;
    cudaStream_t stream;
    float *partials;
    int *counters;
};
constexpr int kScratchEntries = 32;
constexpr size_t kScratchFloats = (size_t)2 * kMaxGrid * 16 * 128;   // [2 G][M <= 16][BN <= 128]
constexpr int kScratchCounters = 1 << 16;                            // tiles over all experts

// Returns false when no scratch can be had (the caller then plans whole
// tiles per CTA, which needs none).  The first call on a stream allocates;
// the allocation is done outside any stream capture of this thread, and the
// counters are cleared on a private stream, so a first call made while the
// stream is being captured does not disturb the capture.
bool scratch_for(cudaStream_t stream, float **partials, int **counters) {
    static std::mutex mu;
    static ScratchEntry table[kScratchEntries];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (table[i].dev == dev && table[i].stream == stream) {
            *partials = table[i].partials;
            *counters = table[i].counters;
            return true;
        }
    if (used == kScratchEntries) return false;
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    float *p = nullptr;
    int *c = nullptr;
    cudaStream_t side = nullptr;
    bool ok = cudaMalloc(&p, kScratchFloats * sizeof(float)) == cudaSuccess &&
              cudaMalloc(&c, kScratchCounters * sizeof(int)) == cudaSuccess &&
              cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking) == cudaSuccess &&
              cudaMemsetAsync(c, 0, kScratchCounters * sizeof(int), side) == cudaSuccess &&
              cudaStreamSynchronize(side) == cudaSuccess;
    if (side) cudaStreamDestroy(side);
    if (!ok) {
        if (p) cudaFree(p);
        if (c) cudaFree(c);
        cudaGetLastError();
    }
    cudaThreadExchangeStreamCaptureMode(&mode);
    if (!ok) return false;
    table[used++] = ScratchEntry{dev, stream, p, c};
    *partials = p;
    *counters = c;
    return true;
}


int round_up(int v, int m) { return (v + m - 1) / m * m; }

// Shared-memory layout of one launch.
struct StreamLayout {
    int stage_bytes, w_pitch, sz_off, sz_rows, z_delta, x_off, x_pitch, blk_bytes, stages,
        red_off, bar_off, smem_bytes;
};

// Packed rows and k per stage for a tile of bns strips (the kernel's RS, SK).
constexpr int stage_rows(int bns) { return 4 * kSPW * (kCW / bns); }

bool stream_layout(int M, int group, int bns, int lay, StreamLayout &L) {
    const int BN = 32 * bns;
    const int RS = stage_rows(bns), SK = 8 * RS;
    L.w_pitch = BN * 4 + 32;
    L.sz_rows = SK / group > 1 ? SK / group : 1;
    // a TMA box lands on a 128-byte boundary: the zero rows start on one
    L.z_delta = round_up(L.sz_rows * BN * 2, 128);
    L.blk_bytes = 4096 + 128 * (group < 256 ? 256 / group : 1);
    int w_area;
    if (lay == kPerm) {
        w_area = bns * (RS / 32) * L.blk_bytes;
        L.sz_off = 0;
    } else {
        L.sz_off = lay == kTma ? bns * RS * 128 : RS * L.w_pitch;
        w_area = L.sz_off + 2 * L.z_delta;
    }
    L.x_pitch = SK * 2 + 64;
    L.x_off = round_up(w_area, 128);
    // slots on 1024-byte boundaries (the span of the 128-byte swizzle)
    L.stage_bytes = round_up(L.x_off + M * L.x_pitch, lay == kTma ? 1024 : 128);
    const int red_bytes = (kCW / bns) * M * BN * 4;
    const int fixed = 1024 + red_bytes + 2 * kMaxStages * 8 + 16 + 128;
    int ns = (kBudget - fixed) / L.stage_bytes;
    if (ns > kMaxStages) ns = kMaxStages;
    if (ns < 2) return false;
    L.stages = ns;
    L.red_off = ns * L.stage_bytes;
    L.bar_off = round_up(L.red_off + red_bytes, 16);
    L.smem_bytes = 1024 + L.bar_off + 2 * ns * 8 + 16;   // + alignment slack of the base
    return true;
}

template <int NT, int BNS, int LAY, bool OG, int MAXE>
cudaError_t launch_stream_kernel(const StreamArgs &sa, const StreamTable<MAXE> &tab,
                                 const CUtensorMap *maps, int grid, int smem, bool pdl,
                                 cudaStream_t stream) {
    auto kern = decode_stream_kernel<NT, BNS, LAY, OG, MAXE>;
    cudaError_t e = ensure_dynamic_smem((const void *)kern, kBudget);
    if (e != cudaSuccess) return e;
    // the whole unified L1/shared array as shared memory, so that a CTA of the
    // next call fits beside one of this call on every SM
    static bool carveout_set = false;
    if (!carveout_set) {
        e = cudaFuncSetAttribute((const void *)kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        carveout_set = true;
    }
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grid, 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = &attr;
    lc.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&lc, kern, sa, tab, maps[0], maps[1], maps[2]);
}

template <int NT, int BNS, int LAY, int MAXE>
cudaError_t dispatch_og(bool og, const StreamArgs &sa, const StreamTable<MAXE> &tab,
                        const CUtensorMap *maps, int grid, int smem, bool pdl,
                        cudaStream_t stream) {
    return og ? launch_stream_kernel<NT, BNS, LAY, true, MAXE>(sa, tab, maps, grid, smem, pdl,
                                                               stream)
              : launch_stream_kernel<NT, BNS, LAY, false, MAXE>(sa, tab, maps, grid, smem, pdl,
                                                                stream);
}

template <int LAY, int MAXE>
cudaError_t dispatch_shape(int nt, int bns, bool og, const StreamArgs &sa,
                           const StreamTable<MAXE> &tab, const CUtensorMap *maps, int grid,
                           int smem, bool pdl, cudaStream_t stream) {
#define W4A16_STREAM(NT_, BNS_) \
    dispatch_og<NT_, BNS_, LAY, MAXE>(og, sa, tab, maps, grid, smem, pdl, stream)
    if (nt == 1) return bns == 1 ? W4A16_STREAM(1, 1) : (bns == 2 ? W4A16_STREAM(1, 2) : W4A16_STREAM(1, 4));
    return bns == 1 ? W4A16_STREAM(2, 1) : (bns == 2 ? W4A16_STREAM(2, 2) : W4A16_STREAM(2, 4));
#undef W4A16_STREAM
}

// The layout a call uses: repacked weights, or natural weights through TMA
// boxes (one GEMM, N % 32 == 0) or through per-row bulk copies.
int layout_for_call(bool permuted, int E, int N) {
    if (permuted) return kPerm;
    return E == 1 && N % 32 == 0 ? kTma : kRows;
}

}  // namespace

int decode_stream_stage_k(int bns) { return 8 * stage_rows(bns); }

// ---------------------------------------------------------------- no-alloc
// Scratch of w4a16_gemm_noalloc: one fixed array in device memory that every
// GPU loading this library holds until the process exits.  Its first
// kNoAllocCounterBytes hold the per-tile arrival counters, the rest the fp32
// partials of shared tiles.  In host code the name below is only a stand-in
// for the array; its device address comes from cudaGetSymbolAddress.
constexpr size_t kNoAllocBytes = (size_t)4 << 20;            // 4 MiB in all
constexpr size_t kNoAllocCounterBytes = (size_t)64 << 10;    // 16384 tiles
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// The array's device address on the current device, looked up once per device.
static bool noalloc_scratch(unsigned char **ptr) {
    static std::mutex mu;
    static unsigned char *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return false;
        }
        addr[dev] = static_cast<unsigned char *>(p);
    }
    *ptr = addr[dev];
    return true;
}

NoAllocResult launch_decode_stream_noalloc(const StreamCall &call, int bns, bool pdl,
                                           cudaStream_t stream) {
    const int M = call.M, N = call.N, K = call.K, group = call.group;
    if (call.E != 1 || call.permuted || !decode_stream_supported(M, N, K, group, bns, false))
        return NoAllocResult{cudaErrorNotSupported, 0, 0};
    // per-row copies of the natural layout: no tensor map to encode
    StreamLayout L;
    if (!stream_layout(M, group, bns, kRows, L)) return NoAllocResult{cudaErrorNotSupported, 0, 0};
    const int BN = 32 * bns, SK = 8 * stage_rows(bns);
    StreamArgs sa = {};
    sa.M = M;
    sa.N = N;
    sa.K = K;
    sa.group = group;
    sa.T = (N + BN - 1) / BN;
    sa.KS = (K + SK - 1) / SK;
    const long long units = (long long)sa.T * sa.KS;
    int grid = device_info().sm_count;
    if (grid > kMaxGrid) grid = kMaxGrid;
    if (grid > units) grid = (int)units;
    // what the call needs: one counter per tile, two fp32 partial tiles per CTA
    const size_t need_counters = (size_t)sa.T * sizeof(int);
    const size_t need_partials = (size_t)2 * grid * M * BN * sizeof(float);
    if (units > (1ll << 30) || need_counters > kNoAllocCounterBytes ||
        need_partials > kNoAllocBytes - kNoAllocCounterBytes)
        return NoAllocResult{cudaErrorInvalidValue, need_counters, need_partials};
    unsigned char *base = nullptr;
    if (!noalloc_scratch(&base)) return NoAllocResult{cudaErrorInvalidSymbol, 0, 0};
    sa.U = (int)units;
    sa.align = 0;                                  // stream-K shares: the scratch is used
    sa.counters = reinterpret_cast<int *>(base);
    sa.scratch = reinterpret_cast<float *>(base + kNoAllocCounterBytes);
    // the counters must read zero when the kernel starts; the array keeps
    // whatever the previous call (on any stream) left there
    cudaError_t e = cudaMemsetAsync(sa.counters, 0, need_counters, stream);
    if (e != cudaSuccess) return NoAllocResult{e, 0, 0};
    sa.stages = L.stages;
    sa.stage_bytes = L.stage_bytes;
    sa.w_pitch = L.w_pitch;
    sa.sz_off = L.sz_off;
    sa.sz_rows = L.sz_rows;
    sa.z_delta = L.z_delta;
    sa.x_off = L.x_off;
    sa.x_pitch = L.x_pitch;
    sa.blk_bytes = L.blk_bytes;
    sa.red_off = L.red_off;
    sa.bar_off = L.bar_off;
    sa.status = device_status_word();
    if (!sa.status) return NoAllocResult{cudaErrorInvalidDevice, 0, 0};
    sa.timeout_ns = 1000000000ull;
    const bool og = group >= 32 * kSPW;
    const int nt = M > 8 ? 2 : 1;
    CUtensorMap maps[3];
    memset(maps, 0, sizeof maps);
    StreamTable<1> tab;
    tab.e[0] = StreamOperands{call.x[0], call.w[0], call.s[0], call.z[0], call.out[0]};
    e = dispatch_shape<kRows, 1>(nt, bns, og, sa, tab, maps, grid, L.smem_bytes, pdl, stream);
    return NoAllocResult{e, need_counters, need_partials};
}

bool decode_stream_supported(int M, int N, int K, int group, int bns, bool perm) {
    const bool g_ok = group == 32 || group == 64 || group == 128 || group == 256 ||
                      group == 512 || group == 1024;
    if (!(g_ok && M >= 1 && M <= 16 && (bns == 1 || bns == 2 || bns == 4) && N % 8 == 0 && K > 0))
        return false;
    if (perm && (K % 256 != 0 || N % 32 != 0)) return false;
    StreamLayout L;
    // the per-row layout is the largest of the two natural ones
    return stream_layout(M, group, bns, perm ? kPerm : kRows, L) &&
           (perm || stream_layout(M, group, bns, kTma, L));
}

// cfg: warps_n = 32-column strips per tile (1, 2 or 4), split_k = 1 for whole
// tiles per CTA or 2 for stream-K shares, ctas = grid size (0: one per SM).
cudaError_t launch_decode_stream(const StreamCall &call, const w4a16_config &cfg,
                                 cudaStream_t stream) {
    const int M = call.M, N = call.N, K = call.K, group = call.group;
    const int bns = cfg.warps_n;
    if (call.E < 1 || call.E > kMaxExperts ||
        !decode_stream_supported(M, N, K, group, bns, call.permuted))
        return cudaErrorNotSupported;
    const int lay = layout_for_call(call.permuted, call.E, N);
    StreamLayout L;
    if (!stream_layout(M, group, bns, lay, L)) return cudaErrorNotSupported;
    const int BN = 32 * bns, RS = stage_rows(bns), SK = 8 * RS;
    StreamArgs sa = {};
    sa.M = M;
    sa.N = N;
    sa.K = K;
    sa.group = group;
    sa.T = (N + BN - 1) / BN;
    sa.KS = (K + SK - 1) / SK;
    const long long units = (long long)call.E * sa.T * sa.KS;
    if (units > (1ll << 30) || (long long)call.E * sa.T > kScratchCounters)
        return cudaErrorNotSupported;
    sa.U = (int)units;
    const int tiles = call.E * sa.T;
    int grid = cfg.ctas > 0 ? cfg.ctas : device_info().sm_count;
    if (grid > kMaxGrid) grid = kMaxGrid;
    sa.align = cfg.split_k == 1 ? 1 : 0;
    if (sa.align) {
        if (grid > tiles) grid = tiles;
    } else {
        if (grid > sa.U) grid = sa.U;
        if (!scratch_for(stream, &sa.scratch, &sa.counters)) {
            // no scratch on this stream: whole tiles per CTA
            sa.align = 1;
            if (grid > tiles) grid = tiles;
        }
    }
    sa.stages = L.stages;
    sa.stage_bytes = L.stage_bytes;
    sa.w_pitch = L.w_pitch;
    sa.sz_off = L.sz_off;
    sa.sz_rows = L.sz_rows;
    sa.z_delta = L.z_delta;
    sa.x_off = L.x_off;
    sa.x_pitch = L.x_pitch;
    sa.blk_bytes = L.blk_bytes;
    sa.red_off = L.red_off;
    sa.bar_off = L.bar_off;
    sa.status = device_status_word();
    if (!sa.status) return cudaErrorInvalidDevice;
    const bool test_timeout = (cfg.flags & W4A16_FLAG_TEST_TIMEOUT) != 0;
    sa.timeout_ns = test_timeout ? 5000000ull : 1000000000ull;
    sa.test_skip_last = test_timeout ? 1 : 0;
    const bool pdl = (cfg.flags & W4A16_FLAG_PDL) != 0;
    const bool og = group >= 32 * kSPW;
    const int nt = M > 8 ? 2 : 1;
    CUtensorMap maps[3];
    memset(maps, 0, sizeof maps);
    if (lay == kTma) {
        // packed [K/8, N] as {32 columns, K/8 rows, N/32 strips}: one box of
        // RS rows x bns strips per stage, 128-byte swizzled; scales and zeros
        // [K/g, N] in boxes of BN columns x sz_rows group rows
        const uint64_t w_dims[3] = {32, (uint64_t)(K / 8), (uint64_t)(N / 32)};
        const uint64_t w_strides[2] = {(uint64_t)N * 4, 128};
        const uint32_t w_box[3] = {32, (uint32_t)RS, (uint32_t)bns};
        if (!make_tmap(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, call.w[0], w_dims, w_strides,
                       w_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_tmap_2d(&maps[1], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, call.s[0], N, K / group,
                          (uint64_t)N * 2, BN, L.sz_rows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_tmap_2d(&maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, call.z[0], N, K / group,
                          (uint64_t)N * 2, BN, L.sz_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    if (call.E == 1) {
        StreamTable<1> tab;
        tab.e[0] = StreamOperands{call.x[0], call.w[0], call.s[0], call.z[0], call.out[0]};
        if (lay == kPerm)
            return dispatch_shape<kPerm, 1>(nt, bns, og, sa, tab, maps, grid, L.smem_bytes, pdl,
                                            stream);
        if (lay == kTma)
            return dispatch_shape<kTma, 1>(nt, bns, og, sa, tab, maps, grid, L.smem_bytes, pdl,
                                           stream);
        return dispatch_shape<kRows, 1>(nt, bns, og, sa, tab, maps, grid, L.smem_bytes, pdl,
                                        stream);
    }
    StreamTable<kMaxExperts> tab;
    for (int e = 0; e < kMaxExperts; ++e)
        tab.e[e] = e < call.E ? StreamOperands{call.x[e], call.w[e], call.s[e], call.z[e],
                                               call.out[e]}
                              : StreamOperands{};
    return lay == kPerm ? dispatch_shape<kPerm, kMaxExperts>(nt, bns, og, sa, tab, maps, grid,
                                                             L.smem_bytes, pdl, stream)
                        : dispatch_shape<kRows, kMaxExperts>(nt, bns, og, sa, tab, maps, grid,
                                                             L.smem_bytes, pdl, stream);
}

}  // namespace w4a16
