// decode_warp.cu -- the decode-regime W4A16 GEMM for the smallest batches
// (M <= 4) with every warp its own weight stream.
//
// What it computes: out[m,n] = sum_k x[m,k] * (q[k,n] - z[g(k),n]) * s[g(k),n],
// fp32 accumulation, fp16 result (page "Beating FP16 with 4-bit Weights: A
// Portable W4A16 GEMM in Triton", sections "The design" and "Things I got
// wrong along the way"; page "Triton Kernel Matches bitsandbytes: Why Both Lose
// to Math", sections "Roofline First" and "Why Marlin Is Still Faster").  The
// per-step arithmetic is decode_math.cuh's zero-free step: the codes enter the
// MMA as exact fp16 subnormals and the zero is removed once per group through
// the x sums, with one fp32 scale per group.
//
// How the work and the bytes move:
//   * Units.  A unit is 32 columns x 512 k of the natural layout: one 8 KB TMA
//     box of packed words (64 rows of 128 bytes, 128-byte swizzled), the
//     unit's scale and zero rows, and the unit's slice of x -- five copies for
//     ~9 KB, so the copy engine is never the limit.
//   * Each CTA owns whole column tiles (a contiguous run of them); the units of
//     its tiles, tile by tile, are cut into one contiguous run per warp.
//   * No warp waits for another while streaming.  Each warp owns a ring of D
//     shared-memory slots with one mbarrier each: its lane 0 issues a unit's
//     copies and, once the warp has computed a unit, refills that slot with the
//     unit D ahead.  There is no producer warp and no CTA-wide barrier in the
//     stream: a slow warp delays only itself.
//   * A tile split between warps is summed in shared memory: each warp stores
//     its fp32 partial and counts its arrival, and the last warp to arrive adds
//     the partials in warp order (a fixed order: bitwise reproducible) and
//     writes the outputs.  A warp whose run holds a whole tile writes it.
//   * With programmatic dependent launch the weights of the first D units are
//     requested before the wait for the previous kernel; x and out are touched
//     only after it.  Every mbarrier wait is bounded in wall time and a wait
//     that gives up records W4A16_ERR_TIMEOUT.
#include <mutex>
#include <string.h>

#include "common.cuh"
#include "decode_math.cuh"
#include "sm100_ptx.cuh"
#include "tmap.cuh"

namespace w4a16 {
namespace {

constexpr int kUnitK = 512;                 // k per unit
constexpr int kUnitRows = kUnitK / 8;       // packed rows per unit
constexpr int kUnitWBytes = kUnitRows * 128;
constexpr int kSteps = kUnitK / 32;         // 32-k MMA steps per unit
constexpr int kHalfK = 256;                 // x arrives as two 256-k boxes
constexpr int kW = 8;                       // warps per CTA
constexpr int kBudget = 220 * 1024;         // shared memory per CTA (one CTA per SM)
constexpr int kMaxDepth = 4;
constexpr int kMaxM = 4;
constexpr int kMaxTilesPerCta = 64;

struct WarpArgs {
    uint16_t *out;
    int *status;
    int M, N, K, group;
    int T, KC;               // column tiles, units per tile
    int G;                   // CTAs
    int D;                   // ring slots per warp
    int aux_bytes;           // per slot: scale rows, zero rows, x
    int s_off, z_off, x_off; // inside the aux part of a slot
    int sr;                  // scale (zero) rows per unit
    int w_area, aux_area, part_off, cnt_off, bar_off;
    uint32_t tx_bytes;
    unsigned long long timeout_ns;
};

__device__ __forceinline__ int perm8w(int g) { return (g >> 1) + ((g & 1) << 2); }

// SG: 32-k steps per scale group inside a unit (16 when a group spans the unit).
template <int SG>
__global__ void __launch_bounds__(32 * kW, 1)
decode_warp_kernel(const __grid_constant__ WarpArgs a, const __grid_constant__ CUtensorMap tm_w,
                   const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_z,
                   const __grid_constant__ CUtensorMap tm_x)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    int *cnt = reinterpret_cast<int *>(smem + a.cnt_off);
    float *part = reinterpret_cast<float *>(smem + a.part_off);   // [kW][2][kMaxM][32]

    pdl_launch_dependents();
    // this CTA's tiles [tc0, tc1) and the runs of its warps (local unit
    // numbers: unit u is chunk u % KC of tile tc0 + u / KC); runs of q + 1
    // units for the first r warps, q for the others, none for warps >= weff
    const int tc0 = (int)((long long)a.T * blockIdx.x / a.G);
    const int tc1 = (int)((long long)a.T * (blockIdx.x + 1) / a.G);
    const int ucta = (tc1 - tc0) * a.KC;
    const int weff = ucta < kW ? ucta : kW;
    const int q = ucta / weff, r = ucta - q * weff;
    auto begin_of = [&](int w) { return w * q + (w < r ? w : r); };
    auto warp_of = [&](int u) {
        const int lim = r * (q + 1);
        return u < lim ? u / (q + 1) : r + (u - lim) / q;
    };
    if (threadIdx.x < kMaxTilesPerCta) cnt[threadIdx.x] = 0;
    __syncthreads();   // counters are zero before any warp counts
    if (warp >= weff) return;

    const int ub = begin_of(warp), ue = begin_of(warp + 1), n = ue - ub;
    uint8_t *wring = smem + warp * a.D * kUnitWBytes;
    uint8_t *aring = smem + a.w_area + warp * a.D * a.aux_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.bar_off) + warp * a.D;
    if (lane == 0) {
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_s);
        prefetch_tmap(&tm_z);
        prefetch_tmap(&tm_x);
        for (int i = 0; i < a.D; ++i) mbar_init(&full[i], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const uint64_t pol_w = l2_evict_first_policy();
    const uint64_t pol_x = l2_evict_last_policy();
    // lane 0: the copies of the unit at (tile it, chunk ik) into slot sl --
    // weights, scales and zeros -- with the barrier armed for the whole unit,
    // x included; x follows separately (it may be the previous kernel's output)
    auto issue_w = [&](int sl, int it, int ik) {
        mbar_arrive_expect_tx(&full[sl], a.tx_bytes);
        uint8_t *ab = aring + sl * a.aux_bytes;
        tma_load_2d(wring + sl * kUnitWBytes, &tm_w, &full[sl], it * 32, ik * kUnitRows, pol_w);
        const int grow = (int)((long long)ik * kUnitK / a.group);
        tma_load_2d(ab + a.s_off, &tm_s, &full[sl], it * 32, grow, pol_w);
        tma_load_2d(ab + a.z_off, &tm_z, &full[sl], it * 32, grow, pol_w);
    };
    auto issue_x = [&](int sl, int ik) {
        uint8_t *xb = aring + sl * a.aux_bytes + a.x_off;
        tma_load_2d(xb, &tm_x, &full[sl], ik * kUnitK, 0, pol_x);
        tma_load_2d(xb + a.M * kHalfK * 2, &tm_x, &full[sl], ik * kUnitK + kHalfK, 0, pol_x);
    };
    int tl = ub / a.KC, kc = ub - (ub / a.KC) * a.KC;   // the unit being computed (local tile)
    int itl = tl, ikc = kc;                              // the next unit to request
    const int first = n < a.D ? n : a.D;
    for (int i = 0; i < first; ++i) {
        if (lane == 0) issue_w(i, tc0 + itl, ikc);
        if (++ikc == a.KC) { ikc = 0; ++itl; }
    }
    pdl_wait();   // x and out may belong to the previous kernel
    if (lane == 0) {
        int xk = kc;
        for (int i = 0; i < first; ++i) {
            issue_x(i, xk);
            if (++xk == a.KC) xk = 0;
        }
    }

    // this thread's four columns of a tile, and its x row
    const int cl = 4 * perm8w(g);
    const bool x_ok = g < a.M;
    const uint32_t x_row = (uint32_t)(a.x_off + (x_ok ? g : 0) * (kHalfK * 2) + t * 16);
    const uint32_t x_half = (uint32_t)(a.M * kHalfK * 2);

    float acc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;

    const int first_tl = tl;
    int slot = 0;
    uint32_t phase = 0;
    for (int i = 0; i < n; ++i) {
        if (!mbar_wait_bounded(&full[slot], phase, a.timeout_ns))
            report_status(a.status, W4A16_ERR_TIMEOUT);
        const uint32_t wb = smem_u32(wring) + slot * kUnitWBytes;
        const uint32_t ab = smem_u32(aring) + slot * a.aux_bytes;
        float dlo[2][4], dhi[2][4], dx[4];
        ZfConsts zk;
#pragma unroll
        for (int sc = 0; sc < kSteps / 4; ++sc) {
            // operands of four steps
            uint4 wv[4], xv[4];
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
                const int u = 4 * sc + s4;                 // step in the unit
                const int rr = 4 * u + t;                  // packed row in the unit
                wv[s4] = lds128(wb + rr * 128 + ((perm8w(g) ^ (rr & 7)) << 4));
                const uint4 v = lds128(ab + x_row + (u >> 3) * x_half + (u & 7) * 64);
                xv[s4] = x_ok ? v : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
                const int u = 4 * sc + s4;
                if (u % SG == 0) {
                    const int gq = u / SG;                  // scale row of this group
                    const uint2 sr = lds64(ab + a.s_off + (gq * 32 + cl) * 2);
                    const uint2 zr = lds64(ab + a.z_off + (gq * 32 + cl) * 2);
                    zk = make_zf_consts(zr, sr);
                }
                uint32_t blo[2], bhi[2];
                blo[0] = __byte_perm(xv[s4].x, xv[s4].z, 0x5410);   // (x0, x4)
                blo[1] = __byte_perm(xv[s4].y, xv[s4].w, 0x5410);   // (x2, x6)
                bhi[0] = __byte_perm(xv[s4].x, xv[s4].z, 0x7632);   // (x1, x5)
                bhi[1] = __byte_perm(xv[s4].y, xv[s4].w, 0x7632);   // (x3, x7)
                if (u % SG == 0)
                    zf_step<true>(dlo, dhi, dx, wv[s4], blo, bhi);
                else
                    zf_step<false>(dlo, dhi, dx, wv[s4], blo, bhi);
                if (u % SG == SG - 1)
                    zf_flush(reinterpret_cast<float (&)[1][2][4]>(acc), dlo, dhi, dx, zk);
            }
        }
        // every read of the slot is done: refill it with the unit D ahead
        // (the warp's reads are ordered before the copies that overwrite them)
        if (i + a.D < n) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                issue_w(slot, tc0 + itl, ikc);
                issue_x(slot, ikc);
            }
            if (++ikc == a.KC) { ikc = 0; ++itl; }
        }
        if (++slot == a.D) {
            slot = 0;
            phase ^= 1;
        }

        // ------------------------------------------------ end of a tile segment
        if (++kc == a.KC || i + 1 == n) {
            const int t_first = tl * a.KC, t_last = t_first + a.KC - 1;   // local units
            const int col0 = (tc0 + tl) * 32;
            if (t_first >= ub && t_last < ue) {
                // the whole tile is this warp's: write it
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int m = 2 * t + (e & 1);
                        const int c = col0 + cl + 2 * j + (e >> 1);
                        if (m < a.M && c < a.N)
                            a.out[(size_t)m * a.N + c] = __half_as_ushort(__float2half_rn(acc[j][e]));
                    }
            } else {
                // a tile split between warps: store this warp's partial, count
                // the arrival; the last warp adds the partials in warp order
                float *mine = part + (warp * 2 + (tl == first_tl ? 0 : 1)) * kMaxM * 32;
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int m = 2 * t + (e & 1);
                        if (m < kMaxM) mine[m * 32 + cl + 2 * j + (e >> 1)] = acc[j][e];
                    }
                __syncwarp();
                const int w_lo = warp_of(t_first), w_hi = warp_of(t_last);
                int last = 0;
                if (lane == 0) {
                    __threadfence_block();
                    last = atomicAdd(&cnt[tl], 1) == w_hi - w_lo;
                    __threadfence_block();
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    float v[kMaxM];
#pragma unroll
                    for (int m = 0; m < kMaxM; ++m) v[m] = 0.f;
                    for (int w = w_lo; w <= w_hi; ++w) {
                        const int sel = begin_of(w) / a.KC == tl ? 0 : 1;
                        const float *src = part + (w * 2 + sel) * kMaxM * 32 + lane;
#pragma unroll
                        for (int m = 0; m < kMaxM; ++m) v[m] += src[m * 32];
                    }
                    if (col0 + lane < a.N)
#pragma unroll
                        for (int m = 0; m < kMaxM; ++m)
                            if (m < a.M)
                                a.out[(size_t)m * a.N + col0 + lane] = __half_as_ushort(__float2half_rn(v[m]));
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
            ++tl;
            kc = 0;
        }
    }
}

int round_up(int v, int m) { return (v + m - 1) / m * m; }

// Shared-memory layout of a launch; false when two slots per warp do not fit.
bool warp_layout(int M, int group, WarpArgs &a, int &smem) {
    const int sr = group < kUnitK ? kUnitK / group : 1;     // scale rows per unit
    a.sr = sr;
    a.s_off = 0;
    a.z_off = round_up(sr * 64, 128);
    a.x_off = 2 * a.z_off;
    a.aux_bytes = round_up(a.x_off + M * kUnitK * 2, 128);
    a.tx_bytes = (uint32_t)(kUnitWBytes + 2 * sr * 64 + M * kUnitK * 2);
    const int per_slot = kUnitWBytes + a.aux_bytes;
    const int fixed = 1024 + kW * 2 * kMaxM * 32 * 4 + kMaxTilesPerCta * 4 + kW * kMaxDepth * 8 + 64;
    int d = (kBudget - fixed) / (kW * per_slot);
    if (d > kMaxDepth) d = kMaxDepth;
    if (d < 2) return false;
    a.D = d;
    a.w_area = kW * d * kUnitWBytes;
    a.aux_area = kW * d * a.aux_bytes;
    a.part_off = a.w_area + a.aux_area;
    a.cnt_off = a.part_off + kW * 2 * kMaxM * 32 * 4;
    a.bar_off = round_up(a.cnt_off + kMaxTilesPerCta * 4, 16);
    smem = 1024 + a.bar_off + kW * d * 8;
    return smem <= kBudget;
}

template <int SG>
cudaError_t launch_warp_kernel(const WarpArgs &a, const CUtensorMap *maps, int smem, bool pdl,
                               cudaStream_t stream) {
    auto kern = decode_warp_kernel<SG>;
    cudaError_t e = ensure_dynamic_smem((const void *)kern, kBudget);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(a.G, 1, 1);
    lc.blockDim = dim3(32 * kW, 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = &attr;
    lc.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&lc, kern, a, maps[0], maps[1], maps[2], maps[3]);
}

int grid_for(int T, int ctas) {
    int G = ctas > 0 ? ctas : device_info().sm_count;
    return G < T ? G : T;
}

}  // namespace

bool decode_warp_supported(int M, int N, int K, int group, int ctas) {
    const bool g_ok = group == 32 || group == 64 || group == 128 || group == 256 ||
                      group == 512 || group == 1024;
    if (!(g_ok && M >= 1 && M <= kMaxM && N % 8 == 0 && K > 0 && K % 8 == 0)) return false;
    const int T = (N + 31) / 32;
    const int G = grid_for(T, ctas);
    if (G < 1 || (T + G - 1) / G > kMaxTilesPerCta) return false;
    WarpArgs a;
    int smem = 0;
    return warp_layout(M, group, a, smem);
}

cudaError_t launch_decode_warp(const GemmArgs &g, const w4a16_config &cfg, cudaStream_t stream) {
    if (!decode_warp_supported(g.M, g.N, g.K, g.group, cfg.ctas)) return cudaErrorNotSupported;
    WarpArgs a = {};
    int smem = 0;
    if (!warp_layout(g.M, g.group, a, smem)) return cudaErrorNotSupported;
    a.out = g.out;
    a.M = g.M;
    a.N = g.N;
    a.K = g.K;
    a.group = g.group;
    a.T = (g.N + 31) / 32;
    a.KC = (g.K + kUnitK - 1) / kUnitK;
    a.G = grid_for(a.T, cfg.ctas);
    a.status = device_status_word();
    if (!a.status) return cudaErrorInvalidDevice;
    a.timeout_ns = 1000000000ull;
    CUtensorMap maps[4];
    if (!make_tmap_2d(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT32, g.packed, g.N, g.K / 8,
                      (uint64_t)g.N * 4, 32, kUnitRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&maps[1], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, g.scales, g.N, g.K / g.group,
                      (uint64_t)g.N * 2, 32, a.sr, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, g.zeros, g.N, g.K / g.group,
                      (uint64_t)g.N * 2, 32, a.sr, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&maps[3], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, g.x, g.K, g.M,
                      (uint64_t)g.K * 2, kHalfK, g.M, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const bool pdl = (cfg.flags & W4A16_FLAG_PDL) != 0;
    const int sg = g.group >= kUnitK ? kSteps : g.group / 32;
    switch (sg) {
    case 1: return launch_warp_kernel<1>(a, maps, smem, pdl, stream);
    case 2: return launch_warp_kernel<2>(a, maps, smem, pdl, stream);
    case 4: return launch_warp_kernel<4>(a, maps, smem, pdl, stream);
    case 8: return launch_warp_kernel<8>(a, maps, smem, pdl, stream);
    default: return launch_warp_kernel<16>(a, maps, smem, pdl, stream);
    }
}


// ------------------------------------------------------------ repacked weights
// The same warp-stream design on the pre-permuted layout (quant.cu's repack):
// a unit is UB consecutive repacked blocks of one strip -- a block is 32
// columns x 256 k, 1024 words in lane order, then its scales and zeros; the
// blocks of a strip are contiguous -- fetched with ONE 1-D bulk copy (no
// tensor map), and x's rows of the unit by one bulk copy each.  The last unit
// of a strip may hold fewer blocks.  Each
// lane's 128-bit read of a step is its MMA fragment, and x enters the MMA as
// it sits in memory.  Up to kMaxExperts GEMMs of one shape per launch: the
// units of all experts' tiles are split between the CTAs as above.
namespace {

constexpr int kPermW = 8;                   // warps per CTA
constexpr int kPermMaxM = 8;                // rows of x: the MMA's 8 batch columns
constexpr int kPermK = 256;                 // k per repacked block
constexpr int kPermSteps = kPermK / 32;
constexpr int kPermWordBytes = 4096;        // the block's packed words

struct PermArgs {
    int *status;
    int M, N, K, group, E;
    int T;                   // 32-column strips per expert
    int KB;                  // 256-k blocks per strip
    int UB, U;               // blocks per unit, units per strip (ceil(KB / UB))
    int blk_bytes;           // 4096 + 128 * groups per block
    int G, D;                // CTAs, ring slots per warp
    int slot_bytes, x_off;   // per slot: UB blocks, then M rows of UB * 256 k of x
    int part_off, cnt_off, bar_off;
    unsigned long long timeout_ns;
};

struct PermTable {
    const uint16_t *x[kMaxExperts];
    const uint8_t *w[kMaxExperts];
    uint16_t *out[kMaxExperts];
};

// SG: 32-k steps per scale group inside a block (8 when a group spans it);
// MAXM: 4 or 8, the rows of x the partial sums are laid out for (M <= MAXM).
template <int SG, int MAXM>
__global__ void __launch_bounds__(32 * kPermW, 1)
decode_warp_perm_kernel(const __grid_constant__ PermArgs a, const __grid_constant__ PermTable tab)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    int *cnt = reinterpret_cast<int *>(smem + a.cnt_off);
    float *part = reinterpret_cast<float *>(smem + a.part_off);   // [kPermW][2][MAXM][32]

    pdl_launch_dependents();
    // this CTA's tiles (over all experts: tile = expert * T + strip) and the
    // runs of its warps, as in decode_warp_kernel
    const int TT = a.E * a.T;
    const int tc0 = (int)((long long)TT * blockIdx.x / a.G);
    const int tc1 = (int)((long long)TT * (blockIdx.x + 1) / a.G);
    const int ucta = (tc1 - tc0) * a.U;
    const int weff = ucta < kPermW ? ucta : kPermW;
    const int q = ucta / weff, r = ucta - q * weff;
    auto begin_of = [&](int w) { return w * q + (w < r ? w : r); };
    auto warp_of = [&](int u) {
        const int lim = r * (q + 1);
        return u < lim ? u / (q + 1) : r + (u - lim) / q;
    };
    if (threadIdx.x < kMaxTilesPerCta) cnt[threadIdx.x] = 0;
    __syncthreads();   // counters are zero before any warp counts
    if (warp >= weff) return;

    const int ub = begin_of(warp), ue = begin_of(warp + 1), n = ue - ub;
    uint8_t *ring = smem + warp * a.D * a.slot_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.bar_off) + warp * a.D;
    if (lane == 0) {
        for (int i = 0; i < a.D; ++i) mbar_init(&full[i], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const uint64_t pol_w = l2_evict_first_policy();
    const uint64_t pol_x = l2_evict_last_policy();
    const int xrow = a.UB * kPermK * 2;   // bytes per row of x in a slot
    auto blocks_of = [&](int iu) {
        const int b = a.KB - iu * a.UB;
        return b < a.UB ? b : a.UB;
    };
    // lane 0: the blocks of (tile it, unit iu) into slot sl, with the barrier
    // armed for the whole unit, x included; x follows separately
    auto issue_w = [&](int sl, int it, int iu) {
        const int e = it / a.T, sn = it - e * a.T, nb = blocks_of(iu);
        mbar_arrive_expect_tx(&full[sl], (uint32_t)(nb * (a.blk_bytes + a.M * kPermK * 2)));
        bulk_load(smem_u32(ring + sl * a.slot_bytes),
                  tab.w[e] + ((size_t)sn * a.KB + (size_t)iu * a.UB) * a.blk_bytes,
                  (uint32_t)(nb * a.blk_bytes), smem_u32(&full[sl]), pol_w);
    };
    auto issue_x = [&](int sl, int it, int iu) {
        const int e = it / a.T, nb = blocks_of(iu);
        for (int m = 0; m < a.M; ++m)
            bulk_load(smem_u32(ring + sl * a.slot_bytes + a.x_off + m * xrow),
                      tab.x[e] + (size_t)m * a.K + (size_t)iu * a.UB * kPermK,
                      (uint32_t)(nb * kPermK * 2), smem_u32(&full[sl]), pol_x);
    };
    int tl = ub / a.U, kc = ub - (ub / a.U) * a.U;   // the unit being computed (local tile)
    int itl = tl, ikc = kc;                              // the next unit to request
    const int first = n < a.D ? n : a.D;
    for (int i = 0; i < first; ++i) {
        if (lane == 0) issue_w(i, tc0 + itl, ikc);
        if (++ikc == a.U) { ikc = 0; ++itl; }
    }
    pdl_wait();   // x and out may belong to the previous kernel
    if (lane == 0) {
        int xt = tl, xk = kc;
        for (int i = 0; i < first; ++i) {
            issue_x(i, tc0 + xt, xk);
            if (++xk == a.U) { xk = 0; ++xt; }
        }
    }

    const bool x_ok = g < a.M;
    const uint32_t x_row = (uint32_t)(a.x_off + (x_ok ? g : 0) * xrow + t * 16);

    float acc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;

    const int first_tl = tl;
    int slot = 0;
    uint32_t phase = 0;
    for (int i = 0; i < n; ++i) {
        if (!mbar_wait_bounded(&full[slot], phase, a.timeout_ns))
            report_status(a.status, W4A16_ERR_TIMEOUT);
        const uint32_t s0 = smem_u32(ring) + slot * a.slot_bytes;
        const int nb = blocks_of(kc);
        for (int b = 0; b < nb; ++b) {
            const uint32_t sb = s0 + b * a.blk_bytes;        // the block
            const uint32_t xb = s0 + x_row + b * (kPermK * 2);   // its x, this thread's row
            float dlo[2][4], dhi[2][4], dx[4];
            ZfConsts zk;
#pragma unroll
            for (int sc = 0; sc < kPermSteps / 4; ++sc) {
                uint4 wv[4], xv[4];
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    const int u = 4 * sc + s4;
                    wv[s4] = lds128(sb + u * 512 + lane * 16);     // the lane's fragment
                    const uint4 v = lds128(xb + u * 64);
                    xv[s4] = x_ok ? v : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    const int u = 4 * sc + s4;
                    if (u % SG == 0) {
                        // four scales then four zeros of the thread's columns
                        const uint4 v = lds128(sb + kPermWordBytes + ((u / SG) * 8 + g) * 16);
                        zk = make_zf_consts(make_uint2(v.z, v.w), make_uint2(v.x, v.y));
                    }
                    // repacked nibble order: nibbles (0,4) / (2,6) hold k (0,1) /
                    // (4,5), nibbles (1,5) / (3,7) hold k (2,3) / (6,7)
                    const uint32_t blo[2] = {xv[s4].x, xv[s4].z};
                    const uint32_t bhi[2] = {xv[s4].y, xv[s4].w};
                    if (u % SG == 0)
                        zf_step<true>(dlo, dhi, dx, wv[s4], blo, bhi);
                    else
                        zf_step<false>(dlo, dhi, dx, wv[s4], blo, bhi);
                    if (u % SG == SG - 1)
                        zf_flush(reinterpret_cast<float (&)[1][2][4]>(acc), dlo, dhi, dx, zk);
                }
            }
        }
        // every read of the slot is done: refill it with the unit D ahead
        if (i + a.D < n) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                issue_w(slot, tc0 + itl, ikc);
                issue_x(slot, tc0 + itl, ikc);
            }
            if (++ikc == a.U) { ikc = 0; ++itl; }
        }
        if (++slot == a.D) {
            slot = 0;
            phase ^= 1;
        }

        // ------------------------------------------------ end of a tile segment
        if (++kc == a.U || i + 1 == n) {
            const int t_first = tl * a.U, t_last = t_first + a.U - 1;   // local units
            const int tg = tc0 + tl, e = tg / a.T, col0 = (tg - e * a.T) * 32;
            uint16_t *out = tab.out[e];
            if (t_first >= ub && t_last < ue) {
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int k2 = 0; k2 < 4; ++k2) {
                        const int m = 2 * t + (k2 & 1);
                        const int c = col0 + 4 * g + 2 * j + (k2 >> 1);
                        if (m < a.M)
                            out[(size_t)m * a.N + c] = __half_as_ushort(__float2half_rn(acc[j][k2]));
                    }
            } else {
                float *mine = part + (warp * 2 + (tl == first_tl ? 0 : 1)) * MAXM * 32;
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int k2 = 0; k2 < 4; ++k2) {
                        const int m = 2 * t + (k2 & 1);
                        if (m < MAXM) mine[m * 32 + 4 * g + 2 * j + (k2 >> 1)] = acc[j][k2];
                    }
                __syncwarp();
                const int w_lo = warp_of(t_first), w_hi = warp_of(t_last);
                int last = 0;
                if (lane == 0) {
                    __threadfence_block();
                    last = atomicAdd(&cnt[tl], 1) == w_hi - w_lo;
                    __threadfence_block();
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    // rows M..MAXM-1 hold zeros (their x rows are zero)
                    float v[MAXM];
#pragma unroll
                    for (int m = 0; m < MAXM; ++m) v[m] = 0.f;
                    for (int w = w_lo; w <= w_hi; ++w) {
                        const int sel = begin_of(w) / a.U == tl ? 0 : 1;
                        const float *src = part + (w * 2 + sel) * MAXM * 32 + lane;
#pragma unroll
                        for (int m = 0; m < MAXM; ++m) v[m] += src[m * 32];
                    }
#pragma unroll
                    for (int m = 0; m < MAXM; ++m)
                        if (m < a.M)
                            out[(size_t)m * a.N + col0 + lane] = __half_as_ushort(__float2half_rn(v[m]));
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) acc[j][k2] = 0.f;
            ++tl;
            kc = 0;
        }
    }
}

int perm_max_m(int M) { return M <= 4 ? 4 : kPermMaxM; }

bool perm_layout(int M, int group, int ub, PermArgs &a, int &smem) {
    const int w = kPermW, maxm = perm_max_m(M);
    const int gps = group < kPermK ? kPermK / group : 1;
    a.UB = ub;
    a.blk_bytes = kPermWordBytes + 128 * gps;
    a.x_off = round_up(ub * a.blk_bytes, 128);
    a.slot_bytes = round_up(a.x_off + M * ub * kPermK * 2, 128);
    const int fixed = 128 + w * 2 * maxm * 32 * 4 + kMaxTilesPerCta * 4 + w * kMaxDepth * 8 + 64;
    int d = (kBudget - fixed) / (w * a.slot_bytes);
    if (d > kMaxDepth) d = kMaxDepth;
    if (d < 2) return false;
    a.D = d;
    a.part_off = w * d * a.slot_bytes;
    a.cnt_off = a.part_off + w * 2 * maxm * 32 * 4;
    a.bar_off = round_up(a.cnt_off + kMaxTilesPerCta * 4, 16);
    smem = 128 + a.bar_off + w * d * 8;
    return smem <= kBudget;
}

// Units of two blocks where two ring slots per warp fit (M <= 4 at group 128),
// else single blocks.  (Six warps with units of two blocks at M = 5..8 were
// measured: faster on some shapes, slower on others, the same on average.)
bool perm_shape(int M, int group, PermArgs &a, int &smem) {
    return perm_layout(M, group, 2, a, smem) || perm_layout(M, group, 1, a, smem);
}

template <int SG>
cudaError_t launch_perm_kernel(const PermArgs &a, const PermTable &tab, int smem, bool pdl,
                               cudaStream_t stream) {
    auto kern = perm_max_m(a.M) == 4 ? decode_warp_perm_kernel<SG, 4>
                                     : decode_warp_perm_kernel<SG, kPermMaxM>;
    cudaError_t e = ensure_dynamic_smem((const void *)kern, kBudget);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(a.G, 1, 1);
    lc.blockDim = dim3(32 * kPermW, 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = &attr;
    lc.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&lc, kern, a, tab);
}

}  // namespace

bool decode_warp_perm_supported(int M, int N, int K, int group, int experts, int ctas) {
    if (!(M >= 1 && M <= kPermMaxM && experts >= 1 && experts <= kMaxExperts &&
          repack_supported(K, N, group)))
        return false;
    const long long TT = (long long)experts * (N / 32);
    const int G = grid_for((int)(TT < 0x7fffffff ? TT : 0x7fffffff), ctas);
    if (G < 1 || (TT + G - 1) / G > kMaxTilesPerCta) return false;
    PermArgs a;
    int smem = 0;
    return perm_shape(M, group, a, smem);
}

cudaError_t launch_decode_warp_perm(const StreamCall &call, const w4a16_config &cfg,
                                    cudaStream_t stream) {
    if (!decode_warp_perm_supported(call.M, call.N, call.K, call.group, call.E, cfg.ctas))
        return cudaErrorNotSupported;
    PermArgs a = {};
    int smem = 0;
    if (!perm_shape(call.M, call.group, a, smem)) return cudaErrorNotSupported;
    a.M = call.M;
    a.N = call.N;
    a.K = call.K;
    a.group = call.group;
    a.E = call.E;
    a.T = call.N / 32;
    a.KB = call.K / kPermK;
    a.U = (a.KB + a.UB - 1) / a.UB;
    a.G = grid_for(a.E * a.T, cfg.ctas);
    a.status = device_status_word();
    if (!a.status) return cudaErrorInvalidDevice;
    a.timeout_ns = 1000000000ull;
    PermTable tab = {};
    for (int e = 0; e < call.E; ++e) {
        tab.x[e] = call.x[e];
        tab.w[e] = reinterpret_cast<const uint8_t *>(call.w[e]);
        tab.out[e] = call.out[e];
    }
    const bool pdl = (cfg.flags & W4A16_FLAG_PDL) != 0;
    const int sg = call.group >= kPermK ? kPermSteps : call.group / 32;
    switch (sg) {
    case 1: return launch_perm_kernel<1>(a, tab, smem, pdl, stream);
    case 2: return launch_perm_kernel<2>(a, tab, smem, pdl, stream);
    case 4: return launch_perm_kernel<4>(a, tab, smem, pdl, stream);
    default: return launch_perm_kernel<8>(a, tab, smem, pdl, stream);
    }
}

}  // namespace w4a16
