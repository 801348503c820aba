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
//   * 4, 8 or 16 consumer warps split a stage: 32-column strips x 32-k steps.
//   * split-K across the CTAs of one thread-block cluster, reduced in a fixed
//     order through distributed shared memory (no atomics, no workspace).
//   * the CTA uses under half of an SM (at most about 108 KB of shared memory;
//     a third of one with 4 consumer warps), and signals programmatic
//     dependent launch at its start, so the next GEMM on the stream can start
//     streaming its weights while this one finishes.  Only x and out wait for
//     the previous kernel (griddepcontrol).
//   * every mbarrier wait is bounded in wall time; a wait that gives up records
//     W4A16_ERR_TIMEOUT in the device status word and the kernel runs to its
//     end without touching memory it does not own.
#include <mutex>

#include "common.cuh"
#include "decode_math.cuh"
#include "sm100_ptx.cuh"
#include "tmap.cuh"

namespace w4a16 {

namespace {

constexpr bool kTmaZeroFree = true;   // M <= 8: decode_math.cuh's zero-free step

constexpr int kStageRows = 32;                 // packed rows per stage
constexpr int kStageK = 8 * kStageRows;        // 256 k per stage
// ring + slots per CTA: about half an SM with 8 or 16 consumer warps, about a
// third with 4 (three small CTAs per SM: two of one GEMM and one of the next)
constexpr int smem_budget(int cw) { return cw == 4 ? 72 * 1024 : 108 * 1024; }
constexpr int kSmemMax = 220 * 1024;           // opt-in limit set on the kernels

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
    int slots_off;            // cluster reduction slots [split][Mc][BN] (leader only)
    unsigned long long timeout_ns;
    int test_skip_last;       // test hook: arm but never load the CTA's last stage
    int w3d;                  // weights through one 3-D box per stage (N % 32 == 0)
};

// consumer lane group g reads 16-byte chunk perm8(g) of its 128-byte row
__device__ __forceinline__ int perm8(int g) { return (g >> 1) + ((g & 1) << 2); }

// ONE_GROUP: a warp's share of a stage (8*BNS*... k rows) lies inside one
// quantization group (group >= 32 * steps per warp), so the group constants
// are formed once per stage and the step loop has no branches.
// BF: x, scales, zeros and out are bfloat16; every weight is dequantized with
// its scale (one bf16 multiply) and the MMAs accumulate straight into running
// sums (decode_math.cuh, bfloat16 section).
template <int NT, int BNS, int CW, bool ONE_GROUP, bool BF>
__global__ void __launch_bounds__(32 * (CW + 1), CW == 4 ? 3 : (CW == 8 ? 2 : 1))
decode_tma_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
                  const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_x,
                  const TmaDecodeArgs a)
{
    constexpr int kConsumerWarps = CW;
    constexpr int kThreads = 32 * (CW + 1);
    constexpr int BN = 32 * BNS;                 // columns per CTA
    constexpr int WK = kConsumerWarps / BNS;     // consumer warps along a stage's 8 steps
    constexpr int SPW = 8 / WK;                  // steps per warp per stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int MB = 8 * NT;                    // batch rows a thread's fragments cover
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + a.slots_off +
                                                  (a.split + WK) * MB * BN * 4);
    uint64_t *empty = full + a.stages;
    uint64_t *cl_done = empty + a.stages;          // leader: the other CTAs' partials landed
    float *slots = reinterpret_cast<float *>(ring + a.slots_off);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == kConsumerWarps * 32) {
        // the descriptors live in parameter memory: start fetching them first
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_s);
        prefetch_tmap(&tm_z);
        prefetch_tmap(&tm_x);
    }
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
        mbar_init(cl_done, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // the leader expects the other CTAs' partials as bulk-copy bytes
    if (a.split > 1 && threadIdx.x == 0 && cluster_ctarank() == 0)
        mbar_arrive_expect_tx(cl_done, (uint32_t)((a.split - 1) * Mc * BN * 4));
    // first half of a split cluster barrier: every CTA's barriers exist before
    // any CTA signals another (the wait comes just before the reduction)
    if (a.split > 1) cluster_arrive();

    float acc[NT][2][4];
    float accb[NT][2][2][4];   // bfloat16 only: running sums of the two k halves
#pragma unroll
    for (int p = 0; p < NT; ++p)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[p][j][r] = accb[p][j][0][r] = accb[p][j][1][r] = 0.f;

    const int g = lane >> 2, t = lane & 3;
    const int wn = warp % BNS, wk = warp / BNS;
    const int cl = 32 * wn + 4 * perm8(g);     // first of the thread's 4 columns in the tile

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
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
                if (a.w3d)
                    tma_load_3d(slot, &tm_w, &full[st], 0, row, col_base >> 5, pol_stream);
                else
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
            // steady state: the ring position and the group row advance
            // incrementally (groups divide the 256-k stage), so the loop trip
            // is a wait and four copy issues
            const int gstep = kStageK / a.group;
            int slot = first < a.stages ? first : 0, round = first < a.stages ? 0 : 1;
            int row = cta_row0 + first * kStageRows;
            int grow = row * 8 / a.group;
            for (int st = first; st < n_st; ++st) {
                if (!mbar_wait_bounded(&empty[slot], (round - 1) & 1, a.timeout_ns))
                    report_status(a.status, W4A16_ERR_TIMEOUT);
                uint8_t *sl = ring + slot * a.stage_bytes;
                mbar_arrive_expect_tx(&full[slot], a.tx_bytes);
                if (st != skip) {
                    if (a.w3d)
                        tma_load_3d(sl, &tm_w, &full[slot], 0, row, col_base >> 5, pol_stream);
                    else
#pragma unroll
                        for (int s = 0; s < BNS; ++s)
                            tma_load_2d(sl + s * 4096, &tm_w, &full[slot], col_base + 32 * s, row,
                                        pol_stream);
                    tma_load_2d(sl + a.s_off, &tm_s, &full[slot], col_base, grow, pol_stream);
                    tma_load_2d(sl + a.z_off, &tm_z, &full[slot], col_base, grow, pol_stream);
                    tma_load_2d(sl + a.x_off, &tm_x, &full[slot], row * 8, m_base, pol_keep);
                }
                row += kStageRows;
                grow += gstep;
                if (++slot == a.stages) { slot = 0; ++round; }
            }
            // no copy of this CTA may still be landing when it exits (normally
            // the consumers have long seen every stage complete; after a
            // timed-out wait this bounds the rest)
            for (int st = max(0, n_st - a.stages); st < n_st; ++st) {
                if (st == skip) continue;
                if (!mbar_wait_bounded(&full[st % a.stages], (st / a.stages) & 1, a.timeout_ns))
                    report_status(a.status, W4A16_ERR_TIMEOUT);
            }
        }
    } else {
        // ------------------------------------------------------ consumers
        // Under programmatic dependent launch this CTA may start while the
        // previous kernel still runs: the consumers sleep in griddepcontrol.wait
        // (no stage can complete before x is loaded after it anyway) instead of
        // spinning on the stage barriers and stealing issue slots from the
        // previous kernel's warps on the same SM.
        pdl_wait();
        const int x0_row = g < Mc ? g : 0;         // rows past M read row 0, then zeroed
        const int x1_row = g + 8 < Mc ? g + 8 : 0;
        const bool x0_ok = g < Mc, x1_ok = g + 8 < Mc;
        int slot = 0;
        uint32_t phase = 0;
        for (int st = 0; st < n_st; ++st) {
            if (!mbar_wait_bounded(&full[slot], phase, a.timeout_ns))
                report_status(a.status, W4A16_ERR_TIMEOUT);
            const uint32_t base = smem_u32(ring) + slot * a.stage_bytes;
            const uint32_t wtile = base + wn * 4096;
            const int r0 = wk * 4 * SPW;                // first row of this warp in the stage
            // all of this warp's operands of the stage first (then the slot is
            // released): the steps below are independent and their MMAs overlap
            uint4 wv[SPW], xv[NT][SPW];
            uint2 sraw[ONE_GROUP ? 1 : SPW], zraw[ONE_GROUP ? 1 : SPW];
#pragma unroll
            for (int u = 0; u < (ONE_GROUP ? 1 : SPW); ++u) {
                const int gi = ((r0 + 4 * u) * 8) / a.group;       // group within the stage
                sraw[u] = lds64(base + a.s_off + (gi * BN + cl) * 2);
                zraw[u] = lds64(base + a.z_off + (gi * BN + cl) * 2);
            }
#pragma unroll
            for (int u = 0; u < SPW; ++u) {
                const int r = r0 + 4 * u + t;           // row within the stage
                wv[u] = lds128(wtile + r * 128 + ((perm8(g) ^ (r & 7)) << 4));
                const uint4 v0 = lds128(base + a.x_off + (x0_row * kStageK + 8 * r) * 2);
                xv[0][u] = x0_ok ? v0 : make_uint4(0, 0, 0, 0);
                if (NT > 1) {
                    const uint4 v1 = lds128(base + a.x_off + (x1_row * kStageK + 8 * r) * 2);
                    xv[NT - 1][u] = x1_ok ? v1 : make_uint4(0, 0, 0, 0);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);   // operands are in registers
            if (++slot == a.stages) { slot = 0; phase ^= 1; }
            if constexpr (BF) {
                GroupConstsBf kb = make_group_consts_bf(zraw[0], sraw[0]);
#pragma unroll
                for (int u = 0; u < SPW; ++u) {
                    if (!ONE_GROUP && u > 0) kb = make_group_consts_bf(zraw[u], sraw[u]);
                    uint32_t bx[NT][4];
#pragma unroll
                    for (int p = 0; p < NT; ++p) x_fragments(xv[p][u], bx[p]);
                    step_mma_bf16<NT>(accb, wv[u], kb, bx);
                }
            } else if constexpr (NT == 1 && kTmaZeroFree) {
                // M <= 8: the zero-free step (codes as fp16 subnormals, the
                // zero removed per group through the x sums)
                float dlo[2][4], dhi[2][4], dx[4];
                ZfConsts zk = make_zf_consts(zraw[0], sraw[0]);
#pragma unroll
                for (int u = 0; u < SPW; ++u) {
                    if (!ONE_GROUP && u > 0) zk = make_zf_consts(zraw[u], sraw[u]);
                    uint32_t blo[2], bhi[2];
                    blo[0] = __byte_perm(xv[0][u].x, xv[0][u].z, 0x5410);   // (x0, x4)
                    blo[1] = __byte_perm(xv[0][u].y, xv[0][u].w, 0x5410);   // (x2, x6)
                    bhi[0] = __byte_perm(xv[0][u].x, xv[0][u].z, 0x7632);   // (x1, x5)
                    bhi[1] = __byte_perm(xv[0][u].y, xv[0][u].w, 0x7632);   // (x3, x7)
                    if (!ONE_GROUP || u == 0)
                        zf_step<true>(dlo, dhi, dx, wv[u], blo, bhi);
                    else
                        zf_step<false>(dlo, dhi, dx, wv[u], blo, bhi);
                    if (!ONE_GROUP)
                        zf_flush(reinterpret_cast<float (&)[1][2][4]>(acc), dlo, dhi, dx, zk);
                }
                if (ONE_GROUP)
                    zf_flush(reinterpret_cast<float (&)[1][2][4]>(acc), dlo, dhi, dx, zk);
            } else {
            GroupConsts k = make_group_consts(zraw[0], sraw[0]);
            // one group per warp-stage: the warp's steps accumulate together
            // and the scale is applied once; otherwise once per step
            float gs[NT][2][2][4];
#pragma unroll
            for (int p = 0; p < NT; ++p)
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int r = 0; r < 4; ++r) gs[p][j][0][r] = gs[p][j][1][r] = 0.f;
#pragma unroll
            for (int u = 0; u < SPW; ++u) {
                if (!ONE_GROUP && u > 0) k = make_group_consts(zraw[u], sraw[u]);
                uint32_t bx[NT][4];
#pragma unroll
                for (int p = 0; p < NT; ++p) x_fragments(xv[p][u], bx[p]);
                step_mma_split<NT>(gs, wv[u], k, bx);
                if (!ONE_GROUP) flush_group_split<NT>(acc, gs, k);
            }
            if (ONE_GROUP) flush_group_split<NT>(acc, gs, k);
            }
        }
        if constexpr (BF) {
#pragma unroll
            for (int p = 0; p < NT; ++p)
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int r = 0; r < 4; ++r) acc[p][j][r] = accb[p][j][0][r] + accb[p][j][1][r];
        }
    }

    // ---------------------------------------------------------- epilogue
    // The consumer warps sum their fragment partials in shared memory (fixed
    // warp order) into this CTA's partial tile [Mc][BN].  With split-K, every
    // CTA but the cluster leader (rank 0) then ships its tile with one bulk
    // copy into its slot of the leader's shared memory -- the copy completes
    // bytes on the leader's barrier -- and exits once the copy has read its
    // source.  The leader sums the slots in rank order: the result does not
    // depend on timing, and there are no atomics and no global workspace.
    float *red = slots + a.split * MB * BN;           // [WK][MB][BN] warp partials
    const int rank = a.split > 1 ? (int)cluster_ctarank() : 0;
    const int E = Mc * BN;
    if (warp < kConsumerWarps) {
#pragma unroll
        for (int p = 0; p < NT; ++p)
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    red[(wk * MB + 8 * p + 2 * t + (r & 1)) * BN + cl + 2 * j + (r >> 1)] =
                        acc[p][j][r];
        named_bar_sync(1, kConsumerWarps * 32);
        float *mine = slots + rank * E;            // this CTA's partial (slot `rank`)
        for (int e = threadIdx.x; e < E; e += kConsumerWarps * 32) {
            const int m = e / BN, c = e - m * BN;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < WK; ++w) v += red[(w * MB + m) * BN + c];
            mine[e] = v;
        }
        if (a.split > 1 && rank != 0) {
            fence_proxy_async_smem();              // the bulk copy reads these writes
            named_bar_sync(1, kConsumerWarps * 32);
            if (threadIdx.x == 0) {
                cluster_wait();                    // the leader's barrier is initialized
                bulk_copy_to_cluster(map_to_rank(smem_u32(mine), 0), mine, (uint32_t)E * 4,
                                     map_to_rank(smem_u32(cl_done), 0));
                bulk_commit();
                bulk_wait_read();
            }
        }
    }
    if (rank != 0) {
        // the producer warp and the non-leader consumers only complete the
        // split cluster barrier (thread 0 already waited on it)
        if (threadIdx.x != 0) cluster_wait();
        return;
    }
    __syncthreads();                               // the leader's own partial is in slot 0
    if (a.split > 1) {
        cluster_wait();
        if (!mbar_wait_cluster_bounded(cl_done, 0, a.timeout_ns))
            report_status(a.status, W4A16_ERR_TIMEOUT);
    }
    pdl_wait();        // out may still be in use by the previous kernel
    for (int e = threadIdx.x; e < E; e += kThreads) {
        float v = 0.f;
        for (int q = 0; q < a.split; ++q) v += slots[q * E + e];
        const int m = e / BN, c = e - m * BN;
        const int col = col_base + c;
        if (col < a.N)
            a.out[(size_t)(m_base + m) * a.N + col] = to_out<BF>(v);
    }
}

int round_up(int v, int m) { return (v + m - 1) / m * m; }

struct Layout {
    int gps, s_off, z_off, x_off, stage_bytes, tx_bytes, stages, slots_off, smem_bytes;
};

// Shared memory: the ring of stages, then (split-K only) the leader's
// reduction slots, then the mbarriers.  The total stays near half an SM so two
// CTAs (of this GEMM and the next one on the stream) can be resident at once.
Layout layout_for(int group, int bns, int nt, int n_st, int split, int cw) {
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
    // [split][MB][BN] CTA partials, then [WK][MB][BN] warp partials (fp32)
    const int slots_bytes = (split + cw / bns) * mb * BN * 4;
    int ns = (smem_budget(cw) - slots_bytes) / L.stage_bytes;
    ns = ns < 2 ? 2 : (ns > 6 ? 6 : ns);
    if (n_st > 0 && ns > n_st) ns = n_st < 2 ? 2 : n_st;
    L.stages = ns;
    L.slots_off = ns * L.stage_bytes;
    L.smem_bytes = L.slots_off + slots_bytes + (2 * ns + 1) * 8 + 1024;
    return L;
}

template <int NT, int BNS, int CW, bool OG, bool BF>
cudaError_t launch_tma(const CUtensorMap &w, const CUtensorMap &s, const CUtensorMap &z,
                       const CUtensorMap &x, const TmaDecodeArgs &da, int tiles, int mchunks,
                       int smem, bool pdl, cudaStream_t stream) {
    const cudaError_t attr_err =
        ensure_dynamic_smem((const void *)decode_tma_kernel<NT, BNS, CW, OG, BF>, kSmemMax);
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(tiles, da.split, mchunks);
    lc.blockDim = dim3(32 * (CW + 1), 1, 1);
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
    return cudaLaunchKernelEx(&lc, decode_tma_kernel<NT, BNS, CW, OG, BF>, w, s, z, x, da);
}


}  // namespace


int consumer_warps(const w4a16_config &cfg) {
    return cfg.warps_k == 16 ? 16 : (cfg.warps_k == 4 ? 4 : 8);
}

int decode_tma_smem_bytes(const w4a16_config &cfg, int M, int group) {
    const int cw = consumer_warps(cfg);
    return layout_for(group, cfg.warps_n, M > 8 ? 2 : 1, cfg.steps, cfg.split_k, cw).smem_bytes;
}

bool decode_tma_supported(const w4a16_config &cfg, int group) {
    const bool g_ok = group == 32 || group == 64 || group == 128 || group == 256;
    return g_ok && (cfg.warps_n == 2 || cfg.warps_n == 4) &&
           (cfg.warps_k == 0 || cfg.warps_k == 4 || cfg.warps_k == 8 || cfg.warps_k == 16) &&
           cfg.split_k >= 1 &&
           cfg.split_k <= 8 && cfg.steps >= 1;
}

// cfg: warps_n = 32-column strips per CTA (2 or 4), split_k = CTAs per cluster
// along K, steps = 256-k stages per CTA.
cudaError_t launch_decode_tma(const GemmArgs &a, const w4a16_config &cfg, cudaStream_t stream) {
    if (!decode_tma_supported(cfg, a.group)) return cudaErrorNotSupported;
    const bool bf = cfg.dtype == W4A16_DTYPE_BF16;
    const int bns = cfg.warps_n;
    const int nt = a.M > 8 ? 2 : 1;
    const int KB = a.K / 8;
    const int rows_per_cta = cfg.steps * kStageRows;
    if ((long long)rows_per_cta * cfg.split_k < KB) return cudaErrorInvalidValue;
    const int cw = consumer_warps(cfg);           // consumer warps per CTA
    const Layout L = layout_for(a.group, bns, nt, cfg.steps, cfg.split_k, cw);
    if (L.smem_bytes > kSmemMax) return cudaErrorNotSupported;
    const int BN = 32 * bns;
    const int mb = 8 * nt;
    CUtensorMap tw, ts, tz, tx;
    // The weight tile of a stage is BNS strips of 32 columns x 32 packed rows
    // (128-byte swizzled, strip s at 4096 s).  With N % 32 == 0 the packed
    // array is also a 3-D tensor {32 columns, K/8 rows, N/32 strips} (strip
    // stride 128 bytes) and one box brings all BNS strips: the single
    // producer thread issues one weight copy per stage instead of BNS.
    const bool w3d = a.N % 32 == 0;
    const uint64_t w_dims[3] = {32, (uint64_t)KB, (uint64_t)(a.N / 32)};
    const uint64_t w_strides[2] = {(uint64_t)a.N * 4, 128};
    const uint32_t w_box[3] = {32, (uint32_t)kStageRows, (uint32_t)bns};
    const bool w_ok = w3d ? make_tmap(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, a.packed, w_dims,
                                      w_strides, w_box, CU_TENSOR_MAP_SWIZZLE_128B)
                          : make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.packed, a.N, KB,
                                         (uint64_t)a.N * 4, 32, kStageRows,
                                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (!w_ok ||
        !make_tmap_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.scales, a.N, a.K / a.group,
                      (uint64_t)a.N * 2, BN, L.gps, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.zeros, a.N, a.K / a.group,
                      (uint64_t)a.N * 2, BN, L.gps, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.x, a.K, a.M, (uint64_t)a.K * 2,
                      kStageK, mb, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    TmaDecodeArgs da;
    da.out = a.out;
    da.status = device_status_word();
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
    da.slots_off = L.slots_off;
    const bool test_timeout = (cfg.flags & W4A16_FLAG_TEST_TIMEOUT) != 0;
    da.timeout_ns = test_timeout ? 5000000ull : 1000000000ull;   // 5 ms in the test mode, else 1 s
    da.test_skip_last = test_timeout ? 1 : 0;
    da.w3d = w3d ? 1 : 0;
    const int tiles = (a.N + BN - 1) / BN;
    const int mchunks = (a.M + 15) / 16;
    if (mchunks > 65535) return cudaErrorInvalidValue;
    const bool pdl = (cfg.flags & W4A16_FLAG_PDL) != 0;
    // steps per warp per stage: 8 * bns / cw; one group per warp-stage if the
    // group spans at least that many 32-k steps
    const bool one_group = a.group >= 32 * (8 * bns / cw);
#define W4A16_TMA_LAUNCH1(NT_, BNS_, CW_, BF_)                                                   \
    (one_group ? launch_tma<NT_, BNS_, CW_, true, BF_>(tw, ts, tz, tx, da, tiles, mchunks,     \
                                                       L.smem_bytes, pdl, stream)              \
               : launch_tma<NT_, BNS_, CW_, false, BF_>(tw, ts, tz, tx, da, tiles, mchunks,    \
                                                        L.smem_bytes, pdl, stream))
#define W4A16_TMA_LAUNCH(NT_, BNS_, CW_) \
    (bf ? W4A16_TMA_LAUNCH1(NT_, BNS_, CW_, true) : W4A16_TMA_LAUNCH1(NT_, BNS_, CW_, false))
    if (cw == 8) {
        if (nt == 1) return bns == 4 ? W4A16_TMA_LAUNCH(1, 4, 8) : W4A16_TMA_LAUNCH(1, 2, 8);
        return bns == 4 ? W4A16_TMA_LAUNCH(2, 4, 8) : W4A16_TMA_LAUNCH(2, 2, 8);
    }
    if (cw == 4) {
        if (nt == 1) return bns == 4 ? W4A16_TMA_LAUNCH(1, 4, 4) : W4A16_TMA_LAUNCH(1, 2, 4);
        return bns == 4 ? W4A16_TMA_LAUNCH(2, 4, 4) : W4A16_TMA_LAUNCH(2, 2, 4);
    }
    if (nt == 1) return bns == 4 ? W4A16_TMA_LAUNCH(1, 4, 16) : W4A16_TMA_LAUNCH(1, 2, 16);
    return bns == 4 ? W4A16_TMA_LAUNCH(2, 4, 16) : W4A16_TMA_LAUNCH(2, 2, 16);
#undef W4A16_TMA_LAUNCH
#undef W4A16_TMA_LAUNCH1
}

}  // namespace w4a16
