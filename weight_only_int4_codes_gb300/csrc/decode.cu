// decode.cu -- W4A16 GEMM for small M (the decode regime, M <= 16 per pass).
//
// What it computes: out[m,n] = sum_k x[m,k] * (q[k,n] - z[g(k),n]) * s[g(k),n],
// fp32 accumulation, fp16 result (page "Beating FP16 with 4-bit Weights: A
// Portable W4A16 GEMM in Triton", sections "The design" and "Things I got wrong
// along the way"; page "Triton Kernel Matches bitsandbytes: Why Both Lose to
// Math", sections "Three Kernel Versions" and "Why Marlin Is Still Faster").
//
// At M <= 16 the GEMM is a race to stream the packed weight out of HBM; the
// design follows from that:
//   * Every packed word is loaded exactly once, as part of a 128-bit load of
//     four neighbouring columns (coalesced along N), with an L2 evict-first
//     hint and no L1 allocation.  (The 8x redundant word load is the first
//     mistake the first page describes.)
//   * Nibbles become fp16 in registers with the magic-exponent trick: OR-ing a
//     nibble into the mantissa of 1024.0 (0x6400, low nibble) or 64.0 (0x5400,
//     nibble shifted by 4) yields 1024+q or 64+q exactly, one LOP3 per two
//     codes.  Subtracting the matching 1024+z / 64+z gives q - z exactly.
//   * The multiply-accumulate runs on the tensor cores through register-fed
//     mma.m16n8k16 with the roles swapped: the 16 "rows" of the MMA are 16
//     output columns of W, the 8 "columns" are batch rows of x.  K may be
//     permuted freely inside the reduction as long as x and W use the same
//     permutation, so each thread's 128-bit word load maps directly onto A
//     fragments, and x is permuted to match with four PRMTs.  CUDA-core FMA
//     cannot keep up with HBM at M >= 2 (it needs M FMAs per weight).
//   * The scale is applied once per group in fp32 to the MMA's group partial
//     (acc += s * sum_k x (q - z)), not per weight.
//   * Split-K: a column tile's K range is split across the warps of a CTA and
//     across the CTAs of one thread-block cluster.  Partials are reduced in a
//     FIXED order: warps through shared memory, then CTAs through distributed
//     shared memory -- every CTA finalizes a slice of the tile, its peers push
//     their partials of that slice into its shared memory, one cluster barrier.
//     No atomics, no global workspace, no spin-waits, bitwise reproducible.  (The pages merge split-K partials
//     with fp32 atomics; the second page names a second-stage reduction as the
//     alternative, which this is.)
#include <map>
#include <mutex>

#include "common.cuh"
#include "decode_math.cuh"
#include "sm100_ptx.cuh"

namespace w4a16 {
namespace {

constexpr bool kRegZeroFree = true;   // M <= 8: decode_math.cuh's zero-free step

struct DecodeArgs {
    const uint16_t *x;
    const uint32_t *packed;
    const uint16_t *scales;
    const uint16_t *zeros;
    uint16_t *out;
    int M, N, K, group;
    int steps;          // 32-row K steps per warp (a multiple of U)
    int rows_per_cta;   // packed rows per CTA = warps_k * steps * 4
    int split;          // CTAs along K = gridDim.y = cluster size
};

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Weight stream: read once, never reused by this SM -> no L1 allocation,
// evict-first in L2.
__device__ __forceinline__ uint4 ld_weights(const uint32_t *ptr, uint64_t pol) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(ptr), "l"(pol));
    return r;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void *ptr) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(ptr));
    return r;
}

__device__ __forceinline__ uint2 ld_nc_v2(const void *ptr) {
    uint2 r;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(ptr));
    return r;
}

// One K-batch of U steps: the words of 4 columns x U steps, plus that batch's
// group scale and zero (a batch never straddles a group).
template <int U>
struct Batch {
    uint4 w[U];
    uint2 s, z;
};

// Threads whose columns lie past N (ragged last tile) load nothing and feed
// zeros: the batch loop itself must stay warp-uniform because mma.sync is a
// warp-collective (.aligned) instruction.
template <int U>
__device__ __forceinline__ void load_batch(Batch<U> &b, bool col_ok, const uint32_t *wptr,
                                           size_t wstride, const uint16_t *sz_s,
                                           const uint16_t *sz_z, uint64_t pol) {
    if (col_ok) {
#pragma unroll
        for (int u = 0; u < U; ++u) b.w[u] = ld_weights(wptr + u * wstride, pol);
        b.s = ld_nc_v2(sz_s);
        b.z = ld_nc_v2(sz_z);
    } else {
#pragma unroll
        for (int u = 0; u < U; ++u) b.w[u] = make_uint4(0, 0, 0, 0);
        b.s = make_uint2(0, 0);
        b.z = make_uint2(0, 0);
    }
}

// The MMA work of one batch (see decode_math.cuh for the fragment mapping):
// thread (g, t) handles, in step u, packed row  row = krow_first + 4u + t.
// fp16: the batch's MMAs accumulate q - z, and the group scale is applied to
// their sum (acc).  bfloat16 (BF): every weight is dequantized with its scale
// first, and the MMAs accumulate into the running sums accb.
template <int NT, int U, bool BF>
__device__ __forceinline__ void compute_batch(float (&acc)[NT][2][4], float (&accb)[NT][2][2][4],
                                              const Batch<U> &b, const uint16_t *xrow0,
                                              const uint16_t *xrow1, bool m0_ok, bool m1_ok,
                                              int krow_first, int t) {
    // x fragments of all U steps first (several loads in flight)
    uint4 xr[NT][U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int koff = 8 * (krow_first + 4 * u + t);
        xr[0][u] = m0_ok ? ld_nc_v4(xrow0 + koff) : make_uint4(0, 0, 0, 0);
        if (NT > 1) xr[NT - 1][u] = m1_ok ? ld_nc_v4(xrow1 + koff) : make_uint4(0, 0, 0, 0);
    }
    if constexpr (BF) {
        const GroupConstsBf k = make_group_consts_bf(b.z, b.s);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint32_t bx[NT][4];
#pragma unroll
            for (int p = 0; p < NT; ++p) x_fragments(xr[p][u], bx[p]);
            step_mma_bf16<NT>(accb, b.w[u], k, bx);
        }
    } else if constexpr (NT == 1 && kRegZeroFree) {
        // M <= 8: the zero-free step (codes as fp16 subnormals, the zero
        // removed per group through the x sums)
        const ZfConsts zk = make_zf_consts(b.z, b.s);
        float dlo[2][4], dhi[2][4], dx[4];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint32_t blo[2], bhi[2];
            blo[0] = __byte_perm(xr[0][u].x, xr[0][u].z, 0x5410);   // (x0, x4)
            blo[1] = __byte_perm(xr[0][u].y, xr[0][u].w, 0x5410);   // (x2, x6)
            bhi[0] = __byte_perm(xr[0][u].x, xr[0][u].z, 0x7632);   // (x1, x5)
            bhi[1] = __byte_perm(xr[0][u].y, xr[0][u].w, 0x7632);   // (x3, x7)
            if (u == 0)
                zf_step<true>(dlo, dhi, dx, b.w[u], blo, bhi);
            else
                zf_step<false>(dlo, dhi, dx, b.w[u], blo, bhi);
        }
        zf_flush(acc, dlo, dhi, dx, zk);
    } else {
        const GroupConsts k = make_group_consts(b.z, b.s);
        float gacc[NT][2][2][4];
#pragma unroll
        for (int p = 0; p < NT; ++p)
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int r = 0; r < 4; ++r) gacc[p][j][0][r] = gacc[p][j][1][r] = 0.f;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint32_t bx[NT][4];
#pragma unroll
            for (int p = 0; p < NT; ++p) x_fragments(xr[p][u], bx[p]);
            step_mma_split<NT>(gacc, b.w[u], k, bx);
        }
        flush_group_split<NT>(acc, gacc, k);
    }
}

// The operands of one GEMM of a launch (one expert of a grouped launch).
struct Operands {
    const uint16_t *x;
    const uint32_t *packed;
    const uint16_t *scales;
    const uint16_t *zeros;
    uint16_t *out;
};

// Up to kMaxExperts weight sets and activations of one grouped launch, passed
// by value in the kernel's parameter block (nothing is allocated per call).
struct ExpertTable {
    Operands e[kMaxExperts];
};

// One CTA's share of one GEMM: column tile blockIdx.x, K slice blockIdx.y,
// 16-row chunk `mchunk` of x.  BF: x, scales, zeros and out are bfloat16.
// Block: 32*WN*WK threads; dynamic shared memory (WK + 1) * 16 * 32*WN + 8 floats.
template <int NT, int WN, int WK, int U, bool BF>
__device__ __forceinline__ void decode_tile(const DecodeArgs &a, const Operands &o, int mchunk)
{
    extern __shared__ float smem[];
    constexpr int BN = 32 * WN;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wn = warp % WN, wk = warp / WN;
    const int g = lane >> 2, t = lane & 3;
    const int m_base = mchunk * 16;
    const int Mc = min(16, a.M - m_base);
    const int col0 = blockIdx.x * BN + wn * 32 + 4 * g;
    const bool col_ok = col0 < a.N;                 // N % 4 == 0: all 4 columns valid
    const int KB = a.K >> 3;                        // packed rows
    // first half of a split cluster barrier: once every CTA has arrived, each
    // one's shared memory exists and may receive its peers' partials
    if (a.split > 1) cluster_arrive();
    const int row0 = blockIdx.y * a.rows_per_cta + wk * a.steps * 4;
    // warp-uniform trip count (independent of col_ok)
    const int nsteps = max(0, min(a.steps, (KB - row0) >> 2));
    const int nbatch = nsteps / U;                  // nsteps is a multiple of U

    const uint64_t pol = evict_first_policy();
    const size_t wstride = (size_t)4 * a.N;         // one step = 4 packed rows
    const uint32_t *wptr = o.packed + (size_t)(row0 + t) * a.N + col0;
    const uint16_t *sptr = o.scales + col0;
    const uint16_t *zptr = o.zeros + col0;
    // group row of batch b: (8 * (row0 + 4*U*b)) / group
    const int rows_per_group = a.group >> 3;

    float acc[NT][2][4];
    float accb[NT][2][2][4];   // bfloat16 only (two k halves)
#pragma unroll
    for (int p = 0; p < NT; ++p)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[p][j][r] = accb[p][j][0][r] = accb[p][j][1][r] = 0.f;

    const int m0 = g, m1 = 8 + g;
    const bool m0_ok = m0 < Mc, m1_ok = m1 < Mc;
    const uint16_t *xrow0 = o.x + (size_t)(m_base + (m0_ok ? m0 : 0)) * a.K;
    const uint16_t *xrow1 = o.x + (size_t)(m_base + (m1_ok ? m1 : 0)) * a.K;

    Batch<U> ba, bb;
    if (nbatch > 0) {
        const size_t grow = (size_t)(row0 / rows_per_group) * a.N;
        load_batch<U>(ba, col_ok, wptr, wstride, sptr + grow, zptr + grow, pol);
    }
    // Everything above only touches the weights.  x and out may belong to the
    // previous kernel on the stream (programmatic dependent launch).
    pdl_wait();
    pdl_launch_dependents();

    for (int bi = 0; bi < nbatch; bi += 2) {
        if (bi + 1 < nbatch) {
            const int r = row0 + 4 * U * (bi + 1);
            const size_t grow = (size_t)(r / rows_per_group) * a.N;
            load_batch<U>(bb, col_ok, wptr + (size_t)(bi + 1) * U * wstride, wstride,
                          sptr + grow, zptr + grow, pol);
        }
        compute_batch<NT, U, BF>(acc, accb, ba, xrow0, xrow1, m0_ok, m1_ok, row0 + 4 * U * bi, t);
        if (bi + 1 < nbatch) {
            if (bi + 2 < nbatch) {
                const int r = row0 + 4 * U * (bi + 2);
                const size_t grow = (size_t)(r / rows_per_group) * a.N;
                load_batch<U>(ba, col_ok, wptr + (size_t)(bi + 2) * U * wstride, wstride,
                              sptr + grow, zptr + grow, pol);
            }
            compute_batch<NT, U, BF>(acc, accb, bb, xrow0, xrow1, m0_ok, m1_ok,
                                     row0 + 4 * U * (bi + 1), t);
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

    // ---- reduction 1: the WK warps of this CTA, through shared memory
    float *red = smem;                    // [WK][16][BN]
#pragma unroll
    for (int p = 0; p < NT; ++p)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int m = 8 * p + 2 * t + (r & 1);
                const int c = wn * 32 + 4 * g + 2 * j + (r >> 1);
                if (m < Mc) red[(wk * 16 + m) * BN + c] = acc[p][j][r];
            }
    __syncthreads();
    const int E = Mc * BN;
    if (a.split > 1) {
        // ---- reduction 2: every CTA pushes its partial of output e into the
        // slot [rank][e - q*per] of the CTA q that finalizes e; one cluster
        // barrier; each CTA sums its slots in rank order (fixed: bitwise
        // reproducible).  No CTA reads another's shared memory.
        const int rank = (int)cluster_ctarank();
        const int per = (E + a.split - 1) / a.split;
        float *slots = smem + WK * 16 * BN;         // [split][per]
        cluster_wait();
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            const int m = e / BN, c = e - m * BN;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < WK; ++w) v += red[(w * 16 + m) * BN + c];
            const int q = e / per;
            st_cluster_f32(map_to_rank(smem_u32(slots + rank * per + (e - q * per)), q), v);
        }
        cluster_arrive();
        cluster_wait();
        const int e0 = rank * per, e1 = min(E, e0 + per);
        for (int e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
            float v = 0.f;
            for (int q = 0; q < a.split; ++q) v += slots[q * per + (e - e0)];
            const int m = e / BN, c = e - m * BN;
            const int col = blockIdx.x * BN + c;
            if (col < a.N)
                o.out[(size_t)(m_base + m) * a.N + col] = to_out<BF>(v);
        }
        return;
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int m = e / BN, c = e - m * BN;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < WK; ++w) v += red[(w * 16 + m) * BN + c];
        const int col = blockIdx.x * BN + c;
        if (col < a.N)
            o.out[(size_t)(m_base + m) * a.N + col] = to_out<BF>(v);
    }
}

// Grid: (ceil(N / (32*WN)), split, ceil(M / 16)); cluster (1, split, 1).
template <int NT, int WN, int WK, int U, bool BF>
__global__ void __launch_bounds__(32 * WN * WK)
decode_kernel(const DecodeArgs a)
{
    const Operands o{a.x, a.packed, a.scales, a.zeros, a.out};
    decode_tile<NT, WN, WK, U, BF>(a, o, blockIdx.z);
}

// Grouped launch of E GEMMs of one shape (MoE experts): grid z = E * ceil(M / 16),
// expert e = z / mchunks.  Same tiles, same arithmetic, one launch.
template <int NT, int WN, int WK, int U>
__global__ void __launch_bounds__(32 * WN * WK)
decode_grouped_kernel(const DecodeArgs a, const ExpertTable tab)
{
    const int mchunks = (a.M + 15) >> 4;
    const int e = blockIdx.z / mchunks;
    decode_tile<NT, WN, WK, U, false>(a, tab.e[e], blockIdx.z - e * mchunks);
}

template <int NT, int WN, int WK, int U, bool BF>
cudaError_t launch_one(const DecodeArgs &da, int strips, int mchunks, bool pdl,
                       cudaStream_t stream) {
    constexpr int BN = 32 * WN;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(strips, da.split, mchunks);
    lc.blockDim = dim3(32 * WN * WK, 1, 1);
    lc.dynamicSmemBytes = ((size_t)(WK + 1) * 16 * BN + 8) * sizeof(float);
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
    return cudaLaunchKernelEx(&lc, decode_kernel<NT, WN, WK, U, BF>, da);
}

template <int NT, int WN, int WK, int U>
cudaError_t launch_grouped_one(const DecodeArgs &da, const ExpertTable &tab, int strips, int zdim,
                               bool pdl, cudaStream_t stream) {
    constexpr int BN = 32 * WN;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(strips, da.split, zdim);
    lc.blockDim = dim3(32 * WN * WK, 1, 1);
    lc.dynamicSmemBytes = ((size_t)(WK + 1) * 16 * BN + 8) * sizeof(float);
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
    return cudaLaunchKernelEx(&lc, decode_grouped_kernel<NT, WN, WK, U>, da, tab);
}

template <int NT, int U>
cudaError_t launch_grouped_shape(const DecodeArgs &da, const ExpertTable &tab, int wn, int wk,
                                 int strips, int zdim, bool pdl, cudaStream_t s) {
    if (wn == 1 && wk == 4) return launch_grouped_one<NT, 1, 4, U>(da, tab, strips, zdim, pdl, s);
    if (wn == 1 && wk == 8) return launch_grouped_one<NT, 1, 8, U>(da, tab, strips, zdim, pdl, s);
    if (wn == 2 && wk == 4) return launch_grouped_one<NT, 2, 4, U>(da, tab, strips, zdim, pdl, s);
    if (wn == 4 && wk == 2) return launch_grouped_one<NT, 4, 2, U>(da, tab, strips, zdim, pdl, s);
    if (wn == 2 && wk == 2) return launch_grouped_one<NT, 2, 2, U>(da, tab, strips, zdim, pdl, s);
    return cudaErrorNotSupported;
}

template <int NT, int U, bool BF>
cudaError_t launch_shape(const DecodeArgs &da, int wn, int wk, int strips, int mchunks,
                         bool pdl, cudaStream_t s) {
    if (wn == 1 && wk == 4) return launch_one<NT, 1, 4, U, BF>(da, strips, mchunks, pdl, s);
    if (wn == 1 && wk == 8) return launch_one<NT, 1, 8, U, BF>(da, strips, mchunks, pdl, s);
    if (wn == 2 && wk == 4) return launch_one<NT, 2, 4, U, BF>(da, strips, mchunks, pdl, s);
    if (wn == 4 && wk == 2) return launch_one<NT, 4, 2, U, BF>(da, strips, mchunks, pdl, s);
    if (wn == 2 && wk == 2) return launch_one<NT, 2, 2, U, BF>(da, strips, mchunks, pdl, s);
    return cudaErrorNotSupported;
}

int steps_per_batch(int group) {
    const int spg = group / 32;
    return spg % 4 == 0 ? 4 : (spg % 2 == 0 ? 2 : 1);
}

}  // namespace

namespace {
template <int NT, int U>
const void *kernel_for(int wn, int wk) {
    if (wn == 1 && wk == 4) return (const void *)decode_kernel<NT, 1, 4, U, false>;
    if (wn == 1 && wk == 8) return (const void *)decode_kernel<NT, 1, 8, U, false>;
    if (wn == 2 && wk == 4) return (const void *)decode_kernel<NT, 2, 4, U, false>;
    if (wn == 4 && wk == 2) return (const void *)decode_kernel<NT, 4, 2, U, false>;
    if (wn == 2 && wk == 2) return (const void *)decode_kernel<NT, 2, 2, U, false>;
    return nullptr;
}
}  // namespace

int decode_ctas_per_sm(const w4a16_config &cfg, int M, int group) {
    const int U = steps_per_batch(group);
    const bool nt2 = M > 8;
    const void *fn = nullptr;
    if (U == 4) fn = nt2 ? kernel_for<2, 4>(cfg.warps_n, cfg.warps_k) : kernel_for<1, 4>(cfg.warps_n, cfg.warps_k);
    else if (U == 2) fn = nt2 ? kernel_for<2, 2>(cfg.warps_n, cfg.warps_k) : kernel_for<1, 2>(cfg.warps_n, cfg.warps_k);
    else fn = nt2 ? kernel_for<2, 1>(cfg.warps_n, cfg.warps_k) : kernel_for<1, 1>(cfg.warps_n, cfg.warps_k);
    const int threads = 32 * cfg.warps_n * cfg.warps_k;
    const size_t smem = ((size_t)(cfg.warps_k + 1) * 16 * 32 * cfg.warps_n + 8) * sizeof(float);
    // occupancy is a property of the kernel, so the answer is cached per kernel
    static std::mutex mu;
    static std::map<const void *, int> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(fn);
        if (it != cache.end()) return it->second;
    }
    int n = 0, ndev = 0;
    if (!(fn && cudaGetDeviceCount(&ndev) == cudaSuccess && ndev > 0 &&
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) == cudaSuccess &&
          n > 0)) {
        cudaGetLastError();
        // no GPU: registers (about 100 per thread at M <= 8, 128 above) bound it
        const int regs = nt2 ? 128 : 104;
        n = 65536 / (regs * threads);
        if (n < 1) n = 1;
    }
    std::lock_guard<std::mutex> lock(mu);
    cache[fn] = n;
    return n;
}

bool decode_config_supported(const w4a16_config &cfg, int /*M*/) {
    const int wn = cfg.warps_n, wk = cfg.warps_k;
    const bool shape_ok = (wn == 1 && (wk == 4 || wk == 8)) || (wn == 2 && (wk == 4 || wk == 2)) ||
                          (wn == 4 && wk == 2);
    return shape_ok && cfg.split_k >= 1 && cfg.split_k <= 8 && cfg.steps >= 1;
}

cudaError_t launch_decode(const GemmArgs &a, const w4a16_config &cfg, cudaStream_t stream) {
    if (!decode_config_supported(cfg, a.M)) return cudaErrorNotSupported;
    const bool bf = cfg.dtype == W4A16_DTYPE_BF16;
    const int U = steps_per_batch(a.group);
    if (cfg.steps % U != 0) return cudaErrorNotSupported;
    DecodeArgs da;
    da.x = a.x;
    da.packed = a.packed;
    da.scales = a.scales;
    da.zeros = a.zeros;
    da.out = a.out;
    da.M = a.M;
    da.N = a.N;
    da.K = a.K;
    da.group = a.group;
    da.steps = cfg.steps;
    da.rows_per_cta = cfg.warps_k * cfg.steps * 4;
    da.split = cfg.split_k;
    // the split CTAs must cover K
    const long long covered = (long long)da.rows_per_cta * da.split;
    if (covered < a.K / 8) return cudaErrorInvalidValue;
    const int strips = (a.N + 32 * cfg.warps_n - 1) / (32 * cfg.warps_n);
    const int mchunks = (a.M + 15) / 16;
    if (mchunks > 65535) return cudaErrorInvalidValue;
    const bool pdl = (cfg.flags & W4A16_FLAG_PDL) != 0;
    const bool nt2 = a.M > 8;
#define W4A16_DECODE(NT_, U_)                                                                   \
    (bf ? launch_shape<NT_, U_, true>(da, cfg.warps_n, cfg.warps_k, strips, mchunks, pdl, stream) \
        : launch_shape<NT_, U_, false>(da, cfg.warps_n, cfg.warps_k, strips, mchunks, pdl, stream))
    switch (U) {
    case 4: return nt2 ? W4A16_DECODE(2, 4) : W4A16_DECODE(1, 4);
    case 2: return nt2 ? W4A16_DECODE(2, 2) : W4A16_DECODE(1, 2);
    default: return nt2 ? W4A16_DECODE(2, 1) : W4A16_DECODE(1, 1);
    }
#undef W4A16_DECODE
}

cudaError_t launch_decode_grouped(const GroupedGemmArgs &a, const w4a16_config &cfg,
                                  cudaStream_t stream) {
    if (!decode_config_supported(cfg, a.M) || a.E < 1 || a.E > kMaxExperts || a.M > 16)
        return cudaErrorNotSupported;
    const int U = steps_per_batch(a.group);
    if (cfg.steps % U != 0) return cudaErrorNotSupported;
    DecodeArgs da = {};
    da.M = a.M;
    da.N = a.N;
    da.K = a.K;
    da.group = a.group;
    da.steps = cfg.steps;
    da.rows_per_cta = cfg.warps_k * cfg.steps * 4;
    da.split = cfg.split_k;
    if ((long long)da.rows_per_cta * da.split < a.K / 8) return cudaErrorInvalidValue;
    ExpertTable tab = {};
    for (int e = 0; e < a.E; ++e)
        tab.e[e] = Operands{a.x[e], a.packed[e], a.scales[e], a.zeros[e], a.out[e]};
    const int strips = (a.N + 32 * cfg.warps_n - 1) / (32 * cfg.warps_n);
    const int zdim = a.E;                    // M <= 16: one 16-row chunk per expert
    const bool pdl = (cfg.flags & W4A16_FLAG_PDL) != 0;
    const bool nt2 = a.M > 8;
#define W4A16_GROUPED(NT_, U_) \
    launch_grouped_shape<NT_, U_>(da, tab, cfg.warps_n, cfg.warps_k, strips, zdim, pdl, stream)
    switch (U) {
    case 4: return nt2 ? W4A16_GROUPED(2, 4) : W4A16_GROUPED(1, 4);
    case 2: return nt2 ? W4A16_GROUPED(2, 2) : W4A16_GROUPED(1, 2);
    default: return nt2 ? W4A16_GROUPED(2, 1) : W4A16_GROUPED(1, 1);
    }
#undef W4A16_GROUPED
}

int decode_steps_per_batch(int group) { return steps_per_batch(group); }

}  // namespace w4a16
