// skinny.cu -- OUT_PROD for narrow src1 (N <= 32), f32 src0.
//
// The rank-r LoRA parameter gradient ("metal: OUT_PROD runs batched, broadcast
// and narrow shapes on the GPU", list item 2: widths that are not multiples of
// 16) is out_prod(x, dy) with N = r in {4, 8, 24}.  Its cost is reading src0
// once from HBM; arithmetic is 2N flops per 4-byte element.
//
// Design (GB300):
//  * lanes split m: each lane owns VW consecutive m (one 16- or 8-byte load
//    per k row), so a warp reads 32*VW*4 contiguous bytes per row and no
//    intra-warp reduction is needed;
//  * warps of a CTA split k; every thread issues the loads of its next chunk of
//    k rows before multiplying the current one (register double buffer), so
//    each thread keeps KW loads in flight;
//  * b's panel (k rows x N) is staged in shared memory and read as broadcast
//    float4s;
//  * the 8 warps' partial sums meet in shared memory (fixed warp order), and
//    the S CTAs that split K form one thread-block cluster whose partials are
//    summed through distributed shared memory (fixed rank order): one writer
//    per dst element, deterministic, no workspace, no atomics;
//  * every head x batch slice is a grid.z index of the same launch.
#include <cooperative_groups.h>

#include <algorithm>

#include "oop_internal.cuh"

namespace cg = cooperative_groups;

namespace oop {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kKW = 8;                    // k rows per warp per chunk
constexpr int kChunk = kWarps * kKW;      // k rows per CTA per chunk
constexpr int kMaxCluster = 8;            // portable cluster size

struct SkinnyArgs {
    const float *a;
    const float *b;
    float *dst;
    int64_t M, K, N;
    int64_t ne02, ne12;
    int64_t dps2, dps3;
    int64_t kc;         // k rows per CTA of a cluster
    int super_rows;     // b rows staged per shared-memory fill
};

template <int VW>
struct VecT;
template <>
struct VecT<4> { using T = float4; };
template <>
struct VecT<2> { using T = float2; };
template <>
struct VecT<1> { using T = float; };

template <int VW>
__device__ __forceinline__ void load_a(float (&v)[VW], const float *row, int64_t m0,
                                       int64_t M, bool ok) {
    if constexpr (VW == 4) {
        float4 t = ok && m0 < M ? __ldg(reinterpret_cast<const float4 *>(row + m0))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else if constexpr (VW == 2) {
        float2 t = ok && m0 < M ? __ldg(reinterpret_cast<const float2 *>(row + m0))
                                : make_float2(0.f, 0.f);
        v[0] = t.x; v[1] = t.y;
    } else {
        v[0] = ok && m0 < M ? __ldg(row + m0) : 0.f;
    }
}

// NP: N rounded up to a multiple of 4 (register accumulators NP x VW).
// VW: consecutive m per lane (4 or 2 with 16/8-byte loads; 1 = scalar loads,
// taken when src0's rows are not aligned for vectors).
template <int NP, int VW>
__global__ void __launch_bounds__(kThreads, 2) skinny_kernel(SkinnyArgs p) {
    constexpr int MT = 32 * VW;                 // m per CTA
    extern __shared__ __align__(16) float smem[];
    float *bs = smem;                           // [super_rows][NP]
    float *red = bs + p.super_rows * NP;        // [kWarps][4][MT]
    float *part = red + kWarps * 4 * MT;        // [NP][MT]

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t slice = blockIdx.z;
    const int64_t i2 = slice % p.ne12, i3 = slice / p.ne12;
    const int64_t j2 = i2 / p.dps2, j3 = i3 / p.dps3;
    const float *a = p.a + (j3 * p.ne02 + j2) * p.K * p.M;
    const float *b = p.b + slice * p.K * p.N;
    float *dst = p.dst + slice * p.N * p.M;

    const int64_t mt0 = static_cast<int64_t>(blockIdx.x) * MT;
    const int64_t m0 = mt0 + lane * VW;
    const int64_t kb = static_cast<int64_t>(blockIdx.y) * p.kc;
    const int64_t ke = min(p.K, kb + p.kc);

    float acc[NP][VW];
#pragma unroll
    for (int n = 0; n < NP; ++n)
#pragma unroll
        for (int v = 0; v < VW; ++v) acc[n][v] = 0.f;

    // Scalar loads must stay inside the row for every element.
    auto load_row = [&](float (&v)[VW], int64_t k, bool ok) {
        const float *row = a + k * p.M;
        if constexpr (VW == 1) {
            load_a<1>(v, row, m0, p.M, ok);
        } else {
            load_a<VW>(v, row, m0, p.M, ok);
        }
    };

    float av[kKW][VW], an[kKW][VW];
#pragma unroll
    for (int j = 0; j < kKW; ++j) {
        const int64_t k = kb + warp * kKW + j;
        load_row(av[j], k, k < ke);
    }

    for (int64_t ks = kb; ks < ke; ks += p.super_rows) {
        const int64_t kse = min(ke, ks + p.super_rows);
        __syncthreads();                         // bs free
        for (int64_t idx = threadIdx.x; idx < (kse - ks) * NP; idx += kThreads) {
            const int64_t r = idx / NP;
            const int n = static_cast<int>(idx % NP);
            bs[idx] = n < p.N ? __ldg(b + (ks + r) * p.N + n) : 0.f;
        }
        __syncthreads();
        for (int64_t kk = ks; kk < kse; kk += kChunk) {
            // prefetch the next chunk's rows of src0 before using this one
            const int64_t kn = kk + kChunk;
#pragma unroll
            for (int j = 0; j < kKW; ++j) {
                const int64_t k = kn + warp * kKW + j;
                load_row(an[j], k, k < ke);
            }
#pragma unroll
            for (int j = 0; j < kKW; ++j) {
                const int64_t r = kk - ks + warp * kKW + j;
                if (kk + warp * kKW + j < kse) {
                    const float *brow = bs + r * NP;
#pragma unroll
                    for (int n4 = 0; n4 < NP; n4 += 4) {
                        const float4 bv = *reinterpret_cast<const float4 *>(brow + n4);
#pragma unroll
                        for (int v = 0; v < VW; ++v) {
                            acc[n4 + 0][v] = fmaf(av[j][v], bv.x, acc[n4 + 0][v]);
                            acc[n4 + 1][v] = fmaf(av[j][v], bv.y, acc[n4 + 1][v]);
                            acc[n4 + 2][v] = fmaf(av[j][v], bv.z, acc[n4 + 2][v]);
                            acc[n4 + 3][v] = fmaf(av[j][v], bv.w, acc[n4 + 3][v]);
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kKW; ++j)
#pragma unroll
                for (int v = 0; v < VW; ++v) av[j][v] = an[j][v];
        }
    }

    // ---- reduce the 8 warps (fixed order), 4 n at a time ----
#pragma unroll
    for (int nc = 0; nc < NP; nc += 4) {
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int v = 0; v < VW; ++v)
                red[(warp * 4 + q) * MT + lane * VW + v] = acc[nc + q][v];
        __syncthreads();
        for (int o = threadIdx.x; o < 4 * MT; o += kThreads) {
            const int q = o / MT, mm = o % MT;
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) s += red[(w * 4 + q) * MT + mm];
            part[(nc + q) * MT + mm] = s;
        }
    }

    // ---- reduce the cluster's CTAs (fixed rank order) and store ----
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int S = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int64_t total = p.N * MT;
    for (int64_t o = static_cast<int64_t>(rank) * kThreads + threadIdx.x; o < total;
         o += static_cast<int64_t>(S) * kThreads) {
        const int64_t n = o / MT;
        const int mm = static_cast<int>(o % MT);
        float s = 0.f;
        for (int q = 0; q < S; ++q) {
            const float *rp = cluster.map_shared_rank(part, q);
            s += rp[n * MT + mm];
        }
        const int64_t m = mt0 + mm;
        if (m < p.M) dst[n * p.M + m] = s;
    }
    cluster.sync();   // keep this CTA's shared memory alive for the readers
}

template <int NP, int VW>
cudaError_t launch_np(const SkinnyArgs &args0, const OutProdShape &s, cudaStream_t stream) {
    constexpr int MT = 32 * VW;
    SkinnyArgs args = args0;
    const int64_t mtiles = (s.M + MT - 1) / MT;
    const int64_t slices = s.ne12 * s.ne13;

    // Split K over a cluster of S CTAs: enough CTAs for about two per SM,
    // at least one chunk of rows each.
    int sms = device_sm_count();
    if (sms <= 0) sms = 152;
    int S = 1;
    while (S < kMaxCluster && mtiles * slices * (S * 2) <= 2 * sms &&
           (s.K + S * 2 - 1) / (S * 2) >= kChunk)
        S *= 2;
    args.kc = ((s.K + S - 1) / S + kKW - 1) / kKW * kKW;
    args.super_rows = std::max<int>(kChunk, (8192 / NP) / kChunk * kChunk);   // 32 KB of b

    const size_t smem = sizeof(float) *
        (static_cast<size_t>(args.super_rows) * NP + kWarps * 4 * MT + NP * MT);
    auto kern = skinny_kernel<NP, VW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;

    if (mtiles > 0x7fffffffLL || slices > 65535) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(mtiles), static_cast<unsigned>(S),
                       static_cast<unsigned>(slices));
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = static_cast<unsigned>(S);
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

template <int VW>
cudaError_t launch_vw(const SkinnyArgs &args, const OutProdShape &s, cudaStream_t stream) {
    const int64_t np = (s.N + 3) / 4 * 4;
    switch (np) {
    case 4: return launch_np<4, VW>(args, s, stream);
    case 8: return launch_np<8, VW>(args, s, stream);
    case 12: return launch_np<12, VW>(args, s, stream);
    case 16: return launch_np<16, VW>(args, s, stream);
    case 20: return launch_np<20, VW == 4 ? 2 : VW>(args, s, stream);
    case 24: return launch_np<24, VW == 4 ? 2 : VW>(args, s, stream);
    case 28: return launch_np<28, VW == 4 ? 2 : VW>(args, s, stream);
    case 32: return launch_np<32, VW == 4 ? 2 : VW>(args, s, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_skinny(const float *a, const float *b, float *dst, const OutProdShape &s,
                          cudaStream_t stream) {
    SkinnyArgs args = {};
    args.a = a;
    args.b = b;
    args.dst = dst;
    args.M = s.M;
    args.K = s.K;
    args.N = s.N;
    args.ne02 = s.ne02;
    args.ne12 = s.ne12;
    args.dps2 = s.dps2;
    args.dps3 = s.dps3;
    if (s.N < 1 || s.N > 32) return cudaErrorInvalidValue;
    // 16-byte rows allow float4 loads; 8-byte rows float2; else scalars.
    const uintptr_t ab = reinterpret_cast<uintptr_t>(a);
    if (ab % 16 == 0 && s.M % 4 == 0) return launch_vw<4>(args, s, stream);
    if (ab % 8 == 0 && s.M % 2 == 0) return launch_vw<2>(args, s, stream);
    return launch_vw<1>(args, s, stream);
}

}  // namespace oop
