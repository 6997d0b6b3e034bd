// skinny_tma.cu -- OUT_PROD for narrow src1 (N <= 32) on large f32 problems:
// a persistent, TMA-fed form of the skinny-N kernel.
//
// The cost of a rank-r gradient is reading src0 once from HBM.  With many
// slices (a batch of LoRA gradients, long sequences) the register
// double-buffered skinny kernel keeps too few bytes in flight to fill HBM
// (it levels off near 3.6 TB/s).  Here:
//  * one CTA per SM walks work items (dst slice, m-tile of 32*VW columns) in a
//    fixed order: item = blockIdx.x + j * gridDim.x;
//  * a TMA warp streams each item's src0 rows (boxes of 64 k x TM m, zero
//    filled past M) and the matching rows of src1 (64 k x N words, one bulk
//    copy) through a ring of shared-memory stages, independently of the
//    consumers, so several stages (17-41 KB each) stay in flight per SM and
//    the next item's rows arrive while the current one is being reduced;
//  * eight consumer warps split each stage's 64 k rows (8 each); lane = VW
//    consecutive m, N*VW fp32 accumulators per thread held as (n, n+1)
//    pairs and updated with packed f32x2 FMAs (half the issue slots of
//    scalar FMAs; the same round-to-nearest products and sums), b read as
//    broadcast float4s; in a full stage, where the registers allow (N <= 20
//    at four m per lane), each row's loads are issued before the previous
//    row's FMAs;
//  * at the end of an item warps 4-7 hand their partials to warps 0-3
//    through shared memory, then warps 0-3 publish theirs and one thread per
//    output adds the four in warp order and writes dst: deterministic, one
//    writer per element, no atomics, no workspace.
// Every lane needs every src1 value of a row, and a broadcast from shared
// memory delivers 4 bytes per wavefront whatever the load width, so a row
// costs N wavefronts for src1 against VW for src0: four m per lane (TM = 128)
// halves that cost per byte against two; N = 28 and 32 keep two m per lane
// (four would not fit in the registers), and so do N = 20 and 24 when items
// of 128 m would leave fewer than two per SM.
// Waits are bounded like the tensor-core kernel's: running out records
// OOP_ERR_DEVICE_TIMEOUT, every role stops, the TMA warp drains its copies.
#include <algorithm>
#include <cstring>

#include "oop_internal.cuh"
#include "tc_ptx.cuh"

namespace oop {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;        // + the TMA warp
constexpr int kTK = 64;                          // k rows per stage
constexpr int kRowsPerWarp = kTK / kConsumerWarps;
constexpr int kMaxStages = 8;
constexpr uint64_t kWaitNs = 1000000000ull;

struct TmaArgs {
    const float *b;
    float *dst;
    int *status;
    int64_t M, K, N, ne02, ne12, dps2, dps3;
    int64_t mtiles, items;      // items = slices * mtiles
    int kstages;                // ceil(K / kTK)
};

// Problems per batch launch (their tensor maps sit in the kernel parameters).
constexpr int kMaxBatch = 48;

struct BatchArgs {
    CUtensorMap maps[kMaxBatch];
    const float *b[kMaxBatch];
    float *dst[kMaxBatch];
    int64_t M[kMaxBatch], K[kMaxBatch];
    int64_t item_off[kMaxBatch + 1];
    int dst_t[kMaxBatch];
    int64_t items;
    int count;
    int *status;
};
static_assert(sizeof(BatchArgs) < 30000, "kernel parameter space");

template <int NP, int VW>
struct Layout {
    static constexpr int TM = 32 * VW;
    static constexpr int A_BYTES = kTK * TM * 4;
    static constexpr int B_BYTES = kTK * NP * 4;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int RED = kConsumerWarps / 2 * NP * TM * 4;   // four warps' partials
    // the next row's loads ahead of the FMAs where the registers allow
    // (nine warps put three on one sub-partition: at most 168 registers)
    static constexpr bool PREFETCH = NP * VW + 2 * (NP + VW) <= 136;
    // as many stages as fit in ~220 KB next to the reduction buffer
    static constexpr int STAGES_FIT = (220 * 1024 - RED - 2048) / STAGE;
    static constexpr int STAGES = STAGES_FIT < kMaxStages ? STAGES_FIT : kMaxStages;
    static_assert(STAGES >= 2, "ring depth");
    static constexpr size_t SMEM = size_t(STAGES) * STAGE + RED + 2 * STAGES * 8 + 16 + 1024;
};

// One k row of a consumer warp: this lane's VW values of src0 and the row of
// src1 (all N values, the same for every lane).
template <int NP, int VW>
struct Row {
    float a[VW];
    float4 b[NP / 4];
};

template <int NP, int VW>
__device__ __forceinline__ void load_row(const float *sa, const float *sb, int row, int lane,
                                         Row<NP, VW> &r) {
    if constexpr (VW == 4) {
        const float4 t = reinterpret_cast<const float4 *>(sa + row * 32 * VW)[lane];
        r.a[0] = t.x;
        r.a[1] = t.y;
        r.a[2] = t.z;
        r.a[3] = t.w;
    } else {
        const float2 t = reinterpret_cast<const float2 *>(sa + row * 32 * VW)[lane];
        r.a[0] = t.x;
        r.a[1] = t.y;
    }
    const float4 *brow = reinterpret_cast<const float4 *>(sb + row * NP);
#pragma unroll
    for (int q = 0; q < NP / 4; ++q) r.b[q] = brow[q];
}

// acc[j][v] holds the sums of n = 2j (low half) and n = 2j + 1 (high half)
// for this lane's m = VW * lane + v.
template <int NP, int VW>
__device__ __forceinline__ void fma_row(const Row<NP, VW> &r, uint64_t (&acc)[NP / 2][VW]) {
#pragma unroll
    for (int v = 0; v < VW; ++v) {
        const uint64_t a2 = ptx::pack2(r.a[v], r.a[v]);
#pragma unroll
        for (int q = 0; q < NP / 4; ++q) {
            acc[2 * q][v] = ptx::fma2(a2, ptx::pack2(r.b[q].x, r.b[q].y), acc[2 * q][v]);
            acc[2 * q + 1][v] = ptx::fma2(a2, ptx::pack2(r.b[q].z, r.b[q].w), acc[2 * q + 1][v]);
        }
    }
}

// A warp's partial in the reduction buffer: rows n of TM floats, this lane's
// VW consecutive m in each.
template <int NP, int VW>
__device__ __forceinline__ void store_partial(float *r, const uint64_t (&acc)[NP / 2][VW]) {
#pragma unroll
    for (int j = 0; j < NP / 2; ++j) {
        float lo[VW], hi[VW];
#pragma unroll
        for (int v = 0; v < VW; ++v) ptx::unpack2(acc[j][v], lo[v], hi[v]);
        float *r0 = r + 2 * j * 32 * VW, *r1 = r0 + 32 * VW;
        if constexpr (VW == 4) {
            *reinterpret_cast<float4 *>(r0) = make_float4(lo[0], lo[1], lo[2], lo[3]);
            *reinterpret_cast<float4 *>(r1) = make_float4(hi[0], hi[1], hi[2], hi[3]);
        } else {
            *reinterpret_cast<float2 *>(r0) = make_float2(lo[0], lo[1]);
            *reinterpret_cast<float2 *>(r1) = make_float2(hi[0], hi[1]);
        }
    }
}

template <int NP, int VW>
__device__ __forceinline__ void add_partial(const float *r, uint64_t (&acc)[NP / 2][VW]) {
#pragma unroll
    for (int j = 0; j < NP / 2; ++j) {
        const float *r0 = r + 2 * j * 32 * VW, *r1 = r0 + 32 * VW;
        if constexpr (VW == 4) {
            const float4 lo = *reinterpret_cast<const float4 *>(r0);
            const float4 hi = *reinterpret_cast<const float4 *>(r1);
            acc[j][0] = ptx::add2(acc[j][0], ptx::pack2(lo.x, hi.x));
            acc[j][1] = ptx::add2(acc[j][1], ptx::pack2(lo.y, hi.y));
            acc[j][2] = ptx::add2(acc[j][2], ptx::pack2(lo.z, hi.z));
            acc[j][3] = ptx::add2(acc[j][3], ptx::pack2(lo.w, hi.w));
        } else {
            const float2 lo = *reinterpret_cast<const float2 *>(r0);
            const float2 hi = *reinterpret_cast<const float2 *>(r1);
            acc[j][0] = ptx::add2(acc[j][0], ptx::pack2(lo.x, hi.x));
            acc[j][1] = ptx::add2(acc[j][1], ptx::pack2(lo.y, hi.y));
        }
    }
}

// What one work item reads and writes: src0 through `map` from row `arow0`
// (k = 0) at m-tile `mt`, src1 rows of NP words from `b`, dst rows of `M`
// floats at `dst`, K rows in `kstages` stages.
struct ItemRef {
    const CUtensorMap *map;
    int64_t arow0, M, K;
    const float *b;
    float *dst;
    int mt, kstages;
    bool dst_t;                   // dst stored transposed: element (m, n) at m * NP + n
};

// The body shared by both kernels: `resolve(item)` gives an item's ItemRef.
// N == NP here (the launchers take this form only for N % 4 == 0).
template <int NP, int VW, class Resolve>
__device__ __forceinline__ void skinny_body(int64_t items, int *status, const Resolve &resolve) {
    using L = Layout<NP, VW>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *red = reinterpret_cast<float *>(smem + L::STAGES * L::STAGE);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::STAGES * L::STAGE + L::RED);
    uint64_t *empty = full + L::STAGES;
    int *abort_flag = reinterpret_cast<int *>(empty + L::STAGES);
    volatile int *abort = abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < L::STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], kConsumerWarps);   // one arrival per warp
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    bool timed_out = false;

    if (warp == kConsumerWarps) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int last_ph[L::STAGES];
            for (int s = 0; s < L::STAGES; ++s) last_ph[s] = -1;
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int64_t item = blockIdx.x; item < items && ok; item += gridDim.x) {
                const ItemRef it = resolve(item);
                if (item == blockIdx.x) ptx::prefetch_tmap(it.map);
                for (int ks = 0; ks < it.kstages; ++ks) {
                    if (!ptx::mbar_wait_bounded(&empty[s], ph ^ 1, abort, true, kWaitNs,
                                                &timed_out)) {
                        ok = false;
                        break;
                    }
                    const int64_t k0 = static_cast<int64_t>(ks) * kTK;
                    const uint32_t bbytes =
                        static_cast<uint32_t>(std::min<int64_t>(kTK, it.K - k0) * NP * 4);
                    uint8_t *st = smem + s * L::STAGE;
                    ptx::mbar_arrive_expect_tx(&full[s], L::A_BYTES + bbytes);
                    ptx::tma_load_2d(st, it.map, &full[s], it.mt * L::TM,
                                     static_cast<int>(it.arow0 + k0));
                    ptx::bulk_load(st + L::A_BYTES, it.b + k0 * NP, bbytes, &full[s]);
                    last_ph[s] = static_cast<int>(ph);
                    if (++s == L::STAGES) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            // copies in flight must land before the CTA's shared memory is released
            for (int i = 0; i < L::STAGES; ++i)
                if (last_ph[i] >= 0)
                    ptx::mbar_wait_bounded(&full[i], static_cast<uint32_t>(last_ph[i]), abort,
                                           false, kWaitNs, &timed_out);
        }
    } else {
        // ---------------- consumers ----------------
        // After a wait runs out the warps keep walking the same items and
        // stages, without waiting or computing, so that all eight still meet
        // at every named barrier.
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
            const ItemRef it = resolve(item);
            uint64_t acc[NP / 2][VW];
#pragma unroll
            for (int j = 0; j < NP / 2; ++j)
#pragma unroll
                for (int v = 0; v < VW; ++v) acc[j][v] = 0;   // +0.0f in both halves
            for (int ks = 0; ks < it.kstages; ++ks) {
                if (ok) {
                    const bool got = ptx::mbar_wait_bounded(&full[s], ph, abort, true, kWaitNs,
                                                            &timed_out);
                    ok = __all_sync(0xffffffffu, got);
                }
                if (ok) {
                    const float *sa = reinterpret_cast<const float *>(smem + s * L::STAGE);
                    const float *sb =
                        reinterpret_cast<const float *>(smem + s * L::STAGE + L::A_BYTES);
                    const int64_t k0 = static_cast<int64_t>(ks) * kTK;
                    const int row0 = warp * kRowsPerWarp;
                    if (k0 + kTK <= it.K) {
                        if constexpr (L::PREFETCH) {
                            // row j + 1's loads go out before row j's FMAs
                            Row<NP, VW> cur, nxt;
                            load_row<NP, VW>(sa, sb, row0, lane, cur);
#pragma unroll
                            for (int j = 0; j < kRowsPerWarp; ++j) {
                                if (j + 1 < kRowsPerWarp)
                                    load_row<NP, VW>(sa, sb, row0 + j + 1, lane, nxt);
                                fma_row<NP, VW>(cur, acc);
                                if (j + 1 < kRowsPerWarp) cur = nxt;
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < kRowsPerWarp; ++j) {
                                Row<NP, VW> cur;
                                load_row<NP, VW>(sa, sb, row0 + j, lane, cur);
                                fma_row<NP, VW>(cur, acc);
                            }
                        }
                    } else {
                        // the last stage of a slice: rows past K belong to the
                        // next slice (src0) or were not copied (src1)
                        for (int j = 0; j < kRowsPerWarp; ++j) {
                            if (k0 + row0 + j < it.K) {
                                Row<NP, VW> cur;
                                load_row<NP, VW>(sa, sb, row0 + j, lane, cur);
                                fma_row<NP, VW>(cur, acc);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&empty[s]);
                }
                if (++s == L::STAGES) {
                    s = 0;
                    ph ^= 1;
                }
            }
            // ---- the warps' partials meet in shared memory (fixed order) ----
            // round 1: warp w + 4 hands its partial to warp w (w < 4)
            const int slot = warp & 3;
            float *mine = red + slot * NP * L::TM + lane * VW;
            if (warp >= 4) store_partial<NP, VW>(mine, acc);
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
            // round 2: warps 0-3 add it and publish the sum in the same slot
            // (each lane rereads and rewrites only its own words), then one
            // thread per output adds the four slots
            if (warp < 4) {
                add_partial<NP, VW>(mine, acc);
                store_partial<NP, VW>(mine, acc);
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
            if (ok) {
                for (int o = threadIdx.x; o < NP * L::TM; o += kConsumers) {
                    const int n = o / L::TM, mm = o % L::TM;
                    float sum = 0.f;
#pragma unroll
                    for (int w = 0; w < 4; ++w) sum += red[(w * NP + n) * L::TM + mm];
                    const int64_t m = static_cast<int64_t>(it.mt) * L::TM + mm;
                    if (m < it.M)
                        it.dst[it.dst_t ? m * NP + n : static_cast<int64_t>(n) * it.M + m] = sum;
                }
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
        }
    }
    if (timed_out) record_status(status, OOP_ERR_DEVICE_TIMEOUT);
}

template <int NP, int VW>
__global__ void __launch_bounds__(kThreads, 1)
    skinny_tma_kernel(const __grid_constant__ CUtensorMap map_a, const TmaArgs p) {
    skinny_body<NP, VW>(p.items, p.status, [&](int64_t item) {
        const int64_t slice = item / p.mtiles;
        const int64_t i2 = slice % p.ne12, i3 = slice / p.ne12;
        ItemRef r;
        r.map = &map_a;
        r.arow0 = (i3 / p.dps3 * p.ne02 + i2 / p.dps2) * p.K;
        r.M = p.M;
        r.K = p.K;
        r.b = p.b + slice * p.K * NP;
        r.dst = p.dst + slice * NP * p.M;
        r.mt = static_cast<int>(item % p.mtiles);
        r.kstages = p.kstages;
        r.dst_t = false;
        return r;
    });
}

// A list of independent single-slice problems in one launch: problem i owns
// items [item_off[i], item_off[i + 1]), one per m-tile, its src0 read through
// its own tensor map (kept in the kernel parameters).
template <int NP, int VW>
__global__ void __launch_bounds__(kThreads, 1)
    skinny_batch_kernel(const __grid_constant__ BatchArgs pb) {
    skinny_body<NP, VW>(pb.items, pb.status, [&](int64_t item) {
        int i = 0;
        while (i + 1 < pb.count && item >= pb.item_off[i + 1]) ++i;
        ItemRef r;
        r.map = &pb.maps[i];
        r.arow0 = 0;
        r.M = pb.M[i];
        r.K = pb.K[i];
        r.b = pb.b[i];
        r.dst = pb.dst[i];
        r.mt = static_cast<int>(item - pb.item_off[i]);
        r.kstages = static_cast<int>((pb.K[i] + kTK - 1) / kTK);
        r.dst_t = pb.dst_t[i] != 0;
        return r;
    });
}

template <int NP, int VW>
cudaError_t launch_tma(const float *a, const float *b, float *dst, const OutProdShape &s,
                       int *status, int sms, cudaStream_t stream) {
    using L = Layout<NP, VW>;
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const int64_t rows = s.K * s.ne02 * s.ne03;
    CUtensorMap map;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(s.M), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(s.M * 4)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(L::TM), kTK};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(a), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    TmaArgs p = {};
    p.b = b;
    p.dst = dst;
    p.status = status;
    p.M = s.M;
    p.K = s.K;
    p.N = s.N;
    p.ne02 = s.ne02;
    p.ne12 = s.ne12;
    p.dps2 = s.dps2;
    p.dps3 = s.dps3;
    p.mtiles = (s.M + L::TM - 1) / L::TM;
    p.items = p.mtiles * s.ne12 * s.ne13;
    p.kstages = static_cast<int>((s.K + kTK - 1) / kTK);
    auto kern = skinny_tma_kernel<NP, VW>;
    static_assert(L::SMEM <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L::SMEM));
    if (e != cudaSuccess) return e;
    const int64_t grid = std::min<int64_t>(p.items, sms);
    kern<<<static_cast<unsigned>(grid), kThreads, L::SMEM, stream>>>(map, p);
    return cudaGetLastError();
}

template <int NP, int VW>
cudaError_t launch_batch_typed(const oop_out_prod_problem *probs, int count, int *status, int sms,
                               cudaStream_t stream) {
    using L = Layout<NP, VW>;
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    BatchArgs pb;
    memset(&pb, 0, sizeof pb);
    int64_t items = 0;
    for (int i = 0; i < count; ++i) {
        const oop_out_prod_problem &q = probs[i];
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(q.M), static_cast<cuuint64_t>(q.K)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(q.M * 4)};
        cuuint32_t box[2] = {static_cast<cuuint32_t>(L::TM), kTK};
        cuuint32_t estr[2] = {1, 1};
        if (enc(&pb.maps[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(q.a), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        pb.b[i] = q.b;
        pb.dst[i] = q.dst;
        pb.M[i] = q.M;
        pb.K[i] = q.K;
        pb.dst_t[i] = q.dst_transposed;
        pb.item_off[i] = items;
        items += (q.M + L::TM - 1) / L::TM;
    }
    pb.item_off[count] = items;
    pb.items = items;
    pb.count = count;
    pb.status = status;
    auto kern = skinny_batch_kernel<NP, VW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L::SMEM));
    if (e != cudaSuccess) return e;
    const int64_t grid = std::min<int64_t>(items, sms);
    kern<<<static_cast<unsigned>(grid), kThreads, L::SMEM, stream>>>(pb);
    return cudaGetLastError();
}

}  // namespace

bool skinny_batch_ok(const oop_out_prod_problem &q, int64_t N) {
    return N % 4 == 0 && N >= 4 && N <= 32 && q.M % 4 == 0 && q.M > 0 && q.K > 0 &&
           q.K < (1LL << 31) && reinterpret_cast<uintptr_t>(q.a) % 16 == 0 &&
           reinterpret_cast<uintptr_t>(q.b) % 16 == 0;
}

int skinny_batch_max() { return kMaxBatch; }

cudaError_t launch_skinny_batch(const oop_out_prod_problem *probs, int count, int64_t N,
                                int *status, cudaStream_t stream) {
    const int sms = device_sm_count();
    if (count < 1 || count > kMaxBatch || sms <= 0) return cudaErrorInvalidValue;
    switch (N) {
    case 4: return launch_batch_typed<4, 4>(probs, count, status, sms, stream);
    case 8: return launch_batch_typed<8, 4>(probs, count, status, sms, stream);
    case 12: return launch_batch_typed<12, 4>(probs, count, status, sms, stream);
    case 16: return launch_batch_typed<16, 4>(probs, count, status, sms, stream);
    case 20: return launch_batch_typed<20, 4>(probs, count, status, sms, stream);
    case 24: return launch_batch_typed<24, 4>(probs, count, status, sms, stream);
    case 28: return launch_batch_typed<28, 2>(probs, count, status, sms, stream);
    case 32: return launch_batch_typed<32, 2>(probs, count, status, sms, stream);
    default: return cudaErrorInvalidValue;
    }
}

// Items of 128 m (four m per lane) up to N = 24, of 64 m above; N = 20 and
// 24 fall back to 64 when 128-wide items would leave fewer than two per SM.
// 0: the persistent form does not apply (fewer than two items per SM).
int64_t skinny_tma_tile_m(const OutProdShape &s, int sms) {
    const int64_t slices = s.ne12 * s.ne13;
    const int64_t need = 2LL * sms;
    if (s.N <= 24 && (s.M + 127) / 128 * slices >= need) return 128;
    if (s.N >= 20 && (s.M + 63) / 64 * slices >= need) return 64;
    return 0;
}

bool skinny_tma_shape_ok(const OutProdShape &s, int sms) {
    return sms > 0 && s.N % 4 == 0 && s.M % 4 == 0 && s.K * s.ne02 * s.ne03 < (1LL << 31) &&
           s.K < (1LL << 31) && skinny_tma_tile_m(s, sms) > 0;
}

bool skinny_tma_ok(const float *a, const float *b, const OutProdShape &s) {
    return reinterpret_cast<uintptr_t>(a) % 16 == 0 && reinterpret_cast<uintptr_t>(b) % 16 == 0 &&
           skinny_tma_shape_ok(s, device_sm_count());
}

cudaError_t launch_skinny_tma(const float *a, const float *b, float *dst, const OutProdShape &s,
                              int *status, cudaStream_t stream) {
    const int sms = device_sm_count();
    const bool wide = skinny_tma_tile_m(s, sms) == 128;
    switch (s.N) {
    case 4: return launch_tma<4, 4>(a, b, dst, s, status, sms, stream);
    case 8: return launch_tma<8, 4>(a, b, dst, s, status, sms, stream);
    case 12: return launch_tma<12, 4>(a, b, dst, s, status, sms, stream);
    case 16: return launch_tma<16, 4>(a, b, dst, s, status, sms, stream);
    case 20:
        return wide ? launch_tma<20, 4>(a, b, dst, s, status, sms, stream)
                    : launch_tma<20, 2>(a, b, dst, s, status, sms, stream);
    case 24:
        return wide ? launch_tma<24, 4>(a, b, dst, s, status, sms, stream)
                    : launch_tma<24, 2>(a, b, dst, s, status, sms, stream);
    case 28: return launch_tma<28, 2>(a, b, dst, s, status, sms, stream);
    case 32: return launch_tma<32, 2>(a, b, dst, s, status, sms, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace oop
