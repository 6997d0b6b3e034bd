// dense_tc.cu -- tensor-core OUT_PROD for sm_103a (tcgen05, 3xTF32).
//
// Per dst slice: D[n][m] = sum_k A[k][m] * B[k][n], A = src0 (f32, or q8_0 /
// q4_0 dequantised in registers), B = the f32 gradient src1.  The gradient can
// reach ~1.5e5, so no operand is ever rounded to a 16-bit format ("metal:
// OUT_PROD multiplies in float staging; a training gradient overflowed half");
// instead each operand is split into two TF32 terms that keep fp32's 8-bit
// exponent: x = hi + lo (+ r, |r| <= 2^-22 |x|), and the product is
// a_hi*b_hi + a_hi*b_lo + a_lo*b_hi (the a_lo*b_lo term is ~2^-22 relative).
//
// Launches per call:
//  1. bsplit: b[slice][k][n] -> bhi, blo [slice][n][Kp] (K-major TF32 words,
//     Kp = K rounded up to 4) in the caller's workspace;
//  2. the tile kernel, one 128 (m) x 128 (n) dst tile per CTA, every head x
//     batch slice in the same grid (grid.y = slice, src0 slice i2/dps2,
//     i3/dps3 -- the broadcast map of "metal: OUT_PROD runs batched,
//     broadcast and narrow shapes on the GPU").
//
// Tile kernel roles (448 threads):
//  warp 0      TMA: raw src0 rows (32 k x one m-tile of f32 words or q8_0 /
//              q4_0 blocks) into a ring, bhi/blo tiles (32 k x 128 n,
//              128-byte swizzle) into the operand stages
//  warp 1      TMEM allocation; one thread issues tcgen05.mma (M128 N128 K8)
//  warps 2-5   src0 producer: raw ring -> dequantise -> split -> the K-major
//              swizzled A images a_hi / a_lo of the operand stage
//  warps 6-13  fold + epilogue: TMEM -> registers -> dst
// When src0's rows are not 16-byte aligned (TMA's rule), the producer loads
// src0 from global memory itself instead of from the ring.
//
// Accumulation.  The tensor core adds each MMA's products into its fp32
// accumulator with an error of up to about one ulp of the accumulator (it
// does not round to nearest), so a long sum dominated by one 1e5-sized
// gradient entry drifts past the 2e-6 * sum|a*b| bound.  Three measures keep
// the error at a few ulps of the result:
//  * the two small cross terms a_lo*b_hi + a_hi*b_lo go to their own
//    accumulator D2, whose magnitude is ~2^-11 of the result, so its
//    accumulation error is negligible; it runs over the whole K;
//  * the big term a_hi*b_hi goes to D1, restarted every `chunk_kb` k-blocks
//    (so at most 4*chunk_kb MMAs accumulate into it);
//  * the fold warps add each finished D1 chunk into a Kahan pair: the sum S
//    lives in TMEM, the compensation C in registers (64 columns per thread).
// TMEM columns: [0,128) D1 buffer 0, [128,256) D1 buffer 1, [256,384) D2,
// [384,512) S; the MMA fills one D1 buffer while the fold drains the other.
//
// Every wait is bounded (1 s of globaltimer); running out records
// OOP_ERR_DEVICE_TIMEOUT, sets a CTA-wide abort flag, drains the copies and
// MMAs already issued, frees TMEM and returns.  Nothing traps.
#include <cudaTypedefs.h>

#include <mutex>

#include "oop_internal.cuh"
#include "tc_ptx.cuh"

namespace oop {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 32;                      // tf32 per 128-byte swizzle row
constexpr int STAGES = 3;
constexpr int THREADS = 448;
constexpr int FOLD_THREADS = 256;
constexpr int A_IMG = BM * BK * 4;          // 16 KB
constexpr int B_IMG = BN * BK * 4;          // 16 KB
constexpr int STAGE_BYTES = 2 * A_IMG + 2 * B_IMG;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_D2 = 2 * BN, COL_S = 3 * BN;
constexpr uint64_t WAIT_NS = 1000000000ull;
constexpr int MAX_RSTAGES = 4;

// Raw src0 staging per type: one TMA box covers 32 k rows of one m-tile.
// Quantised rows: the tile's 4 blocks (136 or 72 bytes) start 0 or 8 bytes
// past a 16-byte boundary, so the box is 8 bytes wider than the blocks.
template <int TYPE>
struct RawA;
template <>
struct RawA<OOP_TYPE_F32> {
    static constexpr int BLOCK = 0;
    static constexpr int BOX_X = BM;                 // f32 elements
    static constexpr int ROW_BYTES = BM * 4;         // bytes per staged k row
    static constexpr int SLOT = ROW_BYTES * BK;      // 16 KB
    static constexpr int RSTAGES = 2;
};
template <>
struct RawA<OOP_TYPE_BF16> {
    static constexpr int BLOCK = 0;
    static constexpr int BOX_X = BM;                 // bf16 elements
    static constexpr int ROW_BYTES = BM * 2;
    static constexpr int SLOT = ROW_BYTES * BK;      // 8 KB
    static constexpr int RSTAGES = 4;
};
template <>
struct RawA<OOP_TYPE_Q8_0> {
    static constexpr int BLOCK = kQ8Bytes;
    static constexpr int BOX_X = 4 * kQ8Bytes + 8;   // 144 bytes
    static constexpr int ROW_BYTES = BOX_X;
    static constexpr int SLOT = 5120;                // 144 * 32 rounded to 1 KB
    static constexpr int RSTAGES = 4;
};
template <>
struct RawA<OOP_TYPE_Q4_0> {
    static constexpr int BLOCK = kQ4Bytes;
    static constexpr int BOX_X = 4 * kQ4Bytes + 8;   // 80 bytes
    static constexpr int ROW_BYTES = BOX_X;
    static constexpr int SLOT = 3072;                // 80 * 32 rounded to 1 KB
    static constexpr int RSTAGES = 4;
};

struct Bars {
    uint64_t bfull[STAGES];       // TMA bytes of operand stage s landed
    uint64_t afull[STAGES];       // the 128 src0-producer threads wrote stage s
    uint64_t empty[STAGES];       // MMAs reading stage s completed
    uint64_t rfull[MAX_RSTAGES];  // raw src0 slot r landed
    uint64_t rempty[MAX_RSTAGES]; // raw src0 slot r consumed by the producer
    uint64_t accf[2];             // D1 buffer b holds a finished chunk
    uint64_t acce[2];             // D1 buffer b was drained by the fold
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
};

template <int TYPE>
constexpr bool elementwise_type() { return TYPE == OOP_TYPE_F32 || TYPE == OOP_TYPE_BF16; }

template <int TYPE>
constexpr size_t smem_bytes() {
    return STAGES * STAGE_BYTES + RawA<TYPE>::RSTAGES * RawA<TYPE>::SLOT + sizeof(Bars) + 1024;
}

struct TcParams {
    const uint8_t *a;
    float *dst;
    int *status;
    int64_t M, K, N, ne02, ne12, dps2, dps3, a_row_bytes;
    int num_kb, chunk_kb, mtiles, ntiles, inject;
    // grouped mode (MUL_MAT_ID_BACK): slices are experts, src1 rows are the
    // routed slots sorted by expert, dst rows are scattered back to slots
    const int *grp_count;         // [E] slots routed to each expert
    const int *grp_offset;        // [E] first sorted slot of each expert
    const int *grp_rows;          // [slots] sorted slot -> dst row
    const int *grp_tiles;         // work list: (expert << 16) | n-tile
    const int *grp_ntiles;        // valid entries in grp_tiles
};

template <int TYPE>
__device__ __forceinline__ float load_a(const uint8_t *row, int64_t m) {
    if constexpr (TYPE == OOP_TYPE_F32) {
        return __ldg(reinterpret_cast<const float *>(row) + m);
    } else if constexpr (TYPE == OOP_TYPE_BF16) {
        return bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short *>(row) + m));
    } else if constexpr (TYPE == OOP_TYPE_Q8_0) {
        const uint8_t *blk = row + (m >> 5) * kQ8Bytes;
        const uint16_t d = __ldg(reinterpret_cast<const unsigned short *>(blk));
        const int8_t q = static_cast<int8_t>(__ldg(blk + 2 + (m & 31)));
        return half_bits_to_float(d) * static_cast<float>(q);
    } else {
        const uint8_t *blk = row + (m >> 5) * kQ4Bytes;
        const uint16_t d = __ldg(reinterpret_cast<const unsigned short *>(blk));
        const int j = static_cast<int>(m & 31);
        const uint8_t byte = __ldg(blk + 2 + (j & 15));
        const int v = j < 16 ? (byte & 0x0f) : (byte >> 4);
        return half_bits_to_float(d) * static_cast<float>(v - 8);
    }
}

// Element r (row of the m-tile) of a staged raw k row.  `off0` is where the
// tile's first block starts inside the staged row.
template <int TYPE>
__device__ __forceinline__ float staged_a(const uint8_t *srow, int r, int off0) {
    if constexpr (TYPE == OOP_TYPE_F32) {
        return reinterpret_cast<const float *>(srow)[r];
    } else if constexpr (TYPE == OOP_TYPE_BF16) {
        return bf16_bits_to_float(reinterpret_cast<const uint16_t *>(srow)[r]);
    } else if constexpr (TYPE == OOP_TYPE_Q8_0) {
        const uint8_t *blk = srow + off0 + (r >> 5) * kQ8Bytes;
        const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
        const int q = static_cast<int8_t>(blk[2 + (r & 31)]);
        return ptx::scaled_small_int(d, q);
    } else {
        const uint8_t *blk = srow + off0 + (r >> 5) * kQ4Bytes;
        const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
        const int j = r & 31;
        const uint8_t byte = blk[2 + (j & 15)];
        const int v = j < 16 ? (byte & 0x0f) : (byte >> 4);
        return ptx::scaled_small_int(d, v - 8);
    }
}

template <int TYPE, bool TMA_A, bool GROUPED>
__global__ void __launch_bounds__(THREADS, 1)
    tc_out_prod_kernel(const __grid_constant__ CUtensorMap map_bhi,
                       const __grid_constant__ CUtensorMap map_blo,
                       const __grid_constant__ CUtensorMap map_a, const TcParams p) {
    using Raw = RawA<TYPE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ring = smem + STAGES * STAGE_BYTES;
    Bars *bars = reinterpret_cast<Bars *>(ring + Raw::RSTAGES * Raw::SLOT);
    volatile int *abort = &bars->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int mt = blockIdx.x % p.mtiles;
    int nt;
    int64_t slice;
    int64_t ncols = p.N;          // valid columns of this tile's slice
    int64_t brow0 = 0;            // grouped: first src1 row of this tile
    if constexpr (GROUPED) {
        const int t = blockIdx.x / p.mtiles;
        if (t >= *p.grp_ntiles) return;              // whole CTA: no work left
        const int packed = p.grp_tiles[t];
        slice = packed >> 16;
        nt = packed & 0xFFFF;
        ncols = p.grp_count[slice];
        brow0 = p.grp_offset[slice] + static_cast<int64_t>(nt) * BN;
    } else {
        nt = blockIdx.x / p.mtiles;
        slice = blockIdx.y;
    }
    const int64_t i2 = slice % p.ne12, i3 = slice / p.ne12;
    const int64_t j2 = i2 / p.dps2, j3 = i3 / p.dps3;
    const int64_t a_row0 = (j3 * p.ne02 + j2) * p.K;     // first src0 row of the slice
    const int nchunks = (p.num_kb + p.chunk_kb - 1) / p.chunk_kb;
    // where this m-tile starts inside a raw row
    int box_x = 0, off0 = 0;
    if constexpr (elementwise_type<TYPE>()) {
        box_x = mt * BM;
    } else {
        const int byte0 = mt * 4 * Raw::BLOCK;
        box_x = byte0 & ~15;
        off0 = byte0 - box_x;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&bars->bfull[s], 1);
            ptx::mbar_init(&bars->afull[s], 128);
            ptx::mbar_init(&bars->empty[s], 1);
        }
        for (int r = 0; r < Raw::RSTAGES; ++r) {
            ptx::mbar_init(&bars->rfull[r], 1);
            ptx::mbar_init(&bars->rempty[r], 128);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&bars->accf[b], 1);
            ptx::mbar_init(&bars->acce[b], FOLD_THREADS);
        }
        ptx::mbar_init(&bars->mma_done, 1);
        bars->abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&map_bhi);
        ptx::prefetch_tmap(&map_blo);
        if constexpr (TMA_A) ptx::prefetch_tmap(&map_a);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&bars->tmem_base, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    bool timed_out = false;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int last_b[STAGES], last_r[MAX_RSTAGES];
            for (int s = 0; s < STAGES; ++s) last_b[s] = -1;
            for (int r = 0; r < MAX_RSTAGES; ++r) last_r[r] = -1;
            for (int kb = 0; kb < p.num_kb; ++kb) {
                if constexpr (TMA_A) {
                    const int r = kb % Raw::RSTAGES;
                    const uint32_t rph = (kb / Raw::RSTAGES) & 1;
                    if (!ptx::mbar_wait_bounded(&bars->rempty[r], rph ^ 1, abort, true, WAIT_NS,
                                                &timed_out))
                        break;
                    ptx::mbar_arrive_expect_tx(&bars->rfull[r],
                                               static_cast<uint32_t>(Raw::ROW_BYTES * BK));
                    ptx::tma_load_2d(ring + r * Raw::SLOT, &map_a, &bars->rfull[r], box_x,
                                     static_cast<int>(a_row0 + static_cast<int64_t>(kb) * BK));
                    last_r[r] = kb;
                }
                const int s = kb % STAGES;
                const uint32_t ph = (kb / STAGES) & 1;
                if (!ptx::mbar_wait_bounded(&bars->empty[s], ph ^ 1, abort, true, WAIT_NS,
                                            &timed_out))
                    break;
                if (p.inject == 1 && kb == 0) continue;   // test hook: drop one stage
                uint8_t *st = smem + s * STAGE_BYTES;
                ptx::mbar_arrive_expect_tx(&bars->bfull[s], 2 * B_IMG);
                if constexpr (GROUPED) {
                    ptx::tma_load_2d(st + 2 * A_IMG, &map_bhi, &bars->bfull[s], kb * BK,
                                     static_cast<int>(brow0));
                    ptx::tma_load_2d(st + 2 * A_IMG + B_IMG, &map_blo, &bars->bfull[s], kb * BK,
                                     static_cast<int>(brow0));
                } else {
                    ptx::tma_load_3d(st + 2 * A_IMG, &map_bhi, &bars->bfull[s], kb * BK,
                                     nt * BN, static_cast<int>(slice));
                    ptx::tma_load_3d(st + 2 * A_IMG + B_IMG, &map_blo, &bars->bfull[s], kb * BK,
                                     nt * BN, static_cast<int>(slice));
                }
                last_b[s] = kb;
            }
            // copies in flight must land before the CTA's smem is released
            for (int s = 0; s < STAGES; ++s)
                if (last_b[s] >= 0)
                    ptx::mbar_wait_bounded(&bars->bfull[s], (last_b[s] / STAGES) & 1, abort,
                                           false, WAIT_NS, &timed_out);
            for (int r = 0; r < Raw::RSTAGES; ++r)
                if (last_r[r] >= 0)
                    ptx::mbar_wait_bounded(&bars->rfull[r], (last_r[r] / Raw::RSTAGES) & 1,
                                           abort, false, WAIT_NS, &timed_out);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_tf32(BM, BN);
            int kb = 0;
            bool ok = true;
            for (int q = 0; q < nchunks && ok; ++q) {
                const int buf = q & 1;
                const uint32_t use = static_cast<uint32_t>(q >> 1);
                if (!ptx::mbar_wait_bounded(&bars->acce[buf], (use & 1) ^ 1, abort, true,
                                            WAIT_NS, &timed_out)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d1 = tmem + static_cast<uint32_t>(buf * BN);
                const uint32_t d2 = tmem + COL_D2;
                const int kb_first = q * p.chunk_kb;
                const int kb_end = min(p.num_kb, kb_first + p.chunk_kb);
                for (; kb < kb_end; ++kb) {
                    const int s = kb % STAGES;
                    const uint32_t ph = (kb / STAGES) & 1;
                    if (!ptx::mbar_wait_bounded(&bars->bfull[s], ph, abort, true, WAIT_NS,
                                                &timed_out) ||
                        !ptx::mbar_wait_bounded(&bars->afull[s], ph, abort, true, WAIT_NS,
                                                &timed_out)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t st = ptx::smem_u32(smem + s * STAGE_BYTES);
                    const uint32_t ahi = st, alo = st + A_IMG;
                    const uint32_t bhi = st + 2 * A_IMG, blo = st + 2 * A_IMG + B_IMG;
#pragma unroll
                    for (int kk = 0; kk < BK / 8; ++kk) {
                        const uint32_t off = kk * 32;   // 8 tf32 along k
                        const uint32_t acc2 = (kb == 0 && kk == 0) ? 0u : 1u;
                        const uint32_t acc1 = (kb == kb_first && kk == 0) ? 0u : 1u;
                        ptx::mma_tf32(d2, ptx::sw128_kmajor_desc(alo + off),
                                      ptx::sw128_kmajor_desc(bhi + off), idesc, acc2);
                        ptx::mma_tf32(d2, ptx::sw128_kmajor_desc(ahi + off),
                                      ptx::sw128_kmajor_desc(blo + off), idesc, 1u);
                        ptx::mma_tf32(d1, ptx::sw128_kmajor_desc(ahi + off),
                                      ptx::sw128_kmajor_desc(bhi + off), idesc, acc1);
                    }
                    ptx::mma_commit(&bars->empty[s]);
                }
                if (!ok) break;
                ptx::mma_commit(&bars->accf[buf]);
            }
            // every MMA issued must finish before TMEM is released
            ptx::mma_commit(&bars->mma_done);
            ptx::mbar_wait_bounded(&bars->mma_done, 0, abort, false, WAIT_NS, &timed_out);
        }
    } else if (warp < 6) {
        // ---------------- src0 producer ----------------
        const int r = (warp - 2) * 32 + lane;              // row of the A image
        const int64_t m = static_cast<int64_t>(mt) * BM + r;
        const bool mok = m < p.M;
        const uint8_t *a_slice = p.a + a_row0 * p.a_row_bytes;
        for (int kb = 0; kb < p.num_kb; ++kb) {
            const int s = kb % STAGES;
            const uint32_t ph = (kb / STAGES) & 1;
            float x[BK];
            const bool kfull = (kb + 1) * BK <= p.K;
            if constexpr (TMA_A) {
                const int rs = kb % Raw::RSTAGES;
                const uint32_t rph = (kb / Raw::RSTAGES) & 1;
                if (!ptx::mbar_wait_bounded(&bars->rfull[rs], rph, abort, true, WAIT_NS,
                                            &timed_out))
                    break;
                const uint8_t *slot = ring + rs * Raw::SLOT;
                // one path per warp: the producer warps never diverge
                if (__all_sync(0xffffffffu, mok) && kfull) {
#pragma unroll
                    for (int j = 0; j < BK; ++j)
                        x[j] = staged_a<TYPE>(slot + j * Raw::ROW_BYTES, r, off0);
                } else {
#pragma unroll
                    for (int j = 0; j < BK; ++j) {
                        const int64_t k = static_cast<int64_t>(kb) * BK + j;
                        const float v = staged_a<TYPE>(slot + j * Raw::ROW_BYTES, r, off0);
                        x[j] = (mok && k < p.K) ? v : 0.f;
                    }
                }
                __syncwarp();
                ptx::mbar_arrive(&bars->rempty[rs]);
            } else {
#pragma unroll
                for (int j = 0; j < BK; ++j) {
                    const int64_t k = static_cast<int64_t>(kb) * BK + j;
                    x[j] = (mok && k < p.K) ? load_a<TYPE>(a_slice + k * p.a_row_bytes, m) : 0.f;
                }
            }
            __syncwarp();
            if (!ptx::mbar_wait_bounded(&bars->empty[s], ph ^ 1, abort, true, WAIT_NS,
                                        &timed_out))
                break;
            __syncwarp();
            uint8_t *ahi = smem + s * STAGE_BYTES;
            uint8_t *alo = ahi + A_IMG;
#pragma unroll
            for (int c = 0; c < BK / 4; ++c) {
                uint32_t h[4], l[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if constexpr (TYPE == OOP_TYPE_F32) {
                        ptx::split_tf32(x[4 * c + e], h[e], l[e]);
                    } else {
                        // d*q has at most 18 significant bits and a bf16 value
                        // 8: x - hi is already a TF32 value (zero for bf16),
                        // no second rounding needed
                        h[e] = ptx::tf32_round_bits(__float_as_uint(x[4 * c + e]));
                        l[e] = __float_as_uint(x[4 * c + e] - __uint_as_float(h[e]));
                    }
                }
                const int off = r * 128 + ((c ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(ahi + off) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4 *>(alo + off) = make_uint4(l[0], l[1], l[2], l[3]);
            }
            __syncwarp();
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&bars->afull[s]);
        }
    } else {
        // ---------------- fold + epilogue ----------------
        const int quad = warp & 3;                          // TMEM lanes 32*quad ..
        const int half = (warp - 6) >> 2;                   // columns 64*half ..
        const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
        const uint32_t col0 = static_cast<uint32_t>(64 * half);
        const int64_t m = static_cast<int64_t>(mt) * BM + 32 * quad + lane;
        float *dst = GROUPED ? p.dst : p.dst + slice * p.N * p.M;
        const int64_t tile_cols = ncols - static_cast<int64_t>(nt) * BN;   // valid columns here
        uint64_t cmp[32];                                   // Kahan compensations, in pairs
#pragma unroll
        for (int j = 0; j < 32; ++j) cmp[j] = 0;
        for (int q = 0; q < nchunks; ++q) {
            const int buf = q & 1;
            const uint32_t use = static_cast<uint32_t>(q >> 1);
            if (!ptx::mbar_wait_bounded(&bars->accf[buf], use & 1, abort, true, WAIT_NS,
                                        &timed_out))
                break;
            ptx::tc_fence_after();
            const bool first = q == 0, last = q == nchunks - 1;
#pragma unroll
            for (int pc = 0; pc < 4; ++pc) {
                const uint32_t col = col0 + pc * 16;
                // tcgen05.ld/st are warp-collective (.sync.aligned): the lanes
                // must be converged after the divergent stores of the last piece
                __syncwarp();
                uint32_t xv[16], sv[16];
                if (first)
                    ptx::tmem_ld16_wait(tmem + lane_off + buf * BN + col, xv);
                else
                    ptx::tmem_ld16x2_wait(tmem + lane_off + buf * BN + col, xv,
                                          tmem + lane_off + COL_S + col, sv);
                if (!first) {
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        // Kahan on two columns at once: the running sum is S - C
                        uint64_t &c2 = cmp[pc * 8 + j / 2];
                        const uint64_t s2 = ptx::pack2(__uint_as_float(sv[j]), __uint_as_float(sv[j + 1]));
                        const uint64_t x2 = ptx::pack2(__uint_as_float(xv[j]), __uint_as_float(xv[j + 1]));
                        const uint64_t y2 = ptx::sub2(x2, c2);
                        const uint64_t t2 = ptx::add2(s2, y2);
                        c2 = ptx::sub2(ptx::sub2(t2, s2), y2);
                        float t0, t1;
                        ptx::unpack2(t2, t0, t1);
                        xv[j] = __float_as_uint(t0);
                        xv[j + 1] = __float_as_uint(t1);
                    }
                }
                // xv now holds S for these 16 columns
                if (last) {
                    uint32_t (&dv)[16] = sv;                // D2, the cross terms
                    __syncwarp();
                    ptx::tmem_ld16_wait(tmem + lane_off + COL_D2 + col, dv);
                    if (m < p.M) {
#pragma unroll
                        for (int j = 0; j < 16; j += 2) {
                            float c0, c1;
                            ptx::unpack2(cmp[pc * 8 + j / 2], c0, c1);
                            const int64_t jc = static_cast<int64_t>(col) + j;   // column in tile
                            int64_t r0 = -1, r1 = -1;                            // dst rows
                            if constexpr (GROUPED) {
                                if (jc < tile_cols) r0 = p.grp_rows[brow0 + jc];
                                if (jc + 1 < tile_cols) r1 = p.grp_rows[brow0 + jc + 1];
                            } else {
                                if (jc < tile_cols) r0 = static_cast<int64_t>(nt) * BN + jc;
                                if (jc + 1 < tile_cols) r1 = static_cast<int64_t>(nt) * BN + jc + 1;
                            }
                            if (r0 >= 0)
                                dst[r0 * p.M + m] = __uint_as_float(xv[j]) + (__uint_as_float(dv[j]) - c0);
                            if (r1 >= 0)
                                dst[r1 * p.M + m] =
                                    __uint_as_float(xv[j + 1]) + (__uint_as_float(dv[j + 1]) - c1);
                        }
                    }
                } else {
                    ptx::tmem_st16(tmem + lane_off + COL_S + col, xv);
                }
            }
            __syncwarp();
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bars->acce[buf]);
        }
    }

    if (timed_out) record_status(p.status, OOP_ERR_DEVICE_TIMEOUT);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// b[slice][k][n] (n fastest) -> bhi, blo [slice][n][Kp] (k fastest), TF32
// split, zero padding for k in [K, Kp).
__global__ void __launch_bounds__(256) bsplit_kernel(const float *__restrict__ b,
                                                     uint32_t *__restrict__ bhi,
                                                     uint32_t *__restrict__ blo, int64_t K,
                                                     int64_t N, int64_t Kp) {
    __shared__ float tile[32][33];
    const int64_t slice = blockIdx.z;
    const int64_t k0 = static_cast<int64_t>(blockIdx.x) * 32;
    const int64_t n0 = static_cast<int64_t>(blockIdx.y) * 32;
    const float *bs = b + slice * K * N;
    const int tx = threadIdx.x, ty = threadIdx.y;
#pragma unroll
    for (int i = ty; i < 32; i += 8) {
        const int64_t k = k0 + i, n = n0 + tx;
        tile[i][tx] = (k < K && n < N) ? __ldg(bs + k * N + n) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int i = ty; i < 32; i += 8) {
        const int64_t n = n0 + i, k = k0 + tx;
        if (n < N && k < Kp) {
            uint32_t h, l;
            ptx::split_tf32(tile[tx][i], h, l);
            const int64_t o = (slice * N + n) * Kp + k;
            bhi[o] = h;
            blo[o] = l;
        }
    }
}

// ---- MUL_MAT_ID_BACK as a grouped product ----------------------------------
// Routing, one CTA: count the slots of each expert, lay them out sorted by
// expert, build the (expert, n-tile) work list.  A slot with an id outside
// [0, E) gets a zero dx row and OOP_ERR_BAD_ID in the status word.  The order
// of slots inside an expert does not matter: every dx row is computed alone.
struct RouteWs {
    int *count, *offset, *ntiles, *tiles, *rows;
};

__global__ void __launch_bounds__(1024) mmid_route_kernel(const int32_t *__restrict__ ids,
                                                          int64_t nslot, int E, int64_t Kw,
                                                          float *dx, RouteWs w, int *status) {
    extern __shared__ int sh[];                   // [E] counts, then [E] cursors
    int *cnt = sh, *cur = sh + E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (int64_t s = threadIdx.x; s < nslot; s += blockDim.x) {
        const int e = ids[s];
        if (e >= 0 && e < E) {
            atomicAdd(&cnt[e], 1);
        } else {
            record_status(status, OOP_ERR_BAD_ID);
            for (int64_t k = 0; k < Kw; ++k) dx[s * Kw + k] = 0.f;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0, nt = 0;
        for (int e = 0; e < E; ++e) {
            w.count[e] = cnt[e];
            w.offset[e] = acc;
            cur[e] = acc;
            for (int t = 0; t * BN < cnt[e]; ++t) w.tiles[nt++] = (e << 16) | t;
            acc += cnt[e];
        }
        *w.ntiles = nt;
    }
    __syncthreads();
    for (int64_t s = threadIdx.x; s < nslot; s += blockDim.x) {
        const int e = ids[s];
        if (e >= 0 && e < E) w.rows[atomicAdd(&cur[e], 1)] = static_cast<int>(s);
    }
}

// Sorted slot j: g[rows[j]][0..R) -> ghi, glo [j][Kp], TF32 split, zero
// padding for r in [R, Kp).  Rows past the routed total are left alone: the
// tile kernel never stores the columns they feed.
__global__ void __launch_bounds__(256) mmid_gsplit_kernel(const float *__restrict__ g,
                                                          const int *__restrict__ rows,
                                                          const int *__restrict__ count, int E,
                                                          uint32_t *__restrict__ ghi,
                                                          uint32_t *__restrict__ glo, int64_t R,
                                                          int64_t Kp) {
    const int64_t j = blockIdx.x;
    __shared__ int total;
    if (threadIdx.x == 0) {
        int t = 0;
        for (int e = 0; e < E; ++e) t += count[e];
        total = t;
    }
    __syncthreads();
    if (j >= total) return;
    const float *src = g + static_cast<int64_t>(rows[j]) * R;
    for (int64_t r = threadIdx.x; r < Kp; r += blockDim.x) {
        uint32_t h = 0, l = 0;
        if (r < R) ptx::split_tf32(__ldg(src + r), h, l);
        ghi[j * Kp + r] = h;
        glo[j * Kp + r] = l;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// bhi / blo: [slices][N][Kp] words, boxes of 32 k x 128 n, 128-byte swizzle.
bool make_b_map(CUtensorMap *map, void *base, int64_t Kp, int64_t N, int64_t slices) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(Kp), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(slices)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(Kp * 4),
                             static_cast<cuuint64_t>(N * Kp * 4)};
    cuuint32_t box[3] = {BK, BN, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// grouped src1: [rows][Kp] words, boxes of 32 k x 128 rows, 128-byte swizzle.
bool make_b_map_2d(CUtensorMap *map, void *base, int64_t Kp, int64_t rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(Kp), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(Kp * 4)};
    cuuint32_t box[2] = {BK, BN};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// raw src0: rows of `a_row_bytes` (all slices stacked), boxes of 32 rows.
template <int TYPE>
bool make_a_map(CUtensorMap *map, const void *base, const OutProdShape &s) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int64_t rows = s.K * s.ne02 * s.ne03;
    cuuint32_t box[2] = {static_cast<cuuint32_t>(RawA<TYPE>::BOX_X), BK};
    cuuint32_t estr[2] = {1, 1};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(s.a_row_bytes)};
    if constexpr (elementwise_type<TYPE>()) {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(s.M), static_cast<cuuint64_t>(rows)};
        const CUtensorMapDataType dt = TYPE == OOP_TYPE_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                             : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        return fn(map, dt, 2, const_cast<void *>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    } else {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(s.a_row_bytes),
                              static_cast<cuuint64_t>(rows)};
        return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
}

int64_t padded_k(int64_t K) { return (K + 3) / 4 * 4; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int g_inject = 0;
thread_local cudaEvent_t g_ev_before = nullptr, g_ev_after = nullptr;
#ifndef OOP_TC_CHUNK_KB
#define OOP_TC_CHUNK_KB 2
#endif
int g_chunk_kb = OOP_TC_CHUNK_KB;      // k-blocks (of 32) per D1 accumulation

template <int TYPE, bool GROUPED>
cudaError_t launch_typed(const void *a, const OutProdShape &s, const CUtensorMap &mhi,
                         const CUtensorMap &mlo, const TcParams &p, int64_t grid_x,
                         int64_t slices, cudaStream_t stream) {
    // TMA needs a 16-byte aligned base and row stride, and rows that fit int32.
    const bool tma_a = reinterpret_cast<uintptr_t>(a) % 16 == 0 && s.a_row_bytes % 16 == 0 &&
                       s.K * s.ne02 * s.ne03 < (1LL << 31);
    CUtensorMap ma;
    if (tma_a) {
        if (!make_a_map<TYPE>(&ma, a, s)) return cudaErrorInvalidValue;
    } else {
        ma = mhi;   // unused by the kernel
    }
    constexpr size_t smem = smem_bytes<TYPE>();
    static_assert(smem <= 232448, "shared memory budget");
    auto run = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        cudaEvent_t before = g_ev_before, after = g_ev_after;
        g_ev_before = g_ev_after = nullptr;
        if (before && (e = cudaEventRecord(before, stream)) != cudaSuccess) return e;
        kern<<<dim3(static_cast<unsigned>(grid_x), static_cast<unsigned>(slices)), THREADS, smem,
               stream>>>(mhi, mlo, ma, p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (after && (e = cudaEventRecord(after, stream)) != cudaSuccess) return e;
        return cudaSuccess;
    };
    return tma_a ? run(tc_out_prod_kernel<TYPE, true, GROUPED>)
                 : run(tc_out_prod_kernel<TYPE, false, GROUPED>);
}

}  // namespace

void tc_set_inject(int v) { g_inject = v; }
void tc_set_profile_events(cudaEvent_t before, cudaEvent_t after) {
    g_ev_before = before;
    g_ev_after = after;
}

size_t tc_workspace_bytes(const OutProdShape &s) {
    const size_t one = align256(static_cast<size_t>(s.ne12 * s.ne13) *
                                static_cast<size_t>(s.N) * static_cast<size_t>(padded_k(s.K)) * 4);
    return 2 * one;
}

cudaError_t launch_dense_tc(const void *a, const float *b, float *dst, const OutProdShape &s,
                            void *workspace, int *status, cudaStream_t stream) {
    const int64_t slices = s.ne12 * s.ne13;
    const int64_t Kp = padded_k(s.K);
    const size_t one = tc_workspace_bytes(s) / 2;
    uint32_t *bhi = static_cast<uint32_t *>(workspace);
    uint32_t *blo = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(workspace) + one);

    const int64_t gk = (Kp + 31) / 32, gn = (s.N + 31) / 32;
    if (gk > 0x7fffffffLL || gn > 65535 || slices > 65535) return cudaErrorInvalidConfiguration;
    bsplit_kernel<<<dim3(static_cast<unsigned>(gk), static_cast<unsigned>(gn),
                         static_cast<unsigned>(slices)),
                    dim3(32, 8), 0, stream>>>(b, bhi, blo, s.K, s.N, Kp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    CUtensorMap mhi, mlo;
    if (!make_b_map(&mhi, bhi, Kp, s.N, slices) || !make_b_map(&mlo, blo, Kp, s.N, slices))
        return cudaErrorInvalidValue;

    TcParams p = {};
    p.a = static_cast<const uint8_t *>(a);
    p.dst = dst;
    p.status = status;
    p.M = s.M;
    p.K = s.K;
    p.N = s.N;
    p.ne02 = s.ne02;
    p.ne12 = s.ne12;
    p.dps2 = s.dps2;
    p.dps3 = s.dps3;
    p.a_row_bytes = s.a_row_bytes;
    const int64_t mtiles = (s.M + BM - 1) / BM, ntiles = (s.N + BN - 1) / BN;
    if (mtiles * ntiles > 0x7fffffffLL || (s.K + BK - 1) / BK > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    p.num_kb = static_cast<int>((s.K + BK - 1) / BK);
    p.chunk_kb = g_chunk_kb;
    p.mtiles = static_cast<int>(mtiles);
    p.ntiles = static_cast<int>(ntiles);
    p.inject = g_inject;
    g_inject = 0;

    switch (s.a_type) {
    case OOP_TYPE_F32:
        return launch_typed<OOP_TYPE_F32, false>(a, s, mhi, mlo, p, mtiles * ntiles, slices, stream);
    case OOP_TYPE_Q8_0:
        return launch_typed<OOP_TYPE_Q8_0, false>(a, s, mhi, mlo, p, mtiles * ntiles, slices, stream);
    case OOP_TYPE_Q4_0:
        return launch_typed<OOP_TYPE_Q4_0, false>(a, s, mhi, mlo, p, mtiles * ntiles, slices, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

// ---- MUL_MAT_ID_BACK launcher ------------------------------------------------

namespace {

struct MmidPlan {
    int64_t nslot, Kp, max_tiles, mtiles;
    size_t off_count, off_offset, off_ntiles, off_tiles, off_rows, off_ghi, off_glo, total;
};

MmidPlan plan_mmid(const MmidShape &s) {
    MmidPlan t = {};
    t.nslot = s.n_used * s.n_tok;
    t.Kp = padded_k(s.N);
    t.max_tiles = (t.nslot + BN - 1) / BN + s.E;
    t.mtiles = (s.K + BM - 1) / BM;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += align256(bytes);
        return at;
    };
    t.off_count = take(sizeof(int) * static_cast<size_t>(s.E));
    t.off_offset = take(sizeof(int) * static_cast<size_t>(s.E));
    t.off_ntiles = take(sizeof(int));
    t.off_tiles = take(sizeof(int) * static_cast<size_t>(t.max_tiles));
    t.off_rows = take(sizeof(int) * static_cast<size_t>(t.nslot));
    t.off_ghi = take(4 * static_cast<size_t>(t.nslot) * static_cast<size_t>(t.Kp));
    t.off_glo = take(4 * static_cast<size_t>(t.nslot) * static_cast<size_t>(t.Kp));
    t.total = o;
    return t;
}

}  // namespace

size_t tc_mmid_workspace_bytes(const MmidShape &s) { return plan_mmid(s).total; }

cudaError_t launch_mmid_tc(const void *W, const int32_t *ids, const float *g, float *dx,
                           const MmidShape &s, void *workspace, int *status,
                           cudaStream_t stream) {
    const MmidPlan t = plan_mmid(s);
    if (s.E > 32767 || s.E < 1 || t.nslot > 0x7fffffffLL || t.max_tiles * t.mtiles > 0x7fffffffLL ||
        s.K * s.N * s.E >= (1LL << 40))
        return cudaErrorInvalidConfiguration;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    RouteWs rw;
    rw.count = reinterpret_cast<int *>(ws + t.off_count);
    rw.offset = reinterpret_cast<int *>(ws + t.off_offset);
    rw.ntiles = reinterpret_cast<int *>(ws + t.off_ntiles);
    rw.tiles = reinterpret_cast<int *>(ws + t.off_tiles);
    rw.rows = reinterpret_cast<int *>(ws + t.off_rows);
    uint32_t *ghi = reinterpret_cast<uint32_t *>(ws + t.off_ghi);
    uint32_t *glo = reinterpret_cast<uint32_t *>(ws + t.off_glo);

    const size_t route_smem = 2 * sizeof(int) * static_cast<size_t>(s.E);
    if (route_smem > 48 * 1024) return cudaErrorInvalidConfiguration;
    mmid_route_kernel<<<1, 1024, route_smem, stream>>>(ids, t.nslot, static_cast<int>(s.E), s.K,
                                                        dx, rw, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    mmid_gsplit_kernel<<<static_cast<unsigned>(t.nslot), 256, 0, stream>>>(
        g, rw.rows, rw.count, static_cast<int>(s.E), ghi, glo, s.N, t.Kp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    CUtensorMap mhi, mlo;
    if (!make_b_map_2d(&mhi, ghi, t.Kp, t.nslot) || !make_b_map_2d(&mlo, glo, t.Kp, t.nslot))
        return cudaErrorInvalidValue;

    // W as src0: slice e has rows r (K = N of W) of K_w elements (M)
    OutProdShape os = {};
    os.M = s.K;
    os.K = s.N;
    os.N = t.nslot;
    os.ne02 = s.E;
    os.ne03 = 1;
    os.ne12 = s.E;
    os.ne13 = 1;
    os.dps2 = 1;
    os.dps3 = 1;
    os.a_type = s.w_type;
    os.a_row_bytes = s.K * (s.w_type == OOP_TYPE_F32 ? 4 : 2);

    TcParams p = {};
    p.a = static_cast<const uint8_t *>(W);
    p.dst = dx;
    p.status = status;
    p.M = os.M;
    p.K = os.K;
    p.N = os.N;
    p.ne02 = os.ne02;
    p.ne12 = os.ne12;
    p.dps2 = 1;
    p.dps3 = 1;
    p.a_row_bytes = os.a_row_bytes;
    p.num_kb = static_cast<int>((os.K + BK - 1) / BK);
    p.chunk_kb = g_chunk_kb;
    p.mtiles = static_cast<int>(t.mtiles);
    p.ntiles = 0;
    p.inject = 0;
    p.grp_count = rw.count;
    p.grp_offset = rw.offset;
    p.grp_rows = rw.rows;
    p.grp_tiles = rw.tiles;
    p.grp_ntiles = rw.ntiles;
    const int64_t grid_x = t.mtiles * t.max_tiles;
    if (s.w_type == OOP_TYPE_F32)
        return launch_typed<OOP_TYPE_F32, true>(W, os, mhi, mlo, p, grid_x, 1, stream);
    if (s.w_type == OOP_TYPE_BF16)
        return launch_typed<OOP_TYPE_BF16, true>(W, os, mhi, mlo, p, grid_x, 1, stream);
    return cudaErrorInvalidValue;
}

}  // namespace oop
