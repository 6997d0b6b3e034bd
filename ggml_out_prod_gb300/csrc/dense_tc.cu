// dense_tc.cu -- tensor-core OUT_PROD for sm_103a (tcgen05, 3xTF32).
//
// Per dst slice: D[n][m] = sum_k A[k][m] * B[k][n], A = src0 (f32, bf16, or
// q8_0 / q4_0 dequantised in registers), B = the f32 gradient src1.  The
// gradient can reach ~1.5e5, so no operand is ever rounded to a 16-bit format
// ("metal: OUT_PROD multiplies in float staging; a training gradient
// overflowed half"); instead each operand is split into two TF32 terms that
// keep fp32's 8-bit exponent: x = hi + lo (+ r, |r| <= 2^-22 |x|), and the
// product is a_hi*b_hi + a_hi*b_lo + a_lo*b_hi (a_lo*b_lo is ~2^-22 relative;
// for bf16 src0 a_lo is zero and its product is skipped).
//
// Launches per call:
//  1. bsplit: b[slice][k][n] -> bhi, blo [slice][n][Kp] (K-major TF32 words,
//     Kp = K rounded up to 4) in the caller's workspace;
//  2. the tile kernel over 128 (m) x 128 (n) dst tiles of every head x batch
//     slice in one grid (src0 slice i2/dps2, i3/dps3 -- the broadcast map of
//     "metal: OUT_PROD runs batched, broadcast and narrow shapes on the GPU");
//  3. (stream-K schedule only) the fix-up that adds the k-partials of tiles
//     shared by two or more CTAs.
//
// Work is a list of (tile, k-block) iterations, tile-major.  Data-parallel
// schedule: CTA c takes the num_kb iterations of tile c.  Stream-K schedule:
// one CTA per SM; the full waves of tiles are taken whole, round-robin (so the
// CTAs run in step along k and share the src0 and src1 rows they read in L2),
// and the iterations of the last, partial wave's tiles are split evenly, CTA
// c taking [I*c/G, I*(c+1)/G) of them, so that wave is not left a tenth full;
// a tile split between CTAs is written as fp32 partials (at most two per CTA:
// its first and last tile of the split range) and summed in k order by the
// fix-up.  Both are deterministic.
//
// Tile kernel roles (640 threads = 20 warps = 5 warpgroups, launched at 96
// registers a thread, which one SM sub-partition holds for its five warps;
// then traded between warpgroups with setmaxnreg):
//  warpgroup 0 (48 registers)
//    warp 0    TMA: raw src0 rows (32 k x one m-tile of the src0 type) into a
//              ring, bhi/blo tiles (32 k x 128 n, 128-byte swizzle) into the
//              B stages
//    warp 1    TMEM allocation; the MMA loop (M128 N128 K8, A from tensor
//              memory, B from shared memory), one elected lane issuing
//    warps 2-3 idle
//  warpgroups 1-2 (72 registers): src0 producer, thread = row of the m-tile
//              = TMEM lane, two warps per lane quarter each taking 16 of the
//              block's 32 k: raw ring -> dequantise -> split -> a_hi / a_lo
//              columns of an A stage in tensor memory (tcgen05.st)
//  warpgroups 3-4 (144 registers): fold + epilogue, TMEM -> registers -> dst
// When src0's rows are not 16-byte aligned (TMA's rule), the producer loads
// src0 from global memory itself instead of from the ring.
//
// Accumulation.  The tensor core adds each MMA's products into its fp32
// accumulator with an error of up to about one ulp of the accumulator (it
// does not round to nearest), so a long sum dominated by one 1e5-sized
// gradient entry drifts past the 2e-6 * sum|a*b| bound.  So:
//  * the two small cross terms a_lo*b_hi + a_hi*b_lo go to their own
//    accumulator D2, whose magnitude is ~2^-11 of the result, so its
//    accumulation error is negligible; it runs over a CTA's whole segment
//    of a tile (all of K in the data-parallel schedule);
//  * the big term a_hi*b_hi goes to D1, restarted every CHUNK_KB k-blocks
//    (so at most 8 MMAs accumulate into it);
//  * the fold warps add each finished D1 chunk into a Kahan pair kept in
//    registers: each fold thread owns one row's 64 columns, their sums S and
//    their compensations C (as bfloat16 pairs).
// TMEM columns: [0,128) D1 buffer 0, [128,256) D1 buffer 1, [256,384) D2,
// [384,448) and [448,512) the two A stages (a_hi in the first 32 columns,
// a_lo in the next 32).  The MMA fills one D1 buffer while the fold drains
// the other.  With S out of tensor memory the tile is 128 columns wide: every
// producer instruction (dequantise, split) and every B byte feeds a third more
// MMA work than at 96, the widest tile with S in tensor memory as well.
//
// Every wait is bounded (1 s of globaltimer); running out records
// OOP_ERR_DEVICE_TIMEOUT, sets a CTA-wide abort flag, drains the copies and
// MMAs already issued, frees TMEM and returns.  Nothing traps.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "oop_internal.cuh"
#include "quant.cuh"
#include "tc_ptx.cuh"

namespace oop {
namespace {

constexpr int BM = 128;
constexpr int BN = kTcTileN;                 // 128
static_assert(BN == 128, "the fold's layout and the TMEM map assume 128 columns");
constexpr int BK = 32;                      // tf32 per 128-byte swizzle row
constexpr int CHUNK_KB = 2;                 // k-blocks per D1 chunk
constexpr int MAX_BSTAGES = 6;              // bhi + blo stages in shared memory
constexpr int A_STAGES = 2;                 // a_hi + a_lo stages in tensor memory
constexpr int THREADS = 640;                // 20 warps = 5 warpgroups
constexpr int MAX_REGS = 96;                // at launch: 5 warps x 32 lanes x 96 fill one SMSP
// Warp roles: warpgroup 0 = TMA (warp 0), MMA (warp 1) and two idle warps;
// warpgroups 1-2 the src0 producer; warpgroups 3-4 the fold.  Once set up,
// the warpgroups trade registers (setmaxnreg): 48 for warpgroup 0, 72 for the
// producer, 144 for the fold, which keeps its 64 running sums and their
// compensations in registers.  The split uses exactly what the block was
// launched with, and each sub-partition's share fits its register file.
constexpr int WARP_PROD0 = 4, WARP_FOLD0 = 12;
constexpr int REGS_CTRL = 48, REGS_PROD = 72, REGS_FOLD = 144;
// a producer that addresses row groups (its rows' offsets differ) gets 8 more
constexpr int REGS_PROD_RG = 80, REGS_FOLD_RG = 136;
static_assert(4 * REGS_CTRL + 8 * REGS_PROD_RG + 8 * REGS_FOLD_RG == THREADS / 32 * MAX_REGS,
              "register split must equal the launch allocation");
static_assert(4 * REGS_CTRL + 8 * REGS_PROD + 8 * REGS_FOLD == THREADS / 32 * MAX_REGS,
              "register split must equal the launch allocation");
static_assert(REGS_CTRL + 2 * REGS_PROD + 2 * REGS_FOLD <= 512, "registers per sub-partition");
constexpr int PRODUCER_THREADS = 256;
constexpr int KH = BK / 2;                  // k per producer thread and block
constexpr int FOLD_THREADS = 256;
constexpr int FOLD_COLS = BN / 2;           // columns per fold thread
constexpr int B_IMG = BN * BK * 4;          // 16 KB
constexpr int STAGE_BYTES = 2 * B_IMG;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_D2 = 2 * BN;
constexpr uint32_t COL_A = 384;
constexpr uint32_t A_COLS = 2 * BK;         // a_hi then a_lo, one column per k
static_assert(3 * BN <= COL_A && COL_A + A_STAGES * A_COLS == TMEM_COLS, "tensor memory map");
constexpr size_t SMEM_LIMIT = 232448;       // dynamic shared memory per CTA
static_assert(BN % 16 == 0 && FOLD_COLS % 16 == 0, "MMA N and fold pieces");
constexpr uint64_t WAIT_NS = 1000000000ull;
constexpr int MAX_RSTAGES = 4;

// Raw src0 staging per type: one TMA box covers 32 k rows of one m-tile.
// Plain types (f32, f16, bf16): the tile's 128 elements of each row.  Blocks
// of 32: the tile's four blocks; blocks of 256 (K-quants): the whole
// super-block that the tile is one half of (its scales sit at the block's
// start).  Those bytes start `off0` past a 16-byte boundary (TMA's rule), so
// the box reaches back to the boundary and is as much wider as the largest
// such offset needs.
constexpr int gcd16(int x) { return (x % 16 == 0) ? 16 : (x % 8 == 0) ? 8 : (x % 4 == 0) ? 4 : (x % 2 == 0) ? 2 : 1; }

// A staged row's bytes: at least `need`, a multiple of 16, and such that
// `rows_per_box` of them fill a multiple of 128 bytes (where each box lands).
constexpr int staged_row_bytes(int need, int rows_per_box) {
    int b = (need + 15) / 16 * 16;
    while ((b * rows_per_box) % 128 != 0) b += 16;
    return b;
}

template <int TYPE>
struct RawA {
    using F = QFormat<TYPE>;
    static constexpr bool PLAIN = F::QK == 1;
    // Rows whose byte length is not a multiple of 16 cannot be a 2-D TMA
    // map's rows; groups of 16 / gcd(row bytes, 16) of them are, at most RG
    // (RG * BYTES is a multiple of 16), so the map's rows are groups of rows
    // and one k-block takes one box per member of a group, box r holding
    // member r of each group.  Used by the block types of the cooperative
    // decode (the q8_0 / q4_0 path stages single rows).
    static constexpr int RG = (PLAIN || TYPE == OOP_TYPE_Q8_0 || TYPE == OOP_TYPE_Q4_0)
                                  ? 1 : 16 / gcd16(F::BYTES);
    static_assert(BK % RG == 0, "a k-block holds whole row groups");
    // the bytes of a row one m-tile needs, and how far past a 16-byte
    // boundary they may start: a multiple of the tile's span in one row, or,
    // for the row-group types, of one block (where a group's member rows start)
    static constexpr int SPAN = PLAIN ? BM * F::BYTES : (F::QK == 32 ? 4 * F::BYTES : F::BYTES);
    static constexpr int MAXOFF = PLAIN ? 0 : 16 - gcd16(RG > 1 ? F::BYTES : SPAN);
    static constexpr int ROW_BYTES = staged_row_bytes(SPAN + MAXOFF, BK / RG);  // per staged k row
    static constexpr int BOX_X = PLAIN ? BM : ROW_BYTES;              // in map elements
    static constexpr int SLOT = (ROW_BYTES * BK + 1023) / 1024 * 1024;
    static constexpr int RSTAGES = TYPE == OOP_TYPE_F32 ? 2 : 4;   // f32: room for 3 B stages
};

// Byte offset, in a src0 row, of the first byte m-tile `mt` needs.
template <int TYPE>
__host__ __device__ __forceinline__ int64_t raw_tile_byte0(int64_t mt) {
    using F = QFormat<TYPE>;
    if constexpr (F::QK == 1) return mt * BM * F::BYTES;
    else if constexpr (F::QK == 32) return mt * 4 * F::BYTES;
    else return (mt >> 1) * F::BYTES;
}

struct Bars {
    // Iteration g (one k-block of one tile) uses ring slot g % RSTAGES, B
    // stage g % b_stages and A stage g % A_STAGES.
    uint64_t rfull[MAX_RSTAGES];  // every TMA copy of the iteration landed (raw src0, B)
    uint64_t rempty[MAX_RSTAGES]; // the producers are done with ring slot r
    uint64_t afull[A_STAGES];     // the producers wrote A stage s (and saw its B land)
    uint64_t bempty[MAX_BSTAGES]; // the iteration's MMAs completed: its B stage and
                                  // its A stage are free
    uint64_t accf[2];             // D1 buffer b holds a finished chunk
    uint64_t acce[2];             // D1 buffer b was drained by the fold
    uint64_t d2free;              // the fold read D2 at the end of a segment
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
};

template <int TYPE>
constexpr bool elementwise_type() { return is_plain_type<TYPE>(); }

// The tile kernel's modes: plain OUT_PROD (every head x batch slice in one
// grid), grouped (MUL_MAT_ID_BACK: slices are experts, src1 rows are the
// routed slots sorted by expert, dst rows scattered back to slots) and
// segmented (MUL_MAT_ID's expert-weight gradient: slice e reduces over its
// own k range).  A compile-time parameter, so that the plain and grouped
// kernels carry none of the segmented mode's state.
constexpr int kModePlain = 0, kModeGrouped = 1, kModeSegmented = 2;

// The grouped and segmented modes' tiles are short in k, so their epilogue
// is a large share of a tile: there the result columns go through shared
// memory (each fold warp stages EPI_COLS columns of its 32 rows at a time)
// to bulk copies, and the fold moves on while the copies drain.
constexpr int EPI_COLS = 32;
constexpr int EPI_BYTES = FOLD_THREADS / 32 * EPI_COLS * 32 * 4;
template <int MODE>
constexpr bool staged_epilogue() { return MODE != kModePlain; }

// Shared memory: [B stages][raw src0 ring][epilogue staging][barriers], from a
// 1024-byte boundary (the 128-byte swizzle's); as many B stages as fit, up to six.
template <int TYPE, int MODE>
constexpr size_t smem_fixed_bytes() {
    return RawA<TYPE>::RSTAGES * RawA<TYPE>::SLOT + (staged_epilogue<MODE>() ? EPI_BYTES : 0) +
           sizeof(Bars) + 1024;
}
template <int TYPE, int MODE>
constexpr int b_stages() {
    return static_cast<int>(std::min<size_t>(
        MAX_BSTAGES, (SMEM_LIMIT - smem_fixed_bytes<TYPE, MODE>()) / STAGE_BYTES));
}
template <int TYPE, int MODE>
constexpr size_t smem_bytes() {
    return b_stages<TYPE, MODE>() * STAGE_BYTES + smem_fixed_bytes<TYPE, MODE>();
}

struct TcParams {
    const uint8_t *a;
    float *dst;
    int *status;
    int64_t M, K, N, ne02, ne12, dps2, dps3, a_row_bytes;
    int num_kb, mtiles, ntiles, inject;
    // stream-K: `ctas` CTAs share `iters` = tiles * num_kb iterations and
    // write the k-partials of shared tiles to `partial` ([ctas][2][BN][BM]);
    // ctas == 0 selects the data-parallel schedule
    int64_t iters;
    int ctas;
    float *partial;
    // persistent != 0 (with ctas == 0): CTA c takes whole tiles c, c + G, ...
    // (G = grid size) of the tile count, which grouped mode reads on the device
    int persistent;
    // grouped mode (MUL_MAT_ID_BACK): slices are experts, src1 rows are the
    // routed slots sorted by expert, dst rows are scattered back to slots
    const int *grp_count;         // [E] slots routed to each expert
    const int *grp_offset;        // [E] first sorted slot of each expert
    const int *grp_rows;          // [slots] sorted slot -> dst row
    const int *grp_tiles;         // work list: (expert << 16) | n-tile
    const int *grp_ntiles;        // valid entries in grp_tiles
    // segmented mode (MUL_MAT_ID's expert-weight gradient; data-parallel
    // only): slice e reduces over its own k range, seg_nkb[e] k-blocks from
    // row seg_off[e] of src0 (one src0 slice holding every segment) and
    // column seg_off[e] of the split src1 (one slice, every segment)
    const int *seg_off;
    const int *seg_nkb;
    // grouped / segmented: results leave through bulk copies (M % 4 == 0 and
    // dst 16-byte aligned, so every column's rows start on 16 bytes)
    int bulk_epi;
};

// First iteration of stream-K CTA c, and the CTA that owns iteration x.
__host__ __device__ __forceinline__ int64_t sk_begin(int64_t iters, int ctas, int64_t c) {
    return iters * c / ctas;
}
__host__ __device__ __forceinline__ int64_t sk_owner(int64_t iters, int ctas, int64_t x) {
    return ((x + 1) * ctas - 1) / iters;
}

// Where tile t sits: m-tile, n-tile, dst slice, its valid src1 rows, and the
// first src0 row (k = 0) of the src0 slice it reads.
struct Tile {
    int mt, nt;
    int64_t slice, ncols, brow0, a_row0;
    int nkb;                      // segmented mode: this tile's k-blocks
    int64_t kofs;                 // segmented mode: src1 k offset
};

template <int MODE>
__device__ __forceinline__ Tile decode_tile(const TcParams &p, int64_t t) {
    constexpr bool GROUPED = MODE == kModeGrouped;
    Tile d;
    if constexpr (GROUPED) {
        // work-list entries innermost: an expert's n-tiles of one m-tile are
        // neighbours, so the second one finds that m-tile of W in L2
        const int64_t entries = *p.grp_ntiles;
        d.mt = static_cast<int>(t / entries);
        const int packed = p.grp_tiles[t % entries];
        d.slice = packed >> 16;
        d.nt = packed & 0xFFFF;
        d.ncols = p.grp_count[d.slice];
        d.brow0 = p.grp_offset[d.slice] + static_cast<int64_t>(d.nt) * BN;
    } else {
        d.mt = static_cast<int>(t % p.mtiles);
        const int64_t rest = t / p.mtiles;
        d.nt = static_cast<int>(rest % p.ntiles);
        d.slice = rest / p.ntiles;
        d.ncols = p.N;
        d.brow0 = 0;
    }
    const int64_t i2 = d.slice % p.ne12, i3 = d.slice / p.ne12;
    d.a_row0 = (i3 / p.dps3 * p.ne02 + i2 / p.dps2) * p.K;
    if constexpr (MODE == kModeSegmented) {
        d.kofs = p.seg_off[d.slice];
        d.nkb = p.seg_nkb[d.slice];
        d.a_row0 = d.kofs;
    }
    return d;
}

// k-blocks of tile t
template <int MODE>
__device__ __forceinline__ int tile_nkb(const TcParams &p, const Tile &t) {
    if constexpr (MODE == kModeSegmented) return t.nkb;
    else return p.num_kb;
}

// A CTA's share of the iterations, in up to two phases: first it0 .. it1 - 1
// (a local count), starting at k-block kb0 of tile tile0, moving `stride`
// tiles on after a tile's last k-block (1 for a contiguous range, the grid
// size for whole tiles taken round-robin); then the global iterations
// b0 .. b1 - 1 (a stream-K range, tile-major), if b0 < b1.
struct Span {
    int64_t it0, it1, tile0, stride;
    int kb0;
    int64_t b0, b1;
};

// Walks a CTA's iterations in order; every role keeps its own copy.  `fresh`
// marks the first iteration of each phase (a new segment, whatever its kb),
// `split` the stream-K phase.
template <int MODE>
struct Walk {
    int64_t it, end, nb0, nb1;
    int tile, stride, kb;
    bool fresh, split;
    Tile t;
    __device__ __forceinline__ Walk(const TcParams &p, const Span &sp)
        : it(sp.it0), end(sp.it1), nb0(sp.b0), nb1(sp.b1), tile(static_cast<int>(sp.tile0)),
          stride(static_cast<int>(sp.stride)), kb(sp.kb0), fresh(true), split(false) {
        if (it < end) t = decode_tile<MODE>(p, tile);
        else second(p);
    }
    // switch to the stream-K range, if any
    __device__ __forceinline__ void second(const TcParams &p) {
        if (nb0 >= nb1) return;
        it = nb0;
        end = nb1;
        nb0 = nb1;
        tile = static_cast<int>(it / p.num_kb);
        kb = static_cast<int>(it % p.num_kb);
        stride = 1;
        fresh = split = true;
        t = decode_tile<MODE>(p, tile);
    }
    __device__ __forceinline__ void next(const TcParams &p) {
        ++it;
        fresh = false;
        if (++kb == tile_nkb<MODE>(p, t)) {
            kb = 0;
            tile += stride;
            if (it < end) t = decode_tile<MODE>(p, tile);
            else second(p);
        }
    }
};

// Position in a ring of N slots: the slot and the parity of its current use
// (the parity a "full" wait expects; an "empty" wait expects its negation).
template <int N>
struct Ring {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next() {
        if (++slot == N) {
            slot = 0;
            phase ^= 1;
        }
    }
};

template <int TYPE>
__device__ __forceinline__ float load_a(const uint8_t *row, int64_t m) {
    return decode_row<TYPE>(row, m);
}

// The scale and offset of one k row's group of elements, for the
// cooperative decode of staged_half: `blk` is the row's block (32-element
// types) or super-block (K-quants); `grp` the warp's group (the 32-block in
// the tile, or the K-quant's 32-element group in its half `h`); `hl` the lane
// half for types with a scale per 16 elements.  x = fmaf(sc, code, of)
// reproduces decode() exactly (of = -0.0 keeps the sign of a zero product).
template <int TYPE>
__device__ __forceinline__ void block_scale(const uint8_t *blk, int grp, int h, int hl, float &sc,
                                            float &of, uint32_t &xw) {
    using namespace qdec;
    if constexpr (TYPE == OOP_TYPE_Q4_1 || TYPE == OOP_TYPE_Q5_1) {
        sc = f16(blk);
        of = f16(blk + 2);
        if constexpr (TYPE == OOP_TYPE_Q5_1) xw = u32(blk + 4);
    } else if constexpr (TYPE == OOP_TYPE_Q5_0) {
        sc = f16(blk);
        of = -0.0f;
        xw = u32(blk + 2);
    } else if constexpr (TYPE == OOP_TYPE_Q4_K || TYPE == OOP_TYPE_Q5_K) {
        uint32_t s6, m6;
        scale_min_k4(blk + 4, 4 * h + grp, s6, m6);
        sc = f16(blk) * static_cast<float>(s6);
        of = -(f16(blk + 2) * static_cast<float>(m6));
    } else if constexpr (TYPE == OOP_TYPE_Q6_K) {
        sc = f16(blk + 208) * static_cast<float>(static_cast<int8_t>(blk[192 + 8 * h + hl + 2 * grp]));
        of = -0.0f;
    } else if constexpr (TYPE == OOP_TYPE_Q2_K) {
        const uint32_t s = blk[8 * h + 2 * grp + hl];
        sc = f16(blk + 80) * static_cast<float>(s & 0xFu);
        of = -(f16(blk + 82) * static_cast<float>(s >> 4));
    } else if constexpr (TYPE == OOP_TYPE_Q3_K) {
        sc = f16(blk + 108) * static_cast<float>(scale_q3k(blk + 96, 8 * h + 2 * grp + hl));
        of = -0.0f;
    }
}

// The code of element `lane` of the group (see block_scale) in row `blk`.
template <int TYPE>
__device__ __forceinline__ int block_code(const uint8_t *blk, int grp, int h, int lane,
                                          uint32_t xw) {
    if constexpr (TYPE == OOP_TYPE_Q4_1) {
        const uint32_t byte = blk[4 + (lane & 15)];
        return static_cast<int>(lane < 16 ? (byte & 0xFu) : (byte >> 4));
    } else if constexpr (TYPE == OOP_TYPE_Q5_0 || TYPE == OOP_TYPE_Q5_1) {
        constexpr int QS = TYPE == OOP_TYPE_Q5_0 ? 6 : 8;
        const uint32_t byte = blk[QS + (lane & 15)];
        const uint32_t lo = lane < 16 ? (byte & 0xFu) : (byte >> 4);
        const int v = static_cast<int>(lo | (((xw >> lane) & 1u) << 4));
        return TYPE == OOP_TYPE_Q5_0 ? v - 16 : v;
    } else if constexpr (TYPE == OOP_TYPE_Q4_K || TYPE == OOP_TYPE_Q5_K) {
        constexpr int QS = TYPE == OOP_TYPE_Q4_K ? 16 : 48;
        const int sb = 4 * h + grp;
        uint32_t q = (blk[QS + 32 * (sb >> 1) + lane] >> (4 * (sb & 1))) & 0xFu;
        if constexpr (TYPE == OOP_TYPE_Q5_K) q |= ((blk[16 + lane] >> sb) & 1u) << 4;
        return static_cast<int>(q);
    } else if constexpr (TYPE == OOP_TYPE_Q6_K) {
        const uint32_t byte = blk[64 * h + lane + 32 * (grp & 1)];
        const uint32_t lo = grp >= 2 ? (byte >> 4) : (byte & 0xFu);
        const uint32_t hi = (blk[128 + 32 * h + lane] >> (2 * grp)) & 3u;
        return static_cast<int>(lo | (hi << 4)) - 32;
    } else if constexpr (TYPE == OOP_TYPE_Q2_K) {
        return static_cast<int>((blk[16 + 32 * h + lane] >> (2 * grp)) & 3u);
    } else if constexpr (TYPE == OOP_TYPE_Q3_K) {
        const int q2 = static_cast<int>((blk[32 + 32 * h + lane] >> (2 * grp)) & 3u);
        return q2 - (((blk[lane] >> (4 * h + grp)) & 1u) ? 0 : 4);
    } else {
        return 0;
    }
}

// The cooperative decode of staged_half straight from global memory, for
// src0 rows TMA cannot stage (row bytes not a multiple of 16): `row0` is this
// warp's group in the first of the 16 k rows, `stride` the row bytes; rows
// nk.. (past K, or all of them for a group past M) are neither read nor used.
template <int TYPE>
__device__ __forceinline__ void global_half(const uint8_t *row0, int64_t stride, int nk,
                                            int quad, int h, int lane, float (&x)[KH]) {
    const int jr = lane & (KH - 1), hl = lane >> 4;
    float sc = 0.f, of = 0.f;
    uint32_t xw = 0;
    if (jr < nk) block_scale<TYPE>(row0 + jr * stride, quad, h, hl, sc, of, xw);
    constexpr bool HALVES = TYPE == OOP_TYPE_Q6_K || TYPE == OOP_TYPE_Q2_K ||
                            TYPE == OOP_TYPE_Q3_K;
    const int src_add = HALVES ? 16 * (lane >> 4) : 0;
#pragma unroll
    for (int j = 0; j < KH; ++j) {
        const float sj = __shfl_sync(0xffffffffu, sc, j + src_add);
        const float oj = __shfl_sync(0xffffffffu, of, j + src_add);
        uint32_t xj = 0;
        if constexpr (TYPE == OOP_TYPE_Q5_0 || TYPE == OOP_TYPE_Q5_1)
            xj = __shfl_sync(0xffffffffu, xw, j);
        x[j] = j < nk ? fmaf(sj, static_cast<float>(block_code<TYPE>(row0 + j * stride, quad, h,
                                                                        lane, xj)),
                             oj)
                      : 0.f;
    }
}

// The 16 src0 values (k rows 16*kh .. 16*kh+15 of a staged k-block) of row
// r of the m-tile.  Lane l of the warp owns row r = 32 * (warp % 4) + l, so a
// warp covers one quantisation block: its 16 scales are read once (lane j
// reads k row j) and passed around with shuffles.
// Where k row j (0 .. BK-1) of a k-block sits in its staged slot: rows in
// order, or (row groups of AG) member j % AG's box holds the block's rows
// j % AG, j % AG + AG, ...
template <int AG>
__device__ __forceinline__ int slot_row(int j) {
    if constexpr (AG <= 1) return j;
    else return (j % AG) * (BK / AG) + j / AG;
}

template <int TYPE, int AG>
__device__ __forceinline__ void staged_half(const uint8_t *slot, int r, uint32_t off0, int lane,
                                            int kh, float (&x)[KH], int mt) {
    using Raw = RawA<TYPE>;
    const uint8_t *rows = slot + kh * KH * Raw::ROW_BYTES;
    if constexpr (TYPE == OOP_TYPE_F32) {
#pragma unroll
        for (int j = 0; j < KH; ++j)
            x[j] = reinterpret_cast<const float *>(rows + j * Raw::ROW_BYTES)[r];
    } else if constexpr (Raw::PLAIN) {
#pragma unroll
        for (int j = 0; j < KH; ++j) x[j] = decode<TYPE>(rows + j * Raw::ROW_BYTES + 2 * r, 0);
    } else if constexpr (TYPE != OOP_TYPE_Q8_0 && TYPE != OOP_TYPE_Q4_0) {
        // The other block types.  Every element is scale * code + offset,
        // where scale and offset depend only on the k row and on which
        // 32 (or 16) elements of the block the element is in -- and the 32
        // lanes of a warp are one such group (or two halves of one).  So lane
        // L works out the scale and offset of row L % 16 for lane half L / 16
        // once; each lane then takes its row's pair by shuffle and adds its
        // own code: one fused multiply-add, the same rounding as decode().
        const int quad = r >> 5;
        const int bofs = QFormat<TYPE>::QK == 32 ? quad * QFormat<TYPE>::BYTES : 0;
        // this warp's bytes of its j-th k row of the block
        auto row_at = [&](int j) -> const uint8_t * {
            if constexpr (AG > 1) {
                const int jb = kh * KH + j;                 // row in the k-block
                return slot + slot_row<AG>(jb) * Raw::ROW_BYTES +
                       ((off0 >> (4 * (jb % AG))) & 15u) + bofs;
            } else {
                return rows + j * Raw::ROW_BYTES + off0 + bofs;
            }
        };
        const int h = mt & 1;                               // K-quants: half of the super-block
        const int jr = lane & (KH - 1), hl = lane >> 4;
        float sc, of;
        uint32_t xw = 0;                                    // q5_0 / q5_1: the fifth bits
        block_scale<TYPE>(row_at(jr), quad, h, hl, sc, of, xw);
        constexpr bool HALVES = TYPE == OOP_TYPE_Q6_K || TYPE == OOP_TYPE_Q2_K ||
                                TYPE == OOP_TYPE_Q3_K;      // a scale per 16 elements
        const int src_add = HALVES ? 16 * (lane >> 4) : 0;
#pragma unroll
        for (int j = 0; j < KH; ++j) {
            const float sj = __shfl_sync(0xffffffffu, sc, j + src_add);
            const float oj = __shfl_sync(0xffffffffu, of, j + src_add);
            uint32_t xj = 0;
            if constexpr (TYPE == OOP_TYPE_Q5_0 || TYPE == OOP_TYPE_Q5_1)
                xj = __shfl_sync(0xffffffffu, xw, j);
            const int q = block_code<TYPE>(row_at(j), quad, h, lane, xj);
            x[j] = fmaf(sj, static_cast<float>(q), oj);
        }
    } else {
        const uint8_t *blk = rows + off0 + (r >> 5) * QFormat<TYPE>::BYTES;
        const float dl = half_bits_to_float(
            *reinterpret_cast<const uint16_t *>(blk + (lane & (KH - 1)) * Raw::ROW_BYTES));
        // d*v two k rows at a time in packed f32x2 arithmetic, exactly: with
        // f = 1.5*2^23 + v (exact), d*f - d*1.5*2^23 is one fused multiply-add
        // whose single rounding is exact because d*v fits in fp32
        const uint64_t big2 = ptx::pack2(-12582912.0f, -12582912.0f);
#pragma unroll
        for (int j = 0; j < KH; j += 2) {
            int v[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                if constexpr (TYPE == OOP_TYPE_Q8_0) {
                    v[e] = static_cast<int8_t>(blk[(j + e) * Raw::ROW_BYTES + 2 + lane]);
                } else {
                    const uint8_t byte = blk[(j + e) * Raw::ROW_BYTES + 2 + (lane & 15)];
                    v[e] = (lane < 16 ? (byte & 0x0f) : (byte >> 4)) - 8;
                }
            }
            const uint64_t d2 = ptx::pack2(__shfl_sync(0xffffffffu, dl, j),
                                           __shfl_sync(0xffffffffu, dl, j + 1));
            const uint64_t f2 = ptx::pack2(__int_as_float(0x4B400000 + v[0]),
                                           __int_as_float(0x4B400000 + v[1]));
            ptx::unpack2(ptx::fma2(d2, f2, ptx::mul2(d2, big2)), x[j], x[j + 1]);
        }
    }
}

// A bounded wait whose outcome the whole warp shares, so that the lanes stay
// converged for the warp-collective tcgen05.ld/st and shuffles after it.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          bool *timed_out) {
    const bool ok = ptx::mbar_wait_bounded(bar, parity, abort, true, WAIT_NS, timed_out);
    return __all_sync(0xffffffffu, ok);
}

// AG: how src0 is staged -- 0 loaded from global memory by the producer, 1
// one TMA row per src0 row, >1 TMA rows of AG src0 rows (RawA::RG).
template <int TYPE, int AG, int MODE>
__global__ void __maxnreg__(MAX_REGS)
    tc_out_prod_kernel(const __grid_constant__ CUtensorMap map_bhi,
                       const __grid_constant__ CUtensorMap map_blo,
                       const __grid_constant__ CUtensorMap map_a, const TcParams p) {
    constexpr bool GROUPED = MODE == kModeGrouped;
    constexpr bool TMA_A = AG > 0;
    using Raw = RawA<TYPE>;
    constexpr int AGD = AG > 1 ? AG : 1;                 // the group size (1: single rows)
    static_assert(Raw::RG % AGD == 0 && (BK / AGD) * Raw::ROW_BYTES % 128 == 0,
                  "row groups: a divisor of RG, each box 128-byte aligned");
    constexpr bool HAS_ALO = !is_tf32_exact<TYPE>();   // bf16 / f16 values are TF32 values
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int BST = b_stages<TYPE, MODE>();
    uint8_t *ring = smem + BST * STAGE_BYTES;
    uint8_t *epi = ring + Raw::RSTAGES * Raw::SLOT;
    Bars *bars = reinterpret_cast<Bars *>(epi + (staged_epilogue<MODE>() ? EPI_BYTES : 0));
    volatile int *abort = &bars->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // The tile kernel is launched as a programmatic dependent of the split
    // pass before it (bsplit / mmid_gsplit): nothing that pass (or the routing
    // before it) writes is read before griddep_wait().  The grouped kernel
    // reads the device-side tile count at once, so it waits here; the other
    // waits after its prologue.
    if constexpr (GROUPED) ptx::griddep_wait();
    // this CTA's iterations [it0, it1)
    int64_t it0, it1;
    Span span = {};
    if (p.ctas > 0) {
        // stream-K: the full waves of whole tiles first, round-robin (all CTAs
        // at the same k, so the src0 and src1 rows they read are shared in
        // L2), then the tail tiles' iterations split evenly; every CTA gets
        // the same number of iterations to within one.  Grouped: the tile
        // count is known on the device only.
        const int64_t tiles =
            GROUPED ? static_cast<int64_t>(p.mtiles) * *p.grp_ntiles : p.iters / p.num_kb;
        const int64_t dp_tiles = tiles / p.ctas * p.ctas;
        const int64_t tail = (tiles - dp_tiles) * p.num_kb, base = dp_tiles * p.num_kb;
        span = {0, dp_tiles / p.ctas * p.num_kb, static_cast<int64_t>(blockIdx.x), p.ctas, 0,
                base + sk_begin(tail, p.ctas, blockIdx.x),
                base + sk_begin(tail, p.ctas, blockIdx.x + 1)};
        it0 = 0;
        it1 = span.it1 + (span.b1 - span.b0);
    } else if (p.persistent) {
        const int64_t tiles =
            GROUPED ? static_cast<int64_t>(p.mtiles) * *p.grp_ntiles : p.iters / p.num_kb;
        it0 = 0;
        if constexpr (MODE == kModeSegmented) {
            // the k-blocks of this CTA's tiles c, c + G, ... (p.iters holds the tile count)
            it1 = 0;
            const int64_t per = static_cast<int64_t>(p.mtiles) * p.ntiles;
            for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) it1 += p.seg_nkb[t / per];
        } else {
            const int64_t mine =
                tiles > blockIdx.x ? (tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
            it1 = mine * p.num_kb;
        }
        span = {it0, it1, static_cast<int64_t>(blockIdx.x), static_cast<int64_t>(gridDim.x), 0};
    } else {
        const int64_t t = static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x;
        if constexpr (GROUPED) {
            if (t >= static_cast<int64_t>(p.mtiles) * *p.grp_ntiles) return;   // no work left
        }
        if constexpr (MODE == kModeSegmented) {
            // this tile's k-block count is its slice's
            it0 = 0;
            it1 = p.seg_nkb[t / (static_cast<int64_t>(p.mtiles) * p.ntiles)];
        } else {
            it0 = t * p.num_kb;
            it1 = it0 + p.num_kb;
        }
        span = {it0, it1, t, 1, 0};
    }
    if (it0 >= it1) return;

    if (threadIdx.x == 0) {
        for (int s = 0; s < BST; ++s) ptx::mbar_init(&bars->bempty[s], 1);
        for (int s = 0; s < A_STAGES; ++s) ptx::mbar_init(&bars->afull[s], PRODUCER_THREADS);
        for (int r = 0; r < Raw::RSTAGES; ++r) {
            ptx::mbar_init(&bars->rfull[r], 1);
            ptx::mbar_init(&bars->rempty[r], PRODUCER_THREADS);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&bars->accf[b], 1);
            ptx::mbar_init(&bars->acce[b], FOLD_THREADS);
        }
        ptx::mbar_init(&bars->d2free, FOLD_THREADS);
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
    if constexpr (!GROUPED) ptx::griddep_wait();   // the split of src1 is complete
    const uint32_t tmem = bars->tmem_base;
    bool timed_out = false;
    // The register split: one setmaxnreg per warpgroup, executed by all its
    // warps at the head of the warpgroup's branch, before any wait, so the
    // fold's request is met once the others have given theirs back.
    if (warp < WARP_PROD0) {
        ptx::setmaxnreg_dec<REGS_CTRL>();
        if (warp == 0) {
            // ---------------- TMA producer ----------------
            if (lane == 0) {
                int last_ph[MAX_RSTAGES];           // parity of each slot's last copy, -1: none
                for (int r = 0; r < MAX_RSTAGES; ++r) last_ph[r] = -1;
                Ring<Raw::RSTAGES> rr;
                Ring<BST> bb;
                int g = 0;
                for (Walk<MODE> w(p, span); w.it < w.end; w.next(p), rr.next(), bb.next(), ++g) {
                    const Tile &t = w.t;
                    // ring slot free (producers done with g - RSTAGES), B stage
                    // free (MMAs of g - BST completed)
                    const int r = rr.slot, s = bb.slot;
                    if (!ptx::mbar_wait_bounded(&bars->rempty[r], rr.phase ^ 1, abort, true, WAIT_NS,
                                                &timed_out) ||
                        !ptx::mbar_wait_bounded(&bars->bempty[s], bb.phase ^ 1, abort, true, WAIT_NS,
                                                &timed_out))
                        break;
                    if (p.inject == 1 && g == 0) continue;   // test hook: drop one iteration
                    uint8_t *st = smem + s * STAGE_BYTES;
                    ptx::mbar_arrive_expect_tx(
                        &bars->rfull[r],
                        static_cast<uint32_t>(2 * B_IMG + (TMA_A ? Raw::ROW_BYTES * BK : 0)));
                    if constexpr (AG == 1) {
                        const int box_x = elementwise_type<TYPE>()
                                              ? t.mt * BM
                                              : static_cast<int>(raw_tile_byte0<TYPE>(t.mt) & ~15);
                        ptx::tma_load_2d(ring + r * Raw::SLOT, &map_a, &bars->rfull[r], box_x,
                                         static_cast<int>(t.a_row0 + static_cast<int64_t>(w.kb) * BK));
                    } else if constexpr (AG > 1) {
                        // box g: member g of the block's BK / AG row groups
                        const int64_t byte0 = raw_tile_byte0<TYPE>(t.mt);
                        const int grp = static_cast<int>((t.a_row0 + static_cast<int64_t>(w.kb) * BK) / AG);
#pragma unroll
                        for (int gm = 0; gm < AG; ++gm)
                            ptx::tma_load_2d(ring + r * Raw::SLOT + gm * (BK / AG) * Raw::ROW_BYTES,
                                             &map_a, &bars->rfull[r],
                                             static_cast<int>((gm * p.a_row_bytes + byte0) & ~15), grp);
                    }
                    if constexpr (GROUPED) {
                        ptx::tma_load_2d(st, &map_bhi, &bars->rfull[r], w.kb * BK,
                                         static_cast<int>(t.brow0));
                        ptx::tma_load_2d(st + B_IMG, &map_blo, &bars->rfull[r], w.kb * BK,
                                         static_cast<int>(t.brow0));
                    } else {
                        // segmented: one src1 slice, each expert's segment at its k offset
                        const int bk = MODE == kModeSegmented
                                           ? static_cast<int>(t.kofs + static_cast<int64_t>(w.kb) * BK)
                                           : w.kb * BK;
                        const int bs = MODE == kModeSegmented ? 0 : static_cast<int>(t.slice);
                        ptx::tma_load_3d(st, &map_bhi, &bars->rfull[r], bk, t.nt * BN, bs);
                        ptx::tma_load_3d(st + B_IMG, &map_blo, &bars->rfull[r], bk, t.nt * BN, bs);
                    }
                    last_ph[r] = static_cast<int>(rr.phase);
                }
                // copies in flight must land before the CTA's smem is released
                for (int r = 0; r < Raw::RSTAGES; ++r)
                    if (last_ph[r] >= 0)
                        ptx::mbar_wait_bounded(&bars->rfull[r], static_cast<uint32_t>(last_ph[r]),
                                               abort, false, WAIT_NS, &timed_out);
            }
        } else if (warp == 1) {
            // ---------------- MMA issuer ----------------
            // The whole warp runs the loop, so its control flow and operands are
            // warp-uniform (kept in uniform registers); one elected lane issues.
            constexpr uint32_t idesc = ptx::idesc_tf32(BM, BN);
            const uint32_t d2 = tmem + COL_D2;
            const uint64_t desc0 = ptx::sw128_kmajor_desc(ptx::smem_u32(smem));
            int g = 0, q = -1, seg = -1;         // iteration, chunk, segment counters
            int seg_kb0 = 0;
            Ring<A_STAGES> aa;
            Ring<BST> bb;
            // A test of a barrier costs ~100 cycles even when its phase is long
            // complete, the warp issues nothing while a test's result is
            // outstanding, and the tensor core queues only about two MMAs beyond
            // the one executing.  So every barrier iteration g+1 needs is tested
            // right after the MMAs of g are issued, all at once (one barrier per
            // lane); the blocking waits run only when that test came back
            // negative.
            bool ready = false;
            for (Walk<MODE> w(p, span); w.it < w.end; ++g) {
                const bool seg_first = w.fresh || w.kb == 0;
                if (seg_first) {
                    ++seg;
                    seg_kb0 = w.kb;
                }
                const int in_chunk = (w.kb - seg_kb0) % CHUNK_KB;
                const bool seg_last = w.kb + 1 == tile_nkb<MODE>(p, w.t) || w.it + 1 == w.end;
                const bool chunk_last = in_chunk == CHUNK_KB - 1 || seg_last;
                if (in_chunk == 0) ++q;
                const int buf = q & 1;
                const int s = bb.slot, sa = aa.slot;
                // D1 buffer drained by the fold; D2 read at the previous segment's
                // end; this block's A stage written (its producers also saw its B
                // stage land)
                // D2 is first written at a segment's second block (its first
                // block keeps every product in the fresh D1 chunk), so the wait for
                // the fold to have read the previous segment's D2 sits there
                const int seg_pos = w.kb - seg_kb0;
                if (!ready &&
                    ((in_chunk == 0 &&
                      !warp_wait(&bars->acce[buf], (static_cast<uint32_t>(q >> 1) & 1) ^ 1, abort,
                                 &timed_out)) ||
                     (seg_pos == 1 && seg > 0 &&
                      !warp_wait(&bars->d2free, static_cast<uint32_t>(seg - 1) & 1, abort,
                                 &timed_out)) ||
                     !warp_wait(&bars->afull[sa], aa.phase, abort, &timed_out)))
                    break;
                ptx::tc_fence_after();
                const uint32_t d1 = tmem + static_cast<uint32_t>(buf * BN);
                const uint32_t ahi = tmem + COL_A + static_cast<uint32_t>(sa) * A_COLS;
                const uint32_t alo = ahi + BK;
                // descriptor start addresses count 16-byte units
                const uint64_t dhi = desc0 + static_cast<uint64_t>((s * STAGE_BYTES) >> 4);
                const uint64_t dlo = dhi + (B_IMG >> 4);
                // the barrier each lane tests for iteration g+1 while g's MMAs are
                // issued: its A stage (lane 0), its D1 buffer if it starts a chunk
                // (lane 1), D2 if it is its segment's second block (lane 2)
                uint64_t *tbar;
                uint32_t tpar;
                {
                    Ring<A_STAGES> an = aa;
                    an.next();
                    tbar = &bars->afull[an.slot];
                    tpar = an.phase;
                }
                if (lane == 1 && chunk_last) {
                    tbar = &bars->acce[(q + 1) & 1];
                    tpar = (static_cast<uint32_t>((q + 1) >> 1) & 1) ^ 1;
                }
                if (lane == 2 && seg_pos == 0 && !seg_last && seg > 0) {
                    tbar = &bars->d2free;
                    tpar = static_cast<uint32_t>(seg - 1) & 1;
                }
                const uint32_t lead = ptx::elect_one() ? 1u : 0u;
                uint32_t ok;
                if constexpr (HAS_ALO) {
                    if (seg_pos == 0)   // every product into the fresh D1, small ones first
                        ok = ptx::mma_block_3xtf32_one_test(d1, ahi, alo, dhi, dlo, idesc, lead, tbar,
                                                            tpar);
                    else                // cross terms into D2, the big term into D1
                        ok = ptx::mma_block_3xtf32_test(d1, d2, ahi, alo, dhi, dlo, idesc,
                                                        in_chunk == 0, seg_pos == 1, lead, tbar, tpar);
                } else {
                    // bf16 / f16 src0: a_lo is zero, one cross term
                    ok = ptx::mma_block_1xlo_test(seg_pos == 0 ? d1 : d2, d1, ahi, dhi, dlo, idesc,
                                                  seg_pos <= 1, in_chunk == 0 && seg_pos != 0, lead,
                                                  tbar, tpar);
                }
                if (lead) {
                    ptx::mma_commit(&bars->bempty[s]);
                    if (chunk_last) ptx::mma_commit(&bars->accf[buf]);
                }
                __syncwarp();
                ready = __all_sync(0xffffffffu, ok != 0);
                w.next(p);
                aa.next();
                bb.next();
            }
            // every MMA issued must finish before TMEM is released
            if (ptx::elect_one()) {
                ptx::mma_commit(&bars->mma_done);
                ptx::mbar_wait_bounded(&bars->mma_done, 0, abort, false, WAIT_NS, &timed_out);
            }
            __syncwarp();
        }                                                  // warps 2 and 3: idle
    } else if (warp < WARP_FOLD0) {
        // ---------------- src0 producer ----------------
        ptx::setmaxnreg_dec<(AG > 1 ? REGS_PROD_RG : REGS_PROD)>();
        const int quad = warp & 3;                       // TMEM lanes 32*quad ..
        const int kh = (warp - WARP_PROD0) >> 2;         // k rows KH*kh .. of each block
        const int r = 32 * quad + lane;                  // row of the m-tile
        const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
        int g = 0;
        bool early_r = false;
        Ring<Raw::RSTAGES> rr;
        Ring<A_STAGES> aa;
        Ring<BST> eb;                                    // bempty of iteration g - A_STAGES
        for (Walk<MODE> w(p, span); w.it < w.end; w.next(p), rr.next(), aa.next(), ++g) {
            const Tile &t = w.t;
            const int64_t m = static_cast<int64_t>(t.mt) * BM + r;
            const bool mok = m < p.M;
            const int64_t k0 = static_cast<int64_t>(w.kb) * BK + kh * KH;
            const bool kfull = k0 + KH <= p.K;
            float x[KH];
            // every copy of this iteration landed: its raw src0 rows and, for
            // the MMA that waits on this warp, its B stage
            const int rs = rr.slot;
            if (!__all_sync(0xffffffffu, early_r) &&
                !warp_wait(&bars->rfull[rs], rr.phase, abort, &timed_out))
                break;
            // early test for g+1 (see the MMA issuer): its latency hides
            // behind this iteration's work
            {
                Ring<Raw::RSTAGES> rn = rr;
                rn.next();
                early_r = ptx::mbar_test_wait(&bars->rfull[rn.slot], rn.phase);
            }
            if constexpr (TMA_A) {
                // how far past its box's 16-byte start the tile's bytes begin:
                // one offset, or (row groups) one per member, 4 bits each
                uint32_t off0 = 0;
                if constexpr (AG > 1) {
                    const int64_t byte0 = raw_tile_byte0<TYPE>(t.mt);
#pragma unroll
                    for (int gm = 0; gm < AG; ++gm)
                        off0 |= static_cast<uint32_t>((gm * p.a_row_bytes + byte0) & 15) << (4 * gm);
                } else if constexpr (!elementwise_type<TYPE>()) {
                    off0 = static_cast<uint32_t>(raw_tile_byte0<TYPE>(t.mt) & 15);
                }
                __syncwarp();
                staged_half<TYPE, AG>(ring + rs * Raw::SLOT, r, off0, lane, kh, x, t.mt);
                // rows past M and k past K read whatever the box holds there
                if (!(__all_sync(0xffffffffu, mok) && kfull)) {
#pragma unroll
                    for (int j = 0; j < KH; ++j)
                        if (!mok || k0 + j >= p.K) x[j] = 0.f;
                }
            } else {
                const uint8_t *a_slice = p.a + t.a_row0 * p.a_row_bytes;
                if constexpr (!Raw::PLAIN && TYPE != OOP_TYPE_Q8_0 && TYPE != OOP_TYPE_Q4_0) {
                    // blocks hold whole 32-element groups, so mok is the same
                    // in every lane: a group past M is neither read nor used
                    using F = QFormat<TYPE>;
                    const uint8_t *row0 = a_slice + k0 * p.a_row_bytes +
                                          raw_tile_byte0<TYPE>(t.mt) +
                                          (F::QK == 32 ? (r >> 5) * F::BYTES : 0);
                    const int nk = static_cast<int>(
                        mok ? std::min<int64_t>(KH, std::max<int64_t>(0, p.K - k0)) : 0);
                    global_half<TYPE>(row0, p.a_row_bytes, nk, r >> 5, t.mt & 1, lane, x);
                } else {
#pragma unroll
                    for (int j = 0; j < KH; ++j) {
                        const int64_t k = k0 + j;
                        x[j] = (mok && k < p.K) ? load_a<TYPE>(a_slice + k * p.a_row_bytes, m)
                                                : 0.f;
                    }
                }
            }
            __syncwarp();
            ptx::mbar_arrive(&bars->rempty[rs]);
            uint32_t hi[KH], lo[KH];
#pragma unroll
            for (int e = 0; e < KH; e += 2) {
                // f32 src0 may hold any finite value: the saturating form
                // keeps fp32's top binade finite; dequantised and bf16 values
                // never reach it
                if constexpr (TYPE == OOP_TYPE_F32) {
                    hi[e] = ptx::tf32_round_bits_sat(__float_as_uint(x[e]));
                    hi[e + 1] = ptx::tf32_round_bits_sat(__float_as_uint(x[e + 1]));
                } else {
                    hi[e] = ptx::tf32_round_bits(__float_as_uint(x[e]));
                    hi[e + 1] = ptx::tf32_round_bits(__float_as_uint(x[e + 1]));
                }
                // x - hi is exact in fp32 (two elements per instruction)
                float r0, r1;
                ptx::unpack2(ptx::sub2(ptx::pack2(x[e], x[e + 1]),
                                       ptx::pack2(__uint_as_float(hi[e]), __uint_as_float(hi[e + 1]))),
                             r0, r1);
                if constexpr (split_needs_rounding<TYPE>()) {
                    lo[e] = ptx::tf32_round_bits(__float_as_uint(r0));
                    lo[e + 1] = ptx::tf32_round_bits(__float_as_uint(r1));
                } else {
                    // d*q has at most 22 significant bits: x - hi is already
                    // a TF32 value, no second rounding needed
                    lo[e] = __float_as_uint(r0);
                    lo[e + 1] = __float_as_uint(r1);
                }
            }
            // A stage g % A_STAGES is free once the MMAs of g - A_STAGES completed
            const int sa = aa.slot;
            if (g >= A_STAGES) {
                if (!warp_wait(&bars->bempty[eb.slot], eb.phase, abort, &timed_out)) break;
                eb.next();
            }
            ptx::tc_fence_after();
            const uint32_t a_st = tmem + lane_off + COL_A + static_cast<uint32_t>(sa) * A_COLS;
            ptx::tmem_st16(a_st + KH * kh, hi);
            if constexpr (HAS_ALO) ptx::tmem_st16(a_st + BK + KH * kh, lo);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bars->afull[sa]);
        }
    } else {
        // ---------------- fold + epilogue ----------------
        ptx::setmaxnreg_inc<(AG > 1 ? REGS_FOLD_RG : REGS_FOLD)>();
        const int quad = warp & 3;                          // TMEM lanes 32*quad ..
        const int half = (warp - WARP_FOLD0) >> 2;          // columns FOLD_COLS*half ..
        const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
        const uint32_t col0 = static_cast<uint32_t>(FOLD_COLS * half);
        const int row = 32 * quad + lane;
        // this thread's running sums S of its 64 columns, and their Kahan
        // compensations C, two columns per register as bfloat16 (C is at most
        // about half an ulp of S, so rounding it to 8 bits costs ~2^-9 ulp of
        // S per fold)
        float sreg[FOLD_COLS];
        uint32_t creg[FOLD_COLS / 2];
        int seg_kb0 = 0;
        bool seg_split0 = false;        // the segment starts the stream-K range
        int q = -1;
        for (Walk<MODE> w(p, span); w.it < w.end; w.next(p)) {
            if (w.fresh || w.kb == 0) {
                seg_kb0 = w.kb;
                seg_split0 = w.fresh && w.split;
            }
            const int in_chunk = (w.kb - seg_kb0) % CHUNK_KB;
            const bool last = w.kb + 1 == tile_nkb<MODE>(p, w.t) || w.it + 1 == w.end;   // segment ends
            if (in_chunk == 0) ++q;
            if (in_chunk != CHUNK_KB - 1 && !last) continue;   // once per chunk
            const Tile &t = w.t;
            const int buf = q & 1;
            if (!warp_wait(&bars->accf[buf], static_cast<uint32_t>(q >> 1) & 1, abort,
                           &timed_out))
                break;
            ptx::tc_fence_after();
            const bool first = w.kb - seg_kb0 < CHUNK_KB;       // segment's first chunk
            // the chunk into (S, C)
#pragma unroll
            for (int pc = 0; pc < FOLD_COLS / 16; ++pc) {
                const uint32_t col = col0 + pc * 16;
                uint32_t xv[16];
                ptx::tmem_ld16_wait(tmem + lane_off + buf * BN + col, xv);
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    float &s0 = sreg[pc * 16 + j], &s1 = sreg[pc * 16 + j + 1];
                    uint32_t &cb = creg[pc * 8 + j / 2];
                    if (first) {            // S = the first chunk, C = 0
                        s0 = __uint_as_float(xv[j]);
                        s1 = __uint_as_float(xv[j + 1]);
                        cb = 0;
                        continue;
                    }
                    // Kahan on two columns at once: the running sum is S - C
                    const uint64_t c2 = ptx::unpack_bf16x2(cb);
                    const uint64_t s2 = ptx::pack2(s0, s1);
                    const uint64_t x2 = ptx::pack2(__uint_as_float(xv[j]), __uint_as_float(xv[j + 1]));
                    const uint64_t y2 = ptx::sub2(x2, c2);
                    const uint64_t t2 = ptx::add2(s2, y2);
                    float n0, n1;
                    ptx::unpack2(ptx::sub2(ptx::sub2(t2, s2), y2), n0, n1);
                    cb = ptx::pack_bf16x2(n0, n1);
                    ptx::unpack2(t2, s0, s1);
                }
            }
            // the D1 buffer is drained: the MMA may refill it during the epilogue
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bars->acce[buf]);
            if (!last) continue;
            // The segment's result S - C + D2 (the cross terms): to dst, or, for
            // a segment that is not the whole tile, to a stream-K partial slot
            // (slot 0 for the CTA's first segment of the split range, 1 for its
            // last).  Each thread writes its row's 64 columns: a warp writes 32
            // consecutive m of one dst row per column.
            const bool whole = seg_kb0 == 0 && w.kb + 1 == tile_nkb<MODE>(p, w.t);
            const bool has_d2 = w.kb > seg_kb0;
            const int64_t m = static_cast<int64_t>(t.mt) * BM + row;
            const int tile_cols = static_cast<int>(
                std::min<int64_t>(BN, t.ncols - static_cast<int64_t>(t.nt) * BN));
            float *part = whole ? nullptr
                                : p.partial + (static_cast<int64_t>(blockIdx.x) * 2 +
                                               (seg_split0 ? 0 : 1)) * (BM * BN) + row;
            // plain: column jc of the tile is dst row nt * BN + jc
            float *dcol = (GROUPED ? p.dst : p.dst + t.slice * p.N * p.M) + m;
            if constexpr (!GROUPED) dcol += static_cast<int64_t>(t.nt) * BN * p.M;
            // grouped: the dst rows of the thread's 64 columns, read once per
            // tile, lane l holding those of columns col0 + l and col0 + 32 + l,
            // handed out by shuffles as the columns are stored
            int rows_lo = 0, rows_hi = 0;
            if constexpr (GROUPED) {
                const int c = static_cast<int>(col0) + lane;
                if (c < tile_cols) rows_lo = p.grp_rows[t.brow0 + c];
                if (c + 32 < tile_cols) rows_hi = p.grp_rows[t.brow0 + c + 32];
            }
            // S - C first: the compensations' registers are free for the loads
#pragma unroll
            for (int j = 0; j < FOLD_COLS; j += 2) {
                float c0, c1;
                ptx::unpack2(ptx::unpack_bf16x2(creg[j / 2]), c0, c1);
                sreg[j] -= c0;
                sreg[j + 1] -= c1;
            }
            if constexpr (staged_epilogue<MODE>()) {
                if (p.bulk_epi && !part) {
                    // Each warp stages its 32 rows of EPI_COLS columns at a
                    // time (a column's rows contiguous, as in dst) and lane l
                    // copies column l's 32 rows to its dst row with a bulk
                    // copy: the warp needs no other warp, so no barrier.
                    // Rows past M are staged but not copied.
                    float *stg =
                        reinterpret_cast<float *>(epi) + (warp - WARP_FOLD0) * EPI_COLS * 32;
                    const int64_t mrow0 = static_cast<int64_t>(t.mt) * BM + 32 * quad;
                    const int64_t nrows = std::min<int64_t>(32, p.M - mrow0);
                    float *dbase = p.dst + mrow0;
                    if constexpr (!GROUPED)
                        dbase += t.slice * p.N * p.M + static_cast<int64_t>(t.nt) * BN * p.M;
#pragma unroll
                    for (int rd = 0; rd < FOLD_COLS / EPI_COLS; ++rd) {
                        ptx::bulk_wait_read();              // this lane's last copy left the staging
                        __syncwarp();
#pragma unroll
                        for (int pp = 0; pp < EPI_COLS / 16; ++pp) {
                            const int pc = rd * (EPI_COLS / 16) + pp;
                            uint32_t dv[16];
                            ptx::tmem_ld16_wait(tmem + lane_off + COL_D2 + col0 + pc * 16, dv);
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                stg[(pp * 16 + j) * 32 + lane] =
                                    sreg[pc * 16 + j] + (has_d2 ? __uint_as_float(dv[j]) : 0.f);
                        }
                        if (rd == FOLD_COLS / EPI_COLS - 1) {
                            // D2 is read: the next segment's cross terms may start
                            ptx::tc_fence_before();
                            ptx::mbar_arrive(&bars->d2free);
                        }
                        ptx::fence_async_shared();
                        __syncwarp();
                        const int jc = static_cast<int>(col0) + rd * EPI_COLS + lane;
                        if (jc < tile_cols && nrows > 0) {
                            const int64_t drow = GROUPED ? (rd == 0 ? rows_lo : rows_hi) : jc;
                            ptx::bulk_store(dbase + drow * p.M, stg + lane * 32,
                                            static_cast<uint32_t>(nrows) * 4);
                        }
                        ptx::bulk_commit();
                    }
                    continue;
                }
            }
#pragma unroll
            for (int pc = 0; pc < FOLD_COLS / 16; ++pc) {
                const int col = static_cast<int>(col0) + pc * 16;
                uint32_t dv[16];
                __syncwarp();                               // converged for tcgen05.ld
                ptx::tmem_ld16_wait(tmem + lane_off + COL_D2 + col, dv);
                if constexpr (GROUPED) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int rel = pc * 16 + j;        // the thread's column
                        const int drow =
                            __shfl_sync(0xffffffffu, rel < 32 ? rows_lo : rows_hi, rel & 31);
                        const float v = sreg[rel] + (has_d2 ? __uint_as_float(dv[j]) : 0.f);
                        const int jc = col + j;
                        if (m < p.M) {
                            if (part)
                                part[jc * BM] = v;
                            else if (jc < tile_cols)
                                dcol[static_cast<int64_t>(drow) * p.M] = v;
                        }
                    }
                    continue;
                }
                if (m >= p.M) continue;
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    // a one-block segment wrote no D2 (it holds an older one)
                    const float v[2] = {sreg[pc * 16 + j] + (has_d2 ? __uint_as_float(dv[j]) : 0.f),
                                        sreg[pc * 16 + j + 1] +
                                            (has_d2 ? __uint_as_float(dv[j + 1]) : 0.f)};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int jc = col + j + e;         // column in the tile
                        if (part)
                            part[jc * BM] = v[e];
                        else if (jc < tile_cols)
                            dcol[static_cast<int64_t>(jc) * p.M] = v[e];
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bars->d2free);
        }
    }

    // the bulk copies of the last epilogue complete before the CTA exits
    if constexpr (staged_epilogue<MODE>()) {
        if (warp >= WARP_FOLD0) ptx::bulk_wait();
    }
    if (timed_out) record_status(p.status, OOP_ERR_DEVICE_TIMEOUT);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Stream-K fix-up, one CTA per tile: a tile whose iterations belong to two or
// more CTAs gets the sum of their partials, in CTA (= k) order, with a Kahan
// compensation, rounded once.  Tiles owned by one CTA were written by it and
// are skipped.
// Sums the partials of the tiles that several CTAs share, in CTA (= k) order
// with a Kahan compensation, and writes them to dst.  Two forms:
//  * EPT = FIX_CHUNKS, BATCH = 1: one CTA per tile, EPT elements per thread,
//    for tiles shared by a few CTAs (each partial read once, coalesced);
//  * EPT = 1, BATCH = FIX_BATCH: grid (tiles, FIX_CHUNKS), one element per
//    thread, the partials read BATCH at a time (independent loads in flight
//    together), for tiles shared by many CTAs (long K on few tiles), where
//    the first form is a long chain of dependent loads on a few SMs.
// Both add the same partials in the same order: the results are identical.
constexpr int FIX_THREADS = 256;
constexpr int FIX_CHUNKS = BM * BN / FIX_THREADS;
constexpr int FIX_BATCH = 8;
static_assert(BM * BN % FIX_THREADS == 0, "fix-up tiling");

template <bool GROUPED, int EPT, int BATCH>
__global__ void __launch_bounds__(FIX_THREADS) sk_fixup_kernel(const float *__restrict__ partial,
                                                               const TcParams p, int64_t t_first) {
    const int64_t t = t_first + blockIdx.x;
    const int64_t tiles = GROUPED ? static_cast<int64_t>(p.mtiles) * *p.grp_ntiles
                                  : p.iters / p.num_kb;
    // the full waves are whole tiles, written by their CTAs; only the tail
    // tiles' iterations were split (the tile kernel's stream-K span)
    const int64_t dp_tiles = tiles / p.ctas * p.ctas;
    if (t >= tiles || t < dp_tiles) return;
    const int64_t iters = (tiles - dp_tiles) * p.num_kb;
    const int64_t x0 = (t - dp_tiles) * p.num_kb, x1 = x0 + p.num_kb - 1;
    const int64_t c0 = sk_owner(iters, p.ctas, x0), c1 = sk_owner(iters, p.ctas, x1);
    if (c0 == c1) return;
    // this thread's elements of the tile: e0 + j * FIX_THREADS, j < EPT
    const int e0 = static_cast<int>(blockIdx.y) * EPT * FIX_THREADS + threadIdx.x;
    float sum[EPT], cmp[EPT];
#pragma unroll
    for (int j = 0; j < EPT; ++j) sum[j] = cmp[j] = 0.f;
    int64_t b_next = sk_begin(iters, p.ctas, c0);
    for (int64_t cb = c0; cb <= c1; cb += BATCH) {
        float v[BATCH][EPT];
        bool use[BATCH];
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
            const int64_t c = cb + i;
            use[i] = false;
            if (c <= c1) {
                const int64_t b0 = b_next;
                b_next = sk_begin(iters, p.ctas, c + 1);
                if (b0 != b_next) {                    // a CTA with iterations
                    // CTA c's segment of this tile is its first (slot 0) if it
                    // starts in it
                    const int slot = b0 >= x0 ? 0 : 1;
                    const float *src = partial + (c * 2 + slot) * (BM * BN) + e0;
#pragma unroll
                    for (int j = 0; j < EPT; ++j) v[i][j] = __ldg(src + j * FIX_THREADS);
                    use[i] = true;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
            if (!use[i]) continue;
#pragma unroll
            for (int j = 0; j < EPT; ++j) {
                const float y = v[i][j] - cmp[j];
                const float s2 = sum[j] + y;
                cmp[j] = (s2 - sum[j]) - y;
                sum[j] = s2;
            }
        }
    }
    const Tile d = decode_tile<GROUPED ? kModeGrouped : kModePlain>(p, t);
    const int64_t tile_cols = d.ncols - static_cast<int64_t>(d.nt) * BN;
    float *out = GROUPED ? p.dst : p.dst + d.slice * p.N * p.M;
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        const int e = e0 + j * FIX_THREADS;
        const int64_t m = static_cast<int64_t>(d.mt) * BM + e % BM;
        const int64_t col = e / BM;                               // column in the tile
        if (m >= p.M || col >= tile_cols) continue;
        const int64_t row = GROUPED ? p.grp_rows[d.brow0 + col]
                                    : static_cast<int64_t>(d.nt) * BN + col;
        out[row * p.M + m] = sum[j] - cmp[j];
    }
}

// The fix-up for tiles t_first .. t_first + count - 1: the tail after the
// full waves (an upper bound, from 0, for the grouped product, whose tile
// count is on the device); the per-element form once a tile has about four
// partials or more.
template <bool GROUPED>
void launch_fixup(const float *partial, const TcParams &p, int64_t t_first, int64_t count,
                  cudaStream_t stream) {
    if (count <= 0) return;
    if (p.ctas >= 4 * count)
        sk_fixup_kernel<GROUPED, 1, FIX_BATCH>
            <<<dim3(static_cast<unsigned>(count), FIX_CHUNKS), FIX_THREADS, 0, stream>>>(partial, p,
                                                                                       t_first);
    else
        sk_fixup_kernel<GROUPED, FIX_CHUNKS, 1>
            <<<static_cast<unsigned>(count), FIX_THREADS, 0, stream>>>(partial, p, t_first);
}

// b[slice][k][n] (n fastest) -> bhi, blo [slice][n][Kp] (k fastest), TF32
// split, zero padding for k in [K, Kp).  64 k x 64 n per CTA through shared
// memory; two consecutive n per thread on the way in (when N is even), two
// consecutive k per thread (8-byte stores) on the way out.
constexpr int kSplitTile = 64;

// The output half shared by both split passes: tile[k][n] (64 x 64, k0, n0)
// -> bhi, blo [slice][n][Kp], two consecutive k per thread (8-byte stores).
__device__ __forceinline__ void store_split_tile(const float (&tile)[kSplitTile][kSplitTile + 1],
                                                 uint32_t *__restrict__ bhi,
                                                 uint32_t *__restrict__ blo, int64_t slice,
                                                 int64_t k0, int64_t n0, int64_t N, int64_t Kp) {
    const int tx = threadIdx.x, ty = threadIdx.y;           // 32 x 8
#pragma unroll
    for (int i = ty; i < kSplitTile; i += 8) {
        const int64_t n = n0 + i, k = k0 + 2 * tx;          // Kp is a multiple of 4
        if (n < N && k < Kp) {
            uint32_t h0, l0, h1, l1;
            ptx::split_tf32(tile[2 * tx][i], h0, l0);
            ptx::split_tf32(tile[2 * tx + 1][i], h1, l1);
            const int64_t o = (slice * N + n) * Kp + k;
            *reinterpret_cast<uint2 *>(bhi + o) = make_uint2(h0, h1);
            *reinterpret_cast<uint2 *>(blo + o) = make_uint2(l0, l1);
        }
    }
}

// The split of a strided src1 view (element strides s0 for n, s1 for k, s2,
// s3 for the slice indices).  When k is the contiguous index (s1 == 1: the
// transposed gradient dy^T of a MUL_MAT backward), lanes read along k, so
// each warp reads 128 contiguous bytes per row; otherwise along n.  Zero
// padding for k in [K, Kp) as in bsplit_kernel.
__global__ void __launch_bounds__(256) bsplit_strided_kernel(
    const float *__restrict__ b, uint32_t *__restrict__ bhi, uint32_t *__restrict__ blo,
    int64_t K, int64_t N, int64_t Kp, int64_t ne12, int64_t s0, int64_t s1, int64_t s2,
    int64_t s3) {
    __shared__ float tile[kSplitTile][kSplitTile + 1];      // [k][n]
    const int64_t slice = blockIdx.z;
    const float *bs = b + (slice % ne12) * s2 + (slice / ne12) * s3;
    const int64_t k0 = static_cast<int64_t>(blockIdx.x) * kSplitTile;
    const int64_t n0 = static_cast<int64_t>(blockIdx.y) * kSplitTile;
    const int tx = threadIdx.x, ty = threadIdx.y;           // 32 x 8
    if (s1 == 1) {
#pragma unroll 4
        for (int i = ty; i < kSplitTile; i += 8) {          // i: n offset
            const int64_t n = n0 + i;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t k = k0 + tx + 32 * h;
                tile[tx + 32 * h][i] = (n < N && k < K) ? __ldg(bs + n * s0 + k) : 0.f;
            }
        }
    } else {
#pragma unroll 4
        for (int i = ty; i < kSplitTile; i += 8) {          // i: k offset
            const int64_t k = k0 + i;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t n = n0 + tx + 32 * h;
                tile[i][tx + 32 * h] = (n < N && k < K) ? __ldg(bs + n * s0 + k * s1) : 0.f;
            }
        }
    }
    __syncthreads();
    store_split_tile(tile, bhi, blo, slice, k0, n0, N, Kp);
    ptx::griddep_launch_dependents();   // as in bsplit_kernel
}

__global__ void __launch_bounds__(256) bsplit_kernel(const float *__restrict__ b,
                                                     uint32_t *__restrict__ bhi,
                                                     uint32_t *__restrict__ blo, int64_t K,
                                                     int64_t N, int64_t Kp) {
    __shared__ float tile[kSplitTile][kSplitTile + 1];      // [k][n]
    const int64_t slice = blockIdx.z;
    const int64_t k0 = static_cast<int64_t>(blockIdx.x) * kSplitTile;
    const int64_t n0 = static_cast<int64_t>(blockIdx.y) * kSplitTile;
    const float *bs = b + slice * K * N;
    const int tx = threadIdx.x, ty = threadIdx.y;           // 32 x 8
    const bool pairs = (N % 2 == 0) && (reinterpret_cast<uintptr_t>(b) % 8 == 0);
#pragma unroll
    for (int i = ty; i < kSplitTile; i += 8) {
        const int64_t k = k0 + i, n = n0 + 2 * tx;
        float v0 = 0.f, v1 = 0.f;
        if (k < K) {
            if (pairs && n + 1 < N) {
                const float2 t = __ldg(reinterpret_cast<const float2 *>(bs + k * N + n));
                v0 = t.x;
                v1 = t.y;
            } else {
                if (n < N) v0 = __ldg(bs + k * N + n);
                if (n + 1 < N) v1 = __ldg(bs + k * N + n + 1);
            }
        }
        tile[i][2 * tx] = v0;
        tile[i][2 * tx + 1] = v1;
    }
    __syncthreads();
    store_split_tile(tile, bhi, blo, slice, k0, n0, N, Kp);
    // the tile kernel after this one may start launching (it waits for this
    // grid to complete before it reads bhi / blo)
    ptx::griddep_launch_dependents();
}

// ---- MoE routing (MUL_MAT_ID_BACK and the expert-weight gradient) ----------
// Both lay the routed slots out sorted by expert in one CTA.  The weight
// gradient sums over each expert's slots, so there the sort is a stable
// counting sort: each expert's slots land in ascending slot order, and the
// order of every such sum is the same in every run.  MUL_MAT_ID_BACK computes
// every slot's dx row alone, so any order gives the same bits and its slots
// are placed by atomic cursors (faster).  Shared memory: [E] counts, [E]
// cursors, then (stable sort) [warps][E] counts of one batch of blockDim slots.
constexpr int kRouteSmemInts = 232448 / 4;

// Threads of a routing CTA for E experts (its shared memory must hold
// (2 + warps) * E ints), 0 when E is too large.
int route_threads(int64_t E) {
    const int64_t warps = std::min<int64_t>(32, kRouteSmemInts / std::max<int64_t>(E, 1) - 2);
    return warps >= 1 ? static_cast<int>(warps) * 32 : 0;
}
size_t route_smem_bytes(int64_t E, int threads) {
    return static_cast<size_t>(2 + threads / 32) * static_cast<size_t>(E) * sizeof(int);
}

// Adds every valid slot's expert to cnt[]; ids are read four batches at a
// time so that their loads are in flight together.  Returns nothing; a slot
// whose id is outside [0, E) is passed to bad(s).
template <typename Bad>
__device__ __forceinline__ void route_count(const int32_t *__restrict__ ids, int64_t nslot, int E,
                                            int *cnt, Bad bad) {
    for (int64_t s0 = threadIdx.x; s0 < nslot; s0 += 4 * static_cast<int64_t>(blockDim.x)) {
        int e4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t s = s0 + u * static_cast<int64_t>(blockDim.x);
            e4[u] = s < nslot ? ids[s] : 0;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t s = s0 + u * static_cast<int64_t>(blockDim.x);
            if (s >= nslot) break;
            if (e4[u] >= 0 && e4[u] < E) atomicAdd(&cnt[e4[u]], 1);
            else bad(s);
        }
    }
}

// rows[cur[e] + (rank of slot s among expert e's slots)] = s, for every valid
// slot, in slot order: batches of blockDim slots, ranked inside a warp by
// __match_any_sync and across warps by the batch's per-warp counts.  cur[]
// ends past each expert's slots.  Called by the whole CTA.
__device__ __forceinline__ void route_place(const int32_t *__restrict__ ids, int64_t nslot, int E,
                                            int *cur, int *wc, int *rows) {
    const int nw = static_cast<int>(blockDim.x >> 5);
    const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
    int e_next = threadIdx.x < nslot ? ids[threadIdx.x] : -1;
    for (int64_t base = 0; base < nslot; base += blockDim.x) {
        const int64_t s = base + threadIdx.x;
        const int e = e_next;
        const int64_t sn = s + blockDim.x;
        e_next = sn < nslot ? ids[sn] : -1;         // the next batch's id, in flight meanwhile
        const bool ok = s < nslot && e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        for (int i = static_cast<int>(threadIdx.x); i < nw * E; i += static_cast<int>(blockDim.x))
            wc[i] = 0;
        __syncthreads();
        if (ok && rank == 0) wc[warp * E + e] = __popc(peers);
        __syncthreads();
        if (ok) {
            int pos = cur[e] + rank;
            for (int w = 0; w < warp; ++w) pos += wc[w * E + e];
            rows[pos] = static_cast<int>(s);
        }
        __syncthreads();
        for (int x = static_cast<int>(threadIdx.x); x < E; x += static_cast<int>(blockDim.x)) {
            int t = 0;
            for (int w = 0; w < nw; ++w) t += wc[w * E + x];
            cur[x] += t;
        }
        __syncthreads();
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
    route_count(ids, nslot, E, cnt, [&](int64_t s) {
        record_status(status, OOP_ERR_BAD_ID);
        for (int64_t k = 0; k < Kw; ++k) dx[s * Kw + k] = 0.f;
    });
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

// Sorted slots j, one warp each (kSplitSlots per CTA): g[rows[j]][0..R) ->
// ghi, glo [j][Kp], TF32 split, zero padding for r in [R, Kp).  With `vec`
// (R a multiple of 4, 16-byte aligned rows) each lane moves four words at a
// time.  Rows past the routed total are left alone: the tile kernel never
// stores the columns they feed.
constexpr int kSplitSlots = 8;

__global__ void __launch_bounds__(32 * kSplitSlots) mmid_gsplit_kernel(
    const float *__restrict__ g, const int *__restrict__ rows, const int *__restrict__ count,
    int E, uint32_t *__restrict__ ghi, uint32_t *__restrict__ glo, int64_t R, int64_t Kp,
    bool vec) {
    __shared__ int total;
    if (threadIdx.x == 0) {
        int t = 0;
        for (int e = 0; e < E; ++e) t += count[e];
        total = t;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kSplitSlots + (threadIdx.x >> 5);
    if (j < total) {
        const float *src = g + static_cast<int64_t>(rows[j]) * R;
        uint32_t *dh = ghi + j * Kp, *dl = glo + j * Kp;
        if (vec) {
            for (int64_t r = 4 * lane; r < Kp; r += 128) {
                uint4 h = make_uint4(0, 0, 0, 0), l = make_uint4(0, 0, 0, 0);
                if (r < R) {
                    const float4 v = __ldg(reinterpret_cast<const float4 *>(src + r));
                    ptx::split_tf32(v.x, h.x, l.x);
                    ptx::split_tf32(v.y, h.y, l.y);
                    ptx::split_tf32(v.z, h.z, l.z);
                    ptx::split_tf32(v.w, h.w, l.w);
                }
                *reinterpret_cast<uint4 *>(dh + r) = h;
                *reinterpret_cast<uint4 *>(dl + r) = l;
            }
        } else {
            for (int64_t r = lane; r < Kp; r += 32) {
                uint32_t h = 0, l = 0;
                if (r < R) ptx::split_tf32(__ldg(src + r), h, l);
                dh[r] = h;
                dl[r] = l;
            }
        }
    }
    ptx::griddep_launch_dependents();   // as in bsplit_kernel
}

// ---- MUL_MAT_ID's expert-weight gradient as a segmented product ------------
// dW_e = sum over the slots routed to e of x_slot (x) dy_slot: OUT_PROD per
// expert whose reduction runs over that expert's slots.  The slots are sorted
// by expert into segments rounded up to whole k-blocks (padding rows are zero
// on both sides, and an expert with no slot gets one block of padding, so its
// dW comes out zero); the tile kernel's segmented mode then gives slice e the
// k range of segment e.  Segment starts are multiples of 32, which keeps every
// TMA x coordinate of the split gradient 16-byte aligned.

// Routing, one CTA: per-expert counts, segment offsets and k-block counts,
// and the sorted-slot list (-1 at padding).  Slots with an id outside [0, E)
// take part in no segment and set OOP_ERR_BAD_ID.
__global__ void __launch_bounds__(1024) wgrad_route_kernel(const int32_t *__restrict__ ids,
                                                           int64_t nslot, int E,
                                                           int64_t rows_max, int *seg_off,
                                                           int *seg_nkb, int *total, int *rows,
                                                           int *status) {
    extern __shared__ int sh[];                   // [E] counts, [E] cursors, [warps][E]
    int *cnt = sh, *cur = sh + E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    for (int64_t j = threadIdx.x; j < rows_max; j += blockDim.x) rows[j] = -1;
    __syncthreads();
    route_count(ids, nslot, E, cnt, [&](int64_t) { record_status(status, OOP_ERR_BAD_ID); });
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int e = 0; e < E; ++e) {
            const int nkb = cnt[e] > 0 ? (cnt[e] + BK - 1) / BK : 1;
            seg_off[e] = acc;
            seg_nkb[e] = nkb;
            cur[e] = acc;
            acc += nkb * BK;
        }
        *total = acc;
    }
    __syncthreads();
    route_place(ids, nslot, E, cur, sh + 2 * E, rows);
}

// Sorted slot j (one per CTA) -> xg[j][0..K) = x[., i % n_x, t] of slot
// s = t * n_used + i, zero at padding.  Rows past the routed total are never
// read and are left alone.
__global__ void __launch_bounds__(256) wgrad_gather_kernel(const float *__restrict__ x,
                                                           const int *__restrict__ rows,
                                                           const int *__restrict__ total,
                                                           float *__restrict__ xg, int64_t K,
                                                           int64_t n_x, int64_t n_used) {
    const int64_t j = blockIdx.x;
    if (j >= *total) return;
    const int s = rows[j];
    float *dst = xg + j * K;
    if (s < 0) {
        for (int64_t k = threadIdx.x; k < K; k += blockDim.x) dst[k] = 0.f;
        return;
    }
    const float *src = x + ((s / n_used) * n_x + (s % n_used) % n_x) * K;
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) dst[k] = __ldg(src + k);
}

// bhi, blo [r][j] (j fastest, row length Kp) = TF32 split of dy[r] of sorted
// slot j, zero at padding: 64 j x 64 r per CTA through shared memory, read
// along r, written along j.
__global__ void __launch_bounds__(256) wgrad_dysplit_kernel(const float *__restrict__ dy,
                                                            const int *__restrict__ rows,
                                                            const int *__restrict__ total,
                                                            uint32_t *__restrict__ bhi,
                                                            uint32_t *__restrict__ blo,
                                                            int64_t N, int64_t Kp) {
    __shared__ float tile[kSplitTile][kSplitTile + 1];      // [j][r]
    const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kSplitTile;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kSplitTile;
    const int64_t tot = *total;
    if (j0 >= tot) return;
    const int tx = threadIdx.x, ty = threadIdx.y;           // 32 x 8
    for (int i = ty; i < kSplitTile; i += 8) {
        const int64_t j = j0 + i;
        const int s = j < tot ? rows[j] : -1;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t r = r0 + tx + 32 * h;
            tile[i][tx + 32 * h] = (s >= 0 && r < N) ? __ldg(dy + static_cast<int64_t>(s) * N + r)
                                                     : 0.f;
        }
    }
    __syncthreads();
    store_split_tile(tile, bhi, blo, 0, j0, r0, N, Kp);
    ptx::griddep_launch_dependents();   // as in bsplit_kernel
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() { return tensor_map_encoder(); }

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
bool make_a_map(CUtensorMap *map, const void *base, const OutProdShape &s, int rg) {
    auto fn = encode_fn();
    if (!fn) return false;
    // map rows: groups of rg src0 rows (rg = 1: the rows themselves)
    const int64_t rows = s.K * s.ne02 * s.ne03 / rg;
    cuuint32_t box[2] = {static_cast<cuuint32_t>(RawA<TYPE>::BOX_X),
                         static_cast<cuuint32_t>(BK / rg)};
    cuuint32_t estr[2] = {1, 1};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(s.a_row_bytes * rg)};
    if constexpr (elementwise_type<TYPE>()) {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(s.M), static_cast<cuuint64_t>(rows)};
        const CUtensorMapDataType dt = TYPE == OOP_TYPE_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                             : CU_TENSOR_MAP_DATA_TYPE_UINT16;
        return fn(map, dt, 2, const_cast<void *>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    } else {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(s.a_row_bytes * rg),
                              static_cast<cuuint64_t>(rows)};
        return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
}

int64_t padded_k(int64_t K) { return (K + 3) / 4 * 4; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// test hooks, set from any host thread
std::atomic<int> g_inject{0};     // the next launch drops one TMA stage
std::atomic<int> g_schedule{0};   // 0 automatic, 1 data-parallel, 2 stream-K
thread_local cudaEvent_t g_ev_before = nullptr, g_ev_after = nullptr;

// Stream-K uses at most this many CTAs (one per SM); its partial slots are
// part of the workspace.
constexpr int kSkMaxCtas = 160;
constexpr size_t kSlotBytes = size_t(BM) * BN * 4;

int device_sms() { return device_sm_count(); }

// Stream-K or data-parallel for `tiles` tiles of `num_kb` k-blocks on `sms`
// SMs.  Returns the stream-K CTA count, 0 for data-parallel.  Stream-K pays
// when the last data-parallel wave would run mostly empty; each CTA then
// costs about eight k-blocks more (partial stores and the fix-up).
int plan_ctas(int64_t tiles, int num_kb, int sms, size_t partial_room) {
    const int64_t iters = tiles * num_kb;
    const int G = static_cast<int>(std::min<int64_t>(std::min(sms, kSkMaxCtas), iters));
    // whole waves only: the stream-K span would be the data-parallel schedule
    if (G <= 0 || g_schedule == 1 || tiles % G == 0 ||
        partial_room < static_cast<size_t>(G) * 2 * kSlotBytes)
        return 0;
    if (g_schedule == 2) return G;
    // in k-block times: data-parallel waves x the k-blocks of a tile, against
    // an even share of the iterations plus the fix-up launch (~8) and the
    // partials of the split tail tiles (~6 per two of them a CTA)
    const int64_t dp = (tiles + G - 1) / G * num_kb;
    const int64_t tail = tiles % G;
    const int64_t sk = (iters + G - 1) / G + 8 + 6 * ((2 * tail + G - 1) / G);
    return sk < dp ? G : 0;
}

template <int TYPE, int MODE>
cudaError_t launch_typed(const void *a, const OutProdShape &s, const CUtensorMap &mhi,
                         const CUtensorMap &mlo, const TcParams &p, dim3 grid,
                         cudaStream_t stream) {
    // TMA needs a 16-byte aligned base and row stride, and rows that fit
    // int32.  Rows of another length are staged in groups of RawA::RG (whose
    // length always is a multiple of 16) when every k-block starts a group:
    // K a multiple of RG, a src0 slice per tile (not the segmented mode).
    constexpr int RG = RawA<TYPE>::RG;
    const bool tma_ok = reinterpret_cast<uintptr_t>(a) % 16 == 0 &&
                        s.K * s.ne02 * s.ne03 < (1LL << 31);
    // the smallest group whose bytes are a multiple of 16 (1: the rows are)
    int group = 1;
    while ((s.a_row_bytes * group) % 16 != 0) group *= 2;
    int ag = 0;
    if (tma_ok && group == 1)
        ag = 1;
    else if (tma_ok && MODE != kModeSegmented && RG % group == 0 && s.K % group == 0)
        ag = group;
    CUtensorMap ma;
    if (ag > 0) {
        if (!make_a_map<TYPE>(&ma, a, s, ag)) return cudaErrorInvalidValue;
    } else {
        ma = mhi;   // unused by the kernel
    }
    constexpr size_t smem = smem_bytes<TYPE, MODE>();
    static_assert(smem <= 232448, "shared memory budget");
    auto run = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        // the kernel's register split hands out exactly what a block of
        // MAX_REGS-register threads holds: any other launch count is refused
        cudaFuncAttributes fa;
        if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
        if (fa.numRegs != MAX_REGS) return cudaErrorInvalidConfiguration;
        cudaEvent_t before = g_ev_before, after = g_ev_after;
        g_ev_before = g_ev_after = nullptr;
        if (before && (e = cudaEventRecord(before, stream)) != cudaSuccess) return e;
        // a programmatic dependent of the split pass launched just before it
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t le = cudaLaunchKernelEx(&cfg, kern, mhi, mlo, ma, p);
        if (le != cudaSuccess) return le;
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        ++g_kernel_launches;
        if (after && (e = cudaEventRecord(after, stream)) != cudaSuccess) return e;
        return cudaSuccess;
    };
    if (ag == 1) return run(tc_out_prod_kernel<TYPE, 1, MODE>);
    if constexpr (MODE != kModeSegmented) {
        if constexpr (RG >= 2)
            if (ag == 2) return run(tc_out_prod_kernel<TYPE, 2, MODE>);
        if constexpr (RG >= 4)
            if (ag == 4) return run(tc_out_prod_kernel<TYPE, 4, MODE>);
        if constexpr (RG >= 8)
            if (ag == 8) return run(tc_out_prod_kernel<TYPE, 8, MODE>);
    }
    return run(tc_out_prod_kernel<TYPE, 0, MODE>);
}

size_t split_bytes(const OutProdShape &s) {
    return align256(static_cast<size_t>(s.ne12 * s.ne13) * static_cast<size_t>(s.N) *
                    static_cast<size_t>(padded_k(s.K)) * 4);
}

int64_t tile_count(const OutProdShape &s) {
    return ((s.M + BM - 1) / BM) * ((s.N + BN - 1) / BN) * s.ne12 * s.ne13;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

void tc_set_inject(int v) { g_inject = v; }
void tc_set_schedule(int v) { g_schedule = v; }
void tc_set_profile_events(cudaEvent_t before, cudaEvent_t after) {
    g_ev_before = before;
    g_ev_after = after;
}

size_t tc_workspace_min_bytes(const OutProdShape &s) { return 2 * split_bytes(s); }

int tc_plan_ctas(const OutProdShape &s, int sms, size_t workspace_bytes) {
    const int64_t num_kb = (s.K + BK - 1) / BK;
    if (num_kb <= 0 || num_kb > 0x7fffffffLL) return 0;
    const size_t split = 2 * split_bytes(s);
    const size_t room = workspace_bytes > split ? workspace_bytes - split : 0;
    return plan_ctas(tile_count(s), static_cast<int>(num_kb), sms, room);
}

size_t tc_workspace_bytes(const OutProdShape &s) {
    const int64_t iters = tile_count(s) * ((s.K + BK - 1) / BK);
    const int64_t ctas = std::min<int64_t>(kSkMaxCtas, iters);
    return tc_workspace_min_bytes(s) + static_cast<size_t>(std::max<int64_t>(ctas, 0)) * 2 * kSlotBytes;
}

cudaError_t launch_dense_tc(const void *a, const float *b, float *dst, const OutProdShape &s,
                            void *workspace, size_t workspace_bytes, int *status,
                            cudaStream_t stream) {
    const int64_t slices = s.ne12 * s.ne13;
    const int64_t Kp = padded_k(s.K);
    const size_t one = split_bytes(s);
    uint32_t *bhi = static_cast<uint32_t *>(workspace);
    uint32_t *blo = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(workspace) + one);
    float *partial = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + 2 * one);

    const int64_t gk = (Kp + kSplitTile - 1) / kSplitTile, gn = (s.N + kSplitTile - 1) / kSplitTile;
    if (gk > 0x7fffffffLL || gn > 65535 || slices > 65535) return cudaErrorInvalidConfiguration;
    const dim3 sgrid(static_cast<unsigned>(gk), static_cast<unsigned>(gn),
                     static_cast<unsigned>(slices));
    if (s.b_strided)
        bsplit_strided_kernel<<<sgrid, dim3(32, 8), 0, stream>>>(
            b, bhi, blo, s.K, s.N, Kp, s.ne12, s.bs[0], s.bs[1], s.bs[2], s.bs[3]);
    else
        bsplit_kernel<<<sgrid, dim3(32, 8), 0, stream>>>(b, bhi, blo, s.K, s.N, Kp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ++g_kernel_launches;

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
    p.mtiles = static_cast<int>(mtiles);
    p.ntiles = static_cast<int>(ntiles);
    p.inject = g_inject.exchange(0);
    const int64_t tiles = mtiles * ntiles * slices;
    p.ctas = tc_plan_ctas(s, device_sms(), workspace_bytes);
    p.iters = tiles * p.num_kb;
    p.partial = partial;
    const dim3 grid = p.ctas > 0 ? dim3(static_cast<unsigned>(p.ctas))
                                 : dim3(static_cast<unsigned>(mtiles * ntiles),
                                        static_cast<unsigned>(slices));

    switch (s.a_type) {
#define OOP_TC_CASE(T) \
    case T: e = launch_typed<T, kModePlain>(a, s, mhi, mlo, p, grid, stream); break;
    OOP_TC_CASE(OOP_TYPE_F32)
    OOP_TC_CASE(OOP_TYPE_F16)
    OOP_TC_CASE(OOP_TYPE_BF16)
    OOP_TC_CASE(OOP_TYPE_Q4_0)
    OOP_TC_CASE(OOP_TYPE_Q4_1)
    OOP_TC_CASE(OOP_TYPE_Q5_0)
    OOP_TC_CASE(OOP_TYPE_Q5_1)
    OOP_TC_CASE(OOP_TYPE_Q8_0)
    OOP_TC_CASE(OOP_TYPE_Q2_K)
    OOP_TC_CASE(OOP_TYPE_Q3_K)
    OOP_TC_CASE(OOP_TYPE_Q4_K)
    OOP_TC_CASE(OOP_TYPE_Q5_K)
    OOP_TC_CASE(OOP_TYPE_Q6_K)
#undef OOP_TC_CASE
    default:
        return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess || p.ctas == 0) return e;
    if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    launch_fixup<false>(partial, p, tiles / p.ctas * p.ctas, tiles % p.ctas, stream);
    e = cudaGetLastError();
    if (e == cudaSuccess) ++g_kernel_launches;
    return e;
}

// ---- MUL_MAT_ID_BACK launcher ------------------------------------------------

namespace {

struct MmidPlan {
    int64_t nslot, Kp, max_tiles, mtiles;
    size_t off_count, off_offset, off_ntiles, off_tiles, off_rows, off_ghi, off_glo, off_part,
        total;
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
    t.off_part = take(static_cast<size_t>(kSkMaxCtas) * 2 * kSlotBytes);   // stream-K partials
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
    ++g_kernel_launches;
    const bool vec = s.N % 4 == 0 && reinterpret_cast<uintptr_t>(g) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(ghi) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(glo) % 16 == 0 && t.Kp % 4 == 0;
    mmid_gsplit_kernel<<<static_cast<unsigned>((t.nslot + kSplitSlots - 1) / kSplitSlots),
                         32 * kSplitSlots, 0, stream>>>(
        g, rw.rows, rw.count, static_cast<int>(s.E), ghi, glo, s.N, t.Kp, vec);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ++g_kernel_launches;

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
    os.a_row_bytes = s.K / type_block_elems(s.w_type) * type_block_bytes(s.w_type);

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
    p.mtiles = static_cast<int>(t.mtiles);
    p.ntiles = 0;
    p.inject = 0;
    p.grp_count = rw.count;
    p.grp_offset = rw.offset;
    p.grp_rows = rw.rows;
    p.grp_tiles = rw.tiles;
    p.grp_ntiles = rw.ntiles;
    p.bulk_epi = p.M % 4 == 0 && reinterpret_cast<uintptr_t>(dx) % 16 == 0;
    // The work list is only known on the device, so the schedule is chosen
    // here: stream-K (one CTA per SM walking the (tile, k-block) iterations
    // the device computes from the list's length) unless data-parallel is
    // forced by the test hook.  Experts' tiles are short in k (K = N of W),
    // so a persistent CTA that flows from one tile into the next saves most
    // of each tile's start-up.
    const int G = std::min(device_sms(), kSkMaxCtas);
    p.ctas = (g_schedule == 2 && G > 0) ? G : 0;
    p.persistent = (g_schedule == 0 && G > 0) ? 1 : 0;
    p.partial = reinterpret_cast<float *>(ws + t.off_part);
    const int64_t max_grid = t.mtiles * t.max_tiles;
    const dim3 grid(static_cast<unsigned>(p.ctas > 0 || p.persistent ? G : max_grid));
    switch (s.w_type) {
#define OOP_TC_CASE(T) \
    case T: e = launch_typed<T, kModeGrouped>(W, os, mhi, mlo, p, grid, stream); break;
    OOP_TC_CASE(OOP_TYPE_F32)
    OOP_TC_CASE(OOP_TYPE_F16)
    OOP_TC_CASE(OOP_TYPE_BF16)
    OOP_TC_CASE(OOP_TYPE_Q4_0)
    OOP_TC_CASE(OOP_TYPE_Q4_1)
    OOP_TC_CASE(OOP_TYPE_Q5_0)
    OOP_TC_CASE(OOP_TYPE_Q5_1)
    OOP_TC_CASE(OOP_TYPE_Q8_0)
    OOP_TC_CASE(OOP_TYPE_Q2_K)
    OOP_TC_CASE(OOP_TYPE_Q3_K)
    OOP_TC_CASE(OOP_TYPE_Q4_K)
    OOP_TC_CASE(OOP_TYPE_Q5_K)
    OOP_TC_CASE(OOP_TYPE_Q6_K)
#undef OOP_TC_CASE
    default:
        return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess || p.ctas == 0) return e;
    launch_fixup<true>(p.partial, p, 0, max_grid, stream);
    e = cudaGetLastError();
    if (e == cudaSuccess) ++g_kernel_launches;
    return e;
}

// ---- the expert-weight gradient launcher ------------------------------------

namespace {

struct WgradPlan {
    int64_t nslot, rows_max, Kp;
    size_t off_seg_off, off_seg_nkb, off_total, off_rows, off_xg, off_bhi, off_blo, total;
};

WgradPlan plan_wgrad(const WgradShape &s) {
    WgradPlan t = {};
    t.nslot = s.n_used * s.n_tok;
    t.rows_max = t.nslot + static_cast<int64_t>(BK) * s.E;      // at most one block of padding each
    t.Kp = padded_k(t.rows_max);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += align256(bytes);
        return at;
    };
    t.off_seg_off = take(sizeof(int) * static_cast<size_t>(s.E));
    t.off_seg_nkb = take(sizeof(int) * static_cast<size_t>(s.E));
    t.off_total = take(sizeof(int));
    t.off_rows = take(sizeof(int) * static_cast<size_t>(t.rows_max));
    t.off_xg = take(4 * static_cast<size_t>(t.rows_max) * static_cast<size_t>(s.K));
    t.off_bhi = take(4 * static_cast<size_t>(s.N) * static_cast<size_t>(t.Kp));
    t.off_blo = take(4 * static_cast<size_t>(s.N) * static_cast<size_t>(t.Kp));
    t.total = o;
    return t;
}

}  // namespace

size_t tc_wgrad_workspace_bytes(const WgradShape &s) { return plan_wgrad(s).total; }

cudaError_t launch_mmid_wgrad(const float *x, const int32_t *ids, const float *dy, float *dW,
                              const WgradShape &s, void *workspace, int *status,
                              cudaStream_t stream) {
    const WgradPlan t = plan_wgrad(s);
    const int64_t mtiles = (s.K + BM - 1) / BM, ntiles = (s.N + BN - 1) / BN;
    if (s.E < 1 || s.E > 65535 || t.rows_max > 0x7fffffffLL || mtiles * ntiles > 0x7fffffffLL ||
        (t.Kp + kSplitTile - 1) / kSplitTile > 0x7fffffffLL || (s.N + kSplitTile - 1) / kSplitTile > 65535)
        return cudaErrorInvalidConfiguration;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int *seg_off = reinterpret_cast<int *>(ws + t.off_seg_off);
    int *seg_nkb = reinterpret_cast<int *>(ws + t.off_seg_nkb);
    int *total = reinterpret_cast<int *>(ws + t.off_total);
    int *rows = reinterpret_cast<int *>(ws + t.off_rows);
    float *xg = reinterpret_cast<float *>(ws + t.off_xg);
    uint32_t *bhi = reinterpret_cast<uint32_t *>(ws + t.off_bhi);
    uint32_t *blo = reinterpret_cast<uint32_t *>(ws + t.off_blo);

    const int route_thr = route_threads(s.E);
    const size_t route_smem = route_smem_bytes(s.E, route_thr);
    if (route_thr == 0) return cudaErrorInvalidConfiguration;
    if (route_smem > 48 * 1024 &&
        cudaFuncSetAttribute(wgrad_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(route_smem)) != cudaSuccess)
        return cudaErrorInvalidConfiguration;
    wgrad_route_kernel<<<1, route_thr, route_smem, stream>>>(ids, t.nslot, static_cast<int>(s.E),
                                                              t.rows_max, seg_off, seg_nkb, total,
                                                              rows, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ++g_kernel_launches;
    wgrad_gather_kernel<<<static_cast<unsigned>(t.rows_max), 256, 0, stream>>>(
        x, rows, total, xg, s.K, s.n_x, s.n_used);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ++g_kernel_launches;
    wgrad_dysplit_kernel<<<dim3(static_cast<unsigned>((t.Kp + kSplitTile - 1) / kSplitTile),
                                static_cast<unsigned>((s.N + kSplitTile - 1) / kSplitTile)),
                           dim3(32, 8), 0, stream>>>(dy, rows, total, bhi, blo, s.N, t.Kp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ++g_kernel_launches;

    CUtensorMap mhi, mlo;
    if (!make_b_map(&mhi, bhi, t.Kp, s.N, 1) || !make_b_map(&mlo, blo, t.Kp, s.N, 1))
        return cudaErrorInvalidValue;

    // the gathered rows xg [rows_max][K] are src0: M = K, one slice, read by
    // every expert's segment
    OutProdShape os = {};
    os.M = s.K;
    os.K = t.rows_max;
    os.N = s.N;
    os.ne02 = os.ne03 = os.ne13 = 1;
    os.ne12 = s.E;
    os.dps2 = s.E;
    os.dps3 = 1;
    os.a_type = OOP_TYPE_F32;
    os.a_row_bytes = 4 * s.K;

    TcParams p = {};
    p.a = reinterpret_cast<const uint8_t *>(xg);
    p.dst = dW;
    p.status = status;
    p.M = s.K;
    p.K = t.rows_max;          // every row of a segment is data or zero padding
    p.N = s.N;
    p.ne02 = 1;
    p.ne12 = s.E;
    p.dps2 = s.E;
    p.dps3 = 1;
    p.a_row_bytes = os.a_row_bytes;
    p.num_kb = 1;
    p.mtiles = static_cast<int>(mtiles);
    p.ntiles = static_cast<int>(ntiles);
    p.seg_off = seg_off;
    p.seg_nkb = seg_nkb;
    p.bulk_epi = p.M % 4 == 0 && reinterpret_cast<uintptr_t>(dW) % 16 == 0;
    // persistent by default: one CTA per SM takes whole tiles round-robin, so
    // the short tiles (a few k-blocks each) flow into one another; the test
    // hook's data-parallel schedule gives each tile its own CTA
    const int64_t tiles = mtiles * ntiles * s.E;
    const int G = std::min(device_sms(), kSkMaxCtas);
    p.persistent = (g_schedule != 1 && G > 0) ? 1 : 0;
    p.iters = tiles;
    const dim3 grid = p.persistent
                          ? dim3(static_cast<unsigned>(std::min<int64_t>(G, tiles)))
                          : dim3(static_cast<unsigned>(mtiles * ntiles), static_cast<unsigned>(s.E));
    return launch_typed<OOP_TYPE_F32, kModeSegmented>(xg, os, mhi, mlo, p, grid, stream);
}

}  // namespace oop
