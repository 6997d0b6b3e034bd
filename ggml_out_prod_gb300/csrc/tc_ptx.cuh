// tc_ptx.cuh -- inline-PTX wrappers for sm_103a: mbarrier, TMA (bulk tensor
// copies), tcgen05 (TMEM alloc, MMA, commit, ld/st) and the TF32 split.
#pragma once

#include <cuda.h>

#include <cstdint>

namespace oop {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier -------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    // The suspend-time hint lets a waiting thread sleep in hardware (it wakes
    // when the phase completes) instead of re-issuing the test.
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the same condition (no suspension).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with parity `parity` to complete, for at most
// `limit_ns` nanoseconds.  Gives up early when *abort is set (and
// honor_abort).  On running out it sets *abort and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  volatile int *abort, bool honor_abort,
                                                  uint64_t limit_ns, bool *timed_out) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 3) == 0) {
            if (honor_abort && *abort) return false;
            if (globaltimer() - t0 > limit_ns) {
                *abort = 1;
                *timed_out = true;
                return false;
            }
        }
    }
}

// Per-warpgroup register budget (every thread of the warpgroup executes the
// same call): give back down to N registers a thread, or wait for registers
// given back by other warpgroups until N are available.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// True in exactly one active lane of the warp (all lanes must call it).
__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// ---- TMA ------------------------------------------------------------------

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// Untiled bulk copy global -> shared, completing `bytes` on `bar` (both
// addresses 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- tcgen05 ----------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// One 32-k block of the 3xTF32 product, A from tensor memory (lanes 0..127 =
// rows, one 32-bit column per k), B from shared memory (descriptors; +2 is
// 32 bytes along the swizzled k row, i.e. 8 tf32), issued as MMAs of 8 k:
//   for kk = 0..3:  d2 (+)= a_lo * b_hi ; d2 += a_hi * b_lo ; d1 (+)= a_hi * b_hi
// (d2 restarted at kk = 0 when `fresh2`, d1 when `fresh1`).  The "one" form
// puts every product into d, restarted: the eight small cross terms first,
// while d is still ~2^-11 of its final size, then the four big terms.
// The blocks are issued by the lanes with `lead` set (one lane) while every
// lane tests one barrier phase (`tbar` / `tpar`, per lane) in the same
// statement; they return that lane's outcome.  The test sits after the eighth
// MMA (the fifth of the bf16 block): by then the issuing lane is held by the
// tensor core's full queue anyway, and the test's ~100-cycle latency passes
// while the last MMAs are issued, instead of stalling the warp before them.
#define OOP_MMA_PROLOGUE                                                        \
    "{\n\t.reg .pred pl, pok, p1, p2, pt;\n\t"                                  \
    ".reg .b32 a0, a1, a2, a3, l0, l1, l2, l3, okr;\n\t"                         \
    ".reg .b64 h0, h1, h2, h3, o0, o1, o2, o3;\n\t"                             \
    "setp.ne.b32 pl, %1, 0;\n\t"                                                \
    "setp.eq.b32 pt, 0, 0;\n\t"                                                 \
    "mov.b32 a0, %4;\n\tadd.u32 a1, %4, 8;\n\tadd.u32 a2, %4, 16;\n\tadd.u32 a3, %4, 24;\n\t" \
    "mov.b32 l0, %5;\n\tadd.u32 l1, %5, 8;\n\tadd.u32 l2, %5, 16;\n\tadd.u32 l3, %5, 24;\n\t" \
    "mov.b64 h0, %6;\n\tadd.u64 h1, %6, 2;\n\tadd.u64 h2, %6, 4;\n\tadd.u64 h3, %6, 6;\n\t" \
    "mov.b64 o0, %7;\n\tadd.u64 o1, %7, 2;\n\tadd.u64 o2, %7, 4;\n\tadd.u64 o3, %7, 6;\n\t"
#define OOP_MMA_TEST "mbarrier.test_wait.parity.shared::cta.b64 pok, [%2], %3;\n\t"
#define OOP_MMA_EPILOGUE "selp.u32 %0, 1, 0, pok;\n\t}"
#define OOP_MMA(d, a, b, acc) "@pl tcgen05.mma.cta_group::1.kind::tf32 [" d "], [" a "], " b ", %8, " acc ";\n\t"

// the 3xTF32 block (d1 = %9, d2 = %10, fresh1 = %11, fresh2 = %12)
__device__ __forceinline__ uint32_t mma_block_3xtf32_test(uint32_t d1, uint32_t d2, uint32_t ahi,
                                                          uint32_t alo, uint64_t bhi, uint64_t blo,
                                                          uint32_t idesc, uint32_t fresh1,
                                                          uint32_t fresh2, uint32_t lead,
                                                          uint64_t *tbar, uint32_t tpar) {
    uint32_t ok;
    asm volatile(OOP_MMA_PROLOGUE
                 "setp.eq.b32 p1, %11, 0;\n\t"
                 "setp.eq.b32 p2, %12, 0;\n\t"
                 OOP_MMA("%10", "l0", "h0", "p2") OOP_MMA("%10", "a0", "o0", "pt")
                 OOP_MMA("%9", "a0", "h0", "p1") OOP_MMA("%10", "l1", "h1", "pt")
                 OOP_MMA("%10", "a1", "o1", "pt") OOP_MMA("%9", "a1", "h1", "pt")
                 OOP_MMA("%10", "l2", "h2", "pt") OOP_MMA("%10", "a2", "o2", "pt")
                 OOP_MMA_TEST
                 OOP_MMA("%9", "a2", "h2", "pt") OOP_MMA("%10", "l3", "h3", "pt")
                 OOP_MMA("%10", "a3", "o3", "pt") OOP_MMA("%9", "a3", "h3", "pt")
                 OOP_MMA_EPILOGUE
                 : "=r"(ok)
                 : "r"(lead), "r"(smem_u32(tbar)), "r"(tpar), "r"(ahi), "r"(alo), "l"(bhi),
                   "l"(blo), "r"(idesc), "r"(d1), "r"(d2), "r"(fresh1), "r"(fresh2)
                 : "memory");
    return ok;
}

// the "one" form (d = %9)
__device__ __forceinline__ uint32_t mma_block_3xtf32_one_test(uint32_t d, uint32_t ahi,
                                                              uint32_t alo, uint64_t bhi,
                                                              uint64_t blo, uint32_t idesc,
                                                              uint32_t lead, uint64_t *tbar,
                                                              uint32_t tpar) {
    uint32_t ok;
    asm volatile(OOP_MMA_PROLOGUE
                 "setp.ne.b32 p1, 0, 0;\n\t"
                 OOP_MMA("%9", "l0", "h0", "p1") OOP_MMA("%9", "a0", "o0", "pt")
                 OOP_MMA("%9", "l1", "h1", "pt") OOP_MMA("%9", "a1", "o1", "pt")
                 OOP_MMA("%9", "l2", "h2", "pt") OOP_MMA("%9", "a2", "o2", "pt")
                 OOP_MMA("%9", "l3", "h3", "pt") OOP_MMA("%9", "a3", "o3", "pt")
                 OOP_MMA_TEST
                 OOP_MMA("%9", "a0", "h0", "pt") OOP_MMA("%9", "a1", "h1", "pt")
                 OOP_MMA("%9", "a2", "h2", "pt") OOP_MMA("%9", "a3", "h3", "pt")
                 OOP_MMA_EPILOGUE
                 : "=r"(ok)
                 : "r"(lead), "r"(smem_u32(tbar)), "r"(tpar), "r"(ahi), "r"(alo), "l"(bhi),
                   "l"(blo), "r"(idesc), "r"(d)
                 : "memory");
    return ok;
}

// A block whose a_lo is zero (bf16 / f16 src0): the cross term a_hi * b_lo
// into dx (restarted at its first MMA when `freshx`), then a_hi * b_hi into
// d1 (restarted when `fresh1`).  (dx = %9, d1 = %10, freshx = %11, fresh1 = %12)
__device__ __forceinline__ uint32_t mma_block_1xlo_test(uint32_t dx, uint32_t d1, uint32_t ahi,
                                                        uint64_t bhi, uint64_t blo, uint32_t idesc,
                                                        uint32_t freshx, uint32_t fresh1,
                                                        uint32_t lead, uint64_t *tbar,
                                                        uint32_t tpar) {
    uint32_t ok;
    asm volatile(OOP_MMA_PROLOGUE
                 "setp.eq.b32 p1, %11, 0;\n\t"
                 "setp.eq.b32 p2, %12, 0;\n\t"
                 OOP_MMA("%9", "a0", "o0", "p1") OOP_MMA("%9", "a1", "o1", "pt")
                 OOP_MMA("%9", "a2", "o2", "pt") OOP_MMA("%9", "a3", "o3", "pt")
                 OOP_MMA("%10", "a0", "h0", "p2")
                 OOP_MMA_TEST
                 OOP_MMA("%10", "a1", "h1", "pt") OOP_MMA("%10", "a2", "h2", "pt")
                 OOP_MMA("%10", "a3", "h3", "pt")
                 OOP_MMA_EPILOGUE
                 : "=r"(ok)
                 : "r"(lead), "r"(smem_u32(tbar)), "r"(tpar), "r"(ahi), "r"(ahi), "l"(bhi),
                   "l"(blo), "r"(idesc), "r"(dx), "r"(d1), "r"(freshx), "r"(fresh1)
                 : "memory");
    return ok;
}
#undef OOP_MMA
#undef OOP_MMA_EPILOGUE
#undef OOP_MMA_TEST
#undef OOP_MMA_PROLOGUE

// Arrive (once) on `bar` when every tcgen05 op this thread issued completes.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from shared to global memory, in this thread's bulk async-group.
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// this thread's bulk copies have read their shared-memory sources
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// this thread's bulk copies are complete
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// shared-memory writes of this thread made visible to the async proxy (bulk copies)
__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread i writes lane (base + i).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// tcgen05.ld fills its destination registers asynchronously; the compiler
// cannot see that, so the load and its wait sit in ONE asm statement and the
// registers are defined only once the data is there.
__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Two 16-column loads, one wait.
__device__ __forceinline__ void tmem_ld16x2_wait(uint32_t ta, uint32_t (&a)[16], uint32_t tb,
                                                 uint32_t (&b)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]),
          "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]),
          "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]),
          "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]),
          "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
        : "r"(ta), "r"(tb)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---- descriptors ------------------------------------------------------------

// Shared-memory matrix descriptor, K-major operand with the 128-byte swizzle:
// rows of 128 bytes (32 tf32 along k), 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
    d |= static_cast<uint64_t>(1) << 16;                  // leading offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride offset: 8 rows x 128 B
    d |= static_cast<uint64_t>(1) << 46;                  // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                  // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::tf32, D f32, A/B tf32, both K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(int m, int n) {
    return (1u << 4)                                   // D format f32
           | (2u << 7)                                 // A format tf32
           | (2u << 10)                                // B format tf32
           | (static_cast<uint32_t>(n >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(m >> 4) << 24);    // M / 16
}

// ---- numerics ---------------------------------------------------------------

// Round an fp32 bit pattern to the nearest TF32 value, ties away from zero:
// add half of the lowest kept bit (bit 13) to the magnitude, clear the 13
// dropped bits.  Exact integer arithmetic on the full-rate ALU.  Only for
// values below (2 - 2^-11) * 2^127 in magnitude (a dequantised q8_0 / q4_0
// element, at most 65504 * 127, always is): above that the carry reaches the
// exponent and the result is +-Inf.
__device__ __forceinline__ uint32_t tf32_round_bits(uint32_t xb) {
    return (xb + 0x1000u) & 0xFFFFE000u;
}

// The same rounding for any finite fp32 value: where rounding to nearest
// would carry into the all-ones exponent (the top 2^-11 of fp32's top
// binade), the result is the largest finite TF32 value of x's sign instead,
// which is x with its 13 low bits cleared.  As unsigned integers, every
// finite value of one sign lies at or below that limit and the carried
// +-Inf pattern lies above it, so one unsigned minimum does it.  A NaN or
// Inf x also comes out finite here; the remainder x - hi is then NaN or Inf,
// so a split of a non-finite value still carries it.
__device__ __forceinline__ uint32_t tf32_round_bits_sat(uint32_t xb) {
    const uint32_t r = (xb + 0x1000u) & 0xFFFFE000u;
    const uint32_t limit = (xb & 0x80000000u) | 0x7F7FE000u;
    return r < limit ? r : limit;
}

// x = hi + lo + r with hi, lo TF32 (low 13 bits zero): hi = x rounded to
// nearest TF32 (saturating, so every finite x gives a finite hi), lo = (x -
// hi) rounded to nearest TF32 (x - hi is exact in f32 and far below the
// top binade), |r| <= 2^-22 |x|.  Never passes through a 16-bit format.
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    hi = tf32_round_bits_sat(__float_as_uint(x));
    const float rest = x - __uint_as_float(hi);
    lo = tf32_round_bits(__float_as_uint(rest));
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the kernel before it on the stream is still
// running; griddep_wait() returns once that kernel has completed and its
// memory is visible.  launch_dependents() lets the next kernel start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Two fp32 lanes in one 64-bit register (sm_100 packed arithmetic).
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Two floats rounded to bfloat16 (nearest even) in one 32-bit register, the
// first in the low half; and back.  bfloat16 keeps fp32's exponent range.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint64_t unpack_bf16x2(uint32_t v) {
    return pack2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

}  // namespace ptx
}  // namespace oop
