// mmid.cu -- MUL_MAT_ID_BACK, one CTA per routed slot.
//
// "Metal kernel_mul_mat_id_back", first bullet: one threadgroup per routed
// slot (i, t); each thread owns columns k of that slot's output row and walks
// the rows r of the routed expert, so every dx element has one writer and no
// expert is copied or transposed.  Here a CTA of 256 threads owns one slot;
// thread t accumulates k = t + 256*j (coalesced reads of each expert row r,
// which is contiguous in k), g's slot column is staged in shared memory.
#include "oop_internal.cuh"

namespace oop {
namespace {

constexpr int kThreads = 256;
constexpr int kPer = 8;     // k columns per thread per pass

template <int TYPE>
__device__ __forceinline__ float w_elem(const void *W, int64_t idx) {
    if constexpr (TYPE == OOP_TYPE_F32) {
        return __ldg(static_cast<const float *>(W) + idx);
    } else {
        return bf16_bits_to_float(__ldg(static_cast<const unsigned short *>(W) + idx));
    }
}

template <int TYPE>
__global__ void __launch_bounds__(kThreads) mmid_slot_kernel(const void *W, const int32_t *ids,
                                                              const float *g, float *dx,
                                                              int64_t K, int64_t N, int64_t E,
                                                              int *status) {
    extern __shared__ float gs[];
    const int64_t slot = blockIdx.x;               // t * n_used + i
    const int32_t e = __ldg(ids + slot);
    float *out = dx + slot * K;
    if (e < 0 || e >= E) {
        for (int64_t k = threadIdx.x; k < K; k += kThreads) out[k] = 0.f;
        if (threadIdx.x == 0) record_status(status, OOP_ERR_BAD_ID);
        return;
    }
    for (int64_t r = threadIdx.x; r < N; r += kThreads) gs[r] = __ldg(g + slot * N + r);
    __syncthreads();
    const int64_t wbase = static_cast<int64_t>(e) * N * K;
    for (int64_t kb = 0; kb < K; kb += kThreads * kPer) {
        float acc[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
        for (int64_t r = 0; r < N; ++r) {
            const float gr = gs[r];
            const int64_t rb = wbase + r * K;
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const int64_t k = kb + threadIdx.x + j * kThreads;
                if (k < K) acc[j] = fmaf(w_elem<TYPE>(W, rb + k), gr, acc[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int64_t k = kb + threadIdx.x + j * kThreads;
            if (k < K) out[k] = acc[j];
        }
    }
}

}  // namespace

cudaError_t launch_mmid_per_slot(const void *W, const int32_t *ids, const float *g, float *dx,
                                 const MmidShape &s, int *status, cudaStream_t stream) {
    const int64_t slots = s.n_used * s.n_tok;
    if (slots > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const size_t smem = sizeof(float) * static_cast<size_t>(s.N);
    if (smem > 200 * 1024) return cudaErrorInvalidValue;
    auto k32 = mmid_slot_kernel<OOP_TYPE_F32>;
    auto kbf = mmid_slot_kernel<OOP_TYPE_BF16>;
    auto kern = s.w_type == OOP_TYPE_F32 ? k32 : kbf;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    kern<<<static_cast<unsigned>(slots), kThreads, smem, stream>>>(W, ids, g, dx, s.K, s.N, s.E,
                                                                   status);
    return cudaGetLastError();
}

}  // namespace oop
