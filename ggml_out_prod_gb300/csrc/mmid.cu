// mmid.cu -- MUL_MAT_ID_BACK, one CTA per routed slot.
//
// "Metal kernel_mul_mat_id_back", first bullet: one threadgroup per routed
// slot (i, t); each thread owns columns k of that slot's output row and walks
// the rows r of the routed expert, so every dx element has one writer and no
// expert is copied or transposed.  Here a CTA of 256 threads owns one slot;
// thread t accumulates k = t + 256*j (coalesced reads of each expert row r,
// which is contiguous in k), g's slot column is staged in shared memory.
#include "oop_internal.cuh"
#include "quant.cuh"

namespace oop {
namespace {

constexpr int kThreads = 256;
constexpr int kPer = 8;     // k columns per thread per pass

// W[k, r, e]: element k of row (e, r), rows of `row_bytes` (any src0 type;
// quantised blocks run along k)
template <int TYPE>
__device__ __forceinline__ float w_elem(const uint8_t *row, int64_t k) {
    if constexpr (TYPE == OOP_TYPE_F32) return __ldg(reinterpret_cast<const float *>(row) + k);
    else return decode_row<TYPE>(row, k);
}

template <int TYPE>
__global__ void __launch_bounds__(kThreads) mmid_slot_kernel(const void *W, const int32_t *ids,
                                                              const float *g, float *dx,
                                                              int64_t K, int64_t N, int64_t E,
                                                              int64_t row_bytes, int *status) {
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
    const uint8_t *wbase = static_cast<const uint8_t *>(W) + static_cast<int64_t>(e) * N * row_bytes;
    for (int64_t kb = 0; kb < K; kb += kThreads * kPer) {
        float acc[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
        for (int64_t r = 0; r < N; ++r) {
            const float gr = gs[r];
            const uint8_t *row = wbase + r * row_bytes;
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const int64_t k = kb + threadIdx.x + j * kThreads;
                if (k < K) acc[j] = fmaf(w_elem<TYPE>(row, k), gr, acc[j]);
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
    decltype(&mmid_slot_kernel<OOP_TYPE_F32>) kern = nullptr;
    switch (s.w_type) {
#define OOP_MMID_CASE(T) \
    case T: kern = mmid_slot_kernel<T>; break;
    OOP_MMID_CASE(OOP_TYPE_F32)
    OOP_MMID_CASE(OOP_TYPE_F16)
    OOP_MMID_CASE(OOP_TYPE_BF16)
    OOP_MMID_CASE(OOP_TYPE_Q4_0)
    OOP_MMID_CASE(OOP_TYPE_Q4_1)
    OOP_MMID_CASE(OOP_TYPE_Q5_0)
    OOP_MMID_CASE(OOP_TYPE_Q5_1)
    OOP_MMID_CASE(OOP_TYPE_Q8_0)
    OOP_MMID_CASE(OOP_TYPE_Q2_K)
    OOP_MMID_CASE(OOP_TYPE_Q3_K)
    OOP_MMID_CASE(OOP_TYPE_Q4_K)
    OOP_MMID_CASE(OOP_TYPE_Q5_K)
    OOP_MMID_CASE(OOP_TYPE_Q6_K)
#undef OOP_MMID_CASE
    default: return cudaErrorInvalidValue;
    }
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    const int64_t row_bytes = s.K / type_block_elems(s.w_type) * type_block_bytes(s.w_type);
    kern<<<static_cast<unsigned>(slots), kThreads, smem, stream>>>(W, ids, g, dx, s.K, s.N, s.E,
                                                                   row_bytes, status);
    return cudaGetLastError();
}

}  // namespace oop
