// dense_simt.cu -- CUDA-core tiled OUT_PROD for any src0 type.
//
// A plain fp32 shared-memory tiled product: 128 (m) x 64 (n) dst tile per CTA,
// k in steps of 16, each thread 8 m x 4 n outputs, fp32 FMA.  Each 16-term
// partial sum is folded into a Kahan pair, so one gradient entry of 1e5
// dominating a long sum does not carry sqrt(K) roundings of its size.
// A quantised or 16-bit src0 is decoded while its tile is staged.  It is kept as a second,
// independent GPU path for cross-checks of the tensor-core kernel and for
// devices paths that the tensor-core kernel rejects; it is not the fast path.
#include "oop_internal.cuh"
#include "quant.cuh"

namespace oop {
namespace {

constexpr int BM = 128, BN = 64, BK = 16, THREADS = 256;

struct SimtArgs {
    const uint8_t *a;
    const float *b;
    float *dst;
    int64_t M, K, N, ne02, ne12, dps2, dps3, a_row_bytes;
};

template <int TYPE>
__device__ __forceinline__ float a_elem(const uint8_t *row, int64_t m) {
    if constexpr (TYPE == OOP_TYPE_F32) return __ldg(reinterpret_cast<const float *>(row) + m);
    else return decode_row<TYPE>(row, m);
}

template <int TYPE>
__global__ void __launch_bounds__(THREADS) simt_kernel(SimtArgs p) {
    __shared__ float As[BK][BM];
    __shared__ float Bs[BK][BN];
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int64_t slice = blockIdx.z;
    const int64_t i2 = slice % p.ne12, i3 = slice / p.ne12;
    const int64_t j2 = i2 / p.dps2, j3 = i3 / p.dps3;
    const uint8_t *a = p.a + (j3 * p.ne02 + j2) * p.K * p.a_row_bytes;
    const float *b = p.b + slice * p.K * p.N;
    float *dst = p.dst + slice * p.N * p.M;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * BM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.y) * BN;

    float acc[8][4], cmp[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = cmp[i][j] = 0.f;

    for (int64_t k0 = 0; k0 < p.K; k0 += BK) {
        // A tile: 16 x 128 elements, 8 per thread
#pragma unroll
        for (int e = 0; e < (BK * BM) / THREADS; ++e) {
            const int idx = tid + e * THREADS;
            const int kk = idx / BM, mm = idx % BM;
            const int64_t k = k0 + kk, m = m0 + mm;
            As[kk][mm] = (k < p.K && m < p.M) ? a_elem<TYPE>(a + k * p.a_row_bytes, m) : 0.f;
        }
#pragma unroll
        for (int e = 0; e < (BK * BN) / THREADS; ++e) {
            const int idx = tid + e * THREADS;
            const int kk = idx / BN, nn = idx % BN;
            const int64_t k = k0 + kk, n = n0 + nn;
            Bs[kk][nn] = (k < p.K && n < p.N) ? __ldg(b + k * p.N + n) : 0.f;
        }
        __syncthreads();
        float part[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) part[i][j] = 0.f;
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float av[8], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                av[i] = As[kk][tx * 4 + i];
                av[4 + i] = As[kk][64 + tx * 4 + i];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][ty * 4 + j];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) part[i][j] = fmaf(av[i], bv[j], part[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float y = part[i][j] - cmp[i][j];
                const float t = acc[i][j] + y;
                cmp[i][j] = (t - acc[i][j]) - y;
                acc[i][j] = t;
            }
        __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t n = n0 + ty * 4 + j;
        if (n >= p.N) continue;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t m = m0 + (i < 4 ? tx * 4 + i : 64 + tx * 4 + (i - 4));
            if (m < p.M) dst[n * p.M + m] = acc[i][j] - cmp[i][j];
        }
    }
}

}  // namespace

cudaError_t launch_dense_simt(const void *a, const float *b, float *dst, const OutProdShape &s,
                              cudaStream_t stream) {
    SimtArgs p = {};
    p.a = static_cast<const uint8_t *>(a);
    p.b = b;
    p.dst = dst;
    p.M = s.M;
    p.K = s.K;
    p.N = s.N;
    p.ne02 = s.ne02;
    p.ne12 = s.ne12;
    p.dps2 = s.dps2;
    p.dps3 = s.dps3;
    p.a_row_bytes = s.a_row_bytes;
    const int64_t slices = s.ne12 * s.ne13;
    const int64_t gx = (s.M + BM - 1) / BM, gy = (s.N + BN - 1) / BN;
    if (gy > 65535 || slices > 65535 || gx > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy), static_cast<unsigned>(slices));
    switch (s.a_type) {
#define OOP_SIMT_CASE(T) \
    case T: simt_kernel<T><<<grid, THREADS, 0, stream>>>(p); break;
    OOP_SIMT_CASE(OOP_TYPE_F32)
    OOP_SIMT_CASE(OOP_TYPE_F16)
    OOP_SIMT_CASE(OOP_TYPE_BF16)
    OOP_SIMT_CASE(OOP_TYPE_Q4_0)
    OOP_SIMT_CASE(OOP_TYPE_Q4_1)
    OOP_SIMT_CASE(OOP_TYPE_Q5_0)
    OOP_SIMT_CASE(OOP_TYPE_Q5_1)
    OOP_SIMT_CASE(OOP_TYPE_Q8_0)
    OOP_SIMT_CASE(OOP_TYPE_Q2_K)
    OOP_SIMT_CASE(OOP_TYPE_Q3_K)
    OOP_SIMT_CASE(OOP_TYPE_Q4_K)
    OOP_SIMT_CASE(OOP_TYPE_Q5_K)
    OOP_SIMT_CASE(OOP_TYPE_Q6_K)
#undef OOP_SIMT_CASE
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace oop
