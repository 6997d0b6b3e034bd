// strided.cu -- OUT_PROD with src1 given as a strided view, and the MUL_MAT
// backward pair built on it.
//
// Both gradients of a MUL_MAT are out-products ("metal: OUT_PROD multiplies
// in float staging; a training gradient overflowed half", scope paragraph):
// src0's is out_prod(src1, grad) and src1's is out_prod(src0, grad^T).  The
// second reads the gradient transposed.  With src1 passed as a view (byte
// strides per dimension) that transpose is never materialised: the
// tensor-core kernel's split pre-pass reads the view directly (it writes its
// own k-major layout anyway); the CUDA-core kernels get the view gathered
// into the dense layout in the workspace first.
#include <algorithm>

#include "oop_internal.cuh"

namespace oop {
namespace {

constexpr int kGatherTile = 64;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// View -> dense src1 [slice][k][n].  64 k x 64 n per CTA through shared
// memory, read along whichever of n and k is contiguous, written along n.
__global__ void __launch_bounds__(256) bgather_kernel(const float *__restrict__ b,
                                                      float *__restrict__ out, int64_t K,
                                                      int64_t N, int64_t ne12, int64_t s0,
                                                      int64_t s1, int64_t s2, int64_t s3) {
    __shared__ float tile[kGatherTile][kGatherTile + 1];   // [k][n]
    const int64_t slice = blockIdx.z;
    const float *bs = b + (slice % ne12) * s2 + (slice / ne12) * s3;
    const int64_t k0 = static_cast<int64_t>(blockIdx.x) * kGatherTile;
    const int64_t n0 = static_cast<int64_t>(blockIdx.y) * kGatherTile;
    const int tx = threadIdx.x, ty = threadIdx.y;           // 32 x 8
    if (s1 == 1 && s0 != 1) {                               // k contiguous
        for (int i = ty; i < kGatherTile; i += 8) {         // i: n offset
            const int64_t n = n0 + i;
            for (int h = 0; h < 2; ++h) {
                const int64_t k = k0 + tx + 32 * h;
                tile[tx + 32 * h][i] = (n < N && k < K) ? __ldg(bs + n * s0 + k) : 0.f;
            }
        }
    } else {
        for (int i = ty; i < kGatherTile; i += 8) {         // i: k offset
            const int64_t k = k0 + i;
            for (int h = 0; h < 2; ++h) {
                const int64_t n = n0 + tx + 32 * h;
                tile[i][tx + 32 * h] = (n < N && k < K) ? __ldg(bs + n * s0 + k * s1) : 0.f;
            }
        }
    }
    __syncthreads();
    float *os = out + slice * K * N;
    for (int i = ty; i < kGatherTile; i += 8) {
        const int64_t k = k0 + i;
        if (k >= K) break;
        for (int h = 0; h < 2; ++h) {
            const int64_t n = n0 + tx + 32 * h;
            if (n < N) os[k * N + n] = tile[i][tx + 32 * h];
        }
    }
}

size_t gather_bytes(const OutProdShape &s) {
    return align256(4 * static_cast<size_t>(s.N) * static_cast<size_t>(s.K) *
                    static_cast<size_t>(s.ne12 * s.ne13));
}

}  // namespace

size_t strided_gather_bytes(const OutProdShape &s) { return gather_bytes(s); }

cudaError_t launch_b_gather(const float *b, const OutProdShape &s, float *out,
                            cudaStream_t stream) {
    const int64_t slices = s.ne12 * s.ne13;
    const int64_t gk = (s.K + kGatherTile - 1) / kGatherTile;
    const int64_t gn = (s.N + kGatherTile - 1) / kGatherTile;
    if (gk > 0x7fffffffLL || gn > 65535 || slices > 65535) return cudaErrorInvalidConfiguration;
    bgather_kernel<<<dim3(static_cast<unsigned>(gk), static_cast<unsigned>(gn),
                          static_cast<unsigned>(slices)),
                     dim3(32, 8), 0, stream>>>(b, out, s.K, s.N, s.ne12, s.bs[0], s.bs[1],
                                              s.bs[2], s.bs[3]);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) ++g_kernel_launches;
    return e;
}

}  // namespace oop

// ---- the MUL_MAT backward pair ----------------------------------------------

namespace oop {
namespace {

// The two OUT_PROD calls of a MUL_MAT backward.  Forward (ggml, with its
// broadcast): y[r,t,i2,i3] = sum_k W[k,r,i2/dps2,i3/dps3] x[k,t,i2,i3].
//  dx = OUT_PROD(a = W {K, R, ne02, ne03}, b = dy^T {T, R, ne12, ne13} as a
//       view of dy: n = t at stride R, k = r at stride 1), dst {K, T, ...};
//  dW = OUT_PROD(a = x, b = dy) with each broadcast group's dps2*dps3 slices
//       taken as one reduction of T*dps2*dps3 rows, which is a plain reshape
//       when the group's slices are adjacent (dps3 == 1 or ne02 == 1).
struct BackPlan {
    int64_t K, R, T, ne02, ne03, ne12, ne13, group;
    bool dw_adjacent;
    int64_t dx_ne_a[4], dx_ne_b[4], dx_nb_b[4], dx_ne_dst[4];
    int64_t dw_ne_a[4], dw_ne_b[4], dw_ne_dst[4];
};

int plan_back(const int64_t ne_w[4], const int64_t ne_x[4], BackPlan *p) {
    if (!ne_w || !ne_x) return OOP_ERR_NULL;
    for (int i = 0; i < 4; ++i)
        if (ne_w[i] < 0 || ne_x[i] < 0) return OOP_ERR_SHAPE;
    if (ne_x[0] != ne_w[0]) return OOP_ERR_SHAPE;
    if (ne_w[2] < 1 || ne_w[3] < 1) return OOP_ERR_BROADCAST;
    if (ne_x[2] % ne_w[2] != 0 || ne_x[3] % ne_w[3] != 0) return OOP_ERR_BROADCAST;
    *p = BackPlan{};
    p->K = ne_w[0];
    p->R = ne_w[1];
    p->ne02 = ne_w[2];
    p->ne03 = ne_w[3];
    p->T = ne_x[1];
    p->ne12 = ne_x[2];
    p->ne13 = ne_x[3];
    const int64_t dps2 = p->ne12 / p->ne02, dps3 = p->ne13 / p->ne03;
    p->group = dps2 * dps3;
    p->dw_adjacent = dps3 == 1 || p->ne02 == 1;
    const int64_t dx_a[4] = {p->K, p->R, p->ne02, p->ne03};
    const int64_t dx_b[4] = {p->T, p->R, p->ne12, p->ne13};
    const int64_t dx_nb[4] = {4 * p->R, 4, 4 * p->R * p->T, 4 * p->R * p->T * p->ne12};
    const int64_t dx_d[4] = {p->K, p->T, p->ne12, p->ne13};
    const int64_t dw_a[4] = {p->K, p->T * p->group, p->ne02, p->ne03};
    const int64_t dw_b[4] = {p->R, p->T * p->group, p->ne02, p->ne03};
    const int64_t dw_d[4] = {p->K, p->R, p->ne02, p->ne03};
    for (int i = 0; i < 4; ++i) {
        p->dx_ne_a[i] = dx_a[i];
        p->dx_ne_b[i] = dx_b[i];
        p->dx_nb_b[i] = dx_nb[i];
        p->dx_ne_dst[i] = dx_d[i];
        p->dw_ne_a[i] = dw_a[i];
        p->dw_ne_b[i] = dw_b[i];
        p->dw_ne_dst[i] = dw_d[i];
    }
    return OOP_OK;
}

}  // namespace
}  // namespace oop

extern "C" {

size_t oop_mul_mat_back_workspace_size(int w_type, const int64_t ne_w[4], const int64_t ne_x[4]) {
    oop::BackPlan p;
    if (oop::plan_back(ne_w, ne_x, &p) != OOP_OK) return 0;
    const size_t dx = oop_out_prod_strided_workspace_size(w_type, p.dx_ne_a, p.dx_ne_b, p.dx_nb_b);
    if (dx == 0 && oop::out_prod_check_shape(w_type, p.dx_ne_a, p.dx_ne_b) != OOP_OK) return 0;
    const size_t dw = p.dw_adjacent
                          ? oop_out_prod_workspace_size(OOP_TYPE_F32, p.dw_ne_a, p.dw_ne_b)
                          : 0;
    return std::max(dx, dw);
}

int oop_mul_mat_back(const void *W, int w_type, const float *x, const float *dy, float *dW,
                     float *dx, const int64_t ne_w[4], const int64_t ne_x[4], void *workspace,
                     size_t workspace_bytes, void *stream) {
    oop::g_kernel_launches = 0;
    oop::BackPlan p;
    int rc = oop::plan_back(ne_w, ne_x, &p);
    if (rc != OOP_OK) return rc;
    if (dW && !p.dw_adjacent) return OOP_ERR_BROADCAST;
    // every check of both products before anything is enqueued
    if (dx) {
        rc = oop::run_out_prod(W, w_type, dy, p.dx_nb_b, dx, p.dx_ne_a, p.dx_ne_b, p.dx_ne_dst,
                               workspace, workspace_bytes, stream, OOP_PATH_AUTO, true);
        if (rc != OOP_OK) return rc;
    } else if (oop::out_prod_check_shape(w_type, p.dx_ne_a, p.dx_ne_b) != OOP_OK) {
        return oop::out_prod_check_shape(w_type, p.dx_ne_a, p.dx_ne_b);
    }
    if (dW) {
        rc = oop::run_out_prod(x, OOP_TYPE_F32, dy, nullptr, dW, p.dw_ne_a, p.dw_ne_b,
                               p.dw_ne_dst, workspace, workspace_bytes, stream, OOP_PATH_AUTO,
                               true);
        if (rc != OOP_OK) return rc;
    }
    int launches = 0;
    if (dx) {
        rc = oop::run_out_prod(W, w_type, dy, p.dx_nb_b, dx, p.dx_ne_a, p.dx_ne_b, p.dx_ne_dst,
                               workspace, workspace_bytes, stream, OOP_PATH_AUTO);
        if (rc != OOP_OK) return rc;
        launches += oop::g_kernel_launches;
    }
    if (dW) {
        rc = oop::run_out_prod(x, OOP_TYPE_F32, dy, nullptr, dW, p.dw_ne_a, p.dw_ne_b,
                               p.dw_ne_dst, workspace, workspace_bytes, stream, OOP_PATH_AUTO);
        if (rc != OOP_OK) return rc;
        launches += oop::g_kernel_launches;
    }
    oop::g_kernel_launches = launches;
    return OOP_OK;
}

}  // extern "C"
