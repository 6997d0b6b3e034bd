// batch.cu -- a list of narrow OUT_PRODs in one launch, and the two LoRA
// adapter gradients of a projection built on it.
//
// The rank-r gradients of LoRA fine-tuning ("metal: OUT_PROD runs batched,
// broadcast and narrow shapes on the GPU", opening list item 2) are many small
// OUT_PRODs: each reads a few MB of src0, less than the product of HBM
// bandwidth and latency, so one launch each is bound by launch and memory
// latency.  Streamed together by one persistent kernel (skinny_tma.cu's batch
// form) they keep HBM busy.
#include <algorithm>
#include <vector>

#include "oop_internal.cuh"

namespace oop {
namespace {

bool aligned(const void *p, uintptr_t n) { return reinterpret_cast<uintptr_t>(p) % n == 0; }

}  // namespace
}  // namespace oop

extern "C" {

int oop_out_prod_batch_max(void) { return oop::skinny_batch_max(); }

int oop_out_prod_batch(const oop_out_prod_problem *problems, int count, int64_t N, void *stream) {
    oop::g_kernel_launches = 0;
    if (count < 0) return OOP_ERR_SHAPE;
    if (count == 0) return OOP_OK;
    if (!problems) return OOP_ERR_NULL;
    if (N < 1 || N > 32) return OOP_ERR_SHAPE;
    // every check before anything is enqueued
    for (int i = 0; i < count; ++i) {
        const oop_out_prod_problem &q = problems[i];
        if (q.M < 0 || q.K < 0) return OOP_ERR_SHAPE;
        const double big = 9.0e18;
        if (static_cast<double>(q.M) * q.K * 4.0 > big ||
            static_cast<double>(q.M) * N * 4.0 > big || static_cast<double>(N) * q.K * 4.0 > big)
            return OOP_ERR_SHAPE;
        if (q.M == 0) continue;
        if (!q.dst) return OOP_ERR_NULL;
        if (!oop::aligned(q.dst, 4)) return OOP_ERR_ALIGN;
        if (q.K == 0) continue;
        if (!q.a || !q.b) return OOP_ERR_NULL;
        if (!oop::aligned(q.a, 4) || !oop::aligned(q.b, 4)) return OOP_ERR_ALIGN;
        // a transposed dst is written by the batched form only
        if (q.dst_transposed && !oop::skinny_batch_ok(q, N))
            return N % 4 != 0 ? OOP_ERR_SHAPE : OOP_ERR_ALIGN;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::vector<oop_out_prod_problem> fused;
    int launches = 0;
    for (int i = 0; i < count; ++i) {
        const oop_out_prod_problem &q = problems[i];
        if (q.M == 0) continue;
        if (q.K == 0) {   // an empty sum
            const int rc = oop::cuda_status(
                cudaMemsetAsync(q.dst, 0, static_cast<size_t>(q.M * N) * 4, st));
            if (rc != OOP_OK) return rc;
            continue;
        }
        if (oop::skinny_batch_ok(q, N)) {
            fused.push_back(q);
            continue;
        }
        const int64_t ne_a[4] = {q.M, q.K, 1, 1}, ne_b[4] = {N, q.K, 1, 1};
        const int64_t ne_d[4] = {q.M, N, 1, 1};
        const int rc = oop::run_out_prod(q.a, OOP_TYPE_F32, q.b, nullptr, q.dst, ne_a, ne_b, ne_d,
                                         nullptr, 0, stream, OOP_PATH_SKINNY);
        if (rc != OOP_OK) return rc;
        launches += oop::g_kernel_launches;
    }
    if (!fused.empty()) {
        int *status = nullptr;
        const int rc = oop::device_status_word(&status);
        if (rc != OOP_OK) return rc;
        const int per = oop::skinny_batch_max();
        for (size_t i = 0; i < fused.size(); i += per) {
            const int n = static_cast<int>(std::min<size_t>(per, fused.size() - i));
            const cudaError_t e = oop::launch_skinny_batch(fused.data() + i, n, N, status, st);
            if (e != cudaSuccess) {
                oop::g_kernel_launches = launches;
                return oop::cuda_status(e);
            }
            ++launches;
        }
    }
    oop::g_kernel_launches = launches;
    return OOP_OK;
}

int oop_lora_backward(const float *x, const float *h, const float *dz, const float *dh, float *dA,
                      float *dB, int64_t K_in, int64_t N_out, int64_t T, int64_t r,
                      void *stream) {
    oop_out_prod_problem p[2] = {};
    p[0].a = x;                 // dA {K_in, r} = OUT_PROD(x, dh)
    p[0].b = dh;
    p[0].dst = dA;
    p[0].M = K_in;
    p[0].K = T;
    p[1].a = dz;                // dB {r, N_out} = OUT_PROD(dz, h), written transposed
    p[1].b = h;
    p[1].dst = dB;
    p[1].M = N_out;
    p[1].K = T;
    p[1].dst_transposed = 1;
    return oop_out_prod_batch(p, 2, r, stream);
}

}  // extern "C"
