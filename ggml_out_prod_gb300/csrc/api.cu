// api.cu -- the C ABI: argument checks, kernel choice, device status word.
//
// Every check runs on the host before anything is enqueued, so a rejected
// call leaves the stream untouched.  The shape contract is ggml's OUT_PROD
// contract ("metal: OUT_PROD runs batched, broadcast and narrow shapes on the
// GPU", review comment, first bullet): dst = {a.ne0, b.ne0, b.ne2, b.ne3},
// b.ne2 % a.ne2 == 0 and b.ne3 % a.ne3 == 0.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "oop_internal.cuh"

namespace oop {

thread_local int g_kernel_launches = 0;

namespace {
constexpr int kSmCacheDevices = 64;
std::atomic<int> g_sm_count[kSmCacheDevices];   // 0 = not yet queried
}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= kSmCacheDevices) {
        int v = 0;
        return cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess ? v : 0;
    }
    int v = g_sm_count[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        return 0;
    g_sm_count[dev].store(v, std::memory_order_relaxed);   // every thread stores the same value
    return v;
}

namespace {

// One status word per device, written by kernels through a pointer.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_status_ptr[kMaxDevices];
int g_device_ok[kMaxDevices];      // 0 unknown, 1 sm_103, -1 other

int current_device(int *dev) {
    if (cudaGetDevice(dev) != cudaSuccess) return OOP_ERR_CUDA;
    if (*dev < 0 || *dev >= kMaxDevices) return OOP_ERR_DEVICE;
    return OOP_OK;
}

// Checks the device is sm_103 and returns its status-word address.
int device_setup(int **status) {
    int dev = 0;
    int rc = current_device(&dev);
    if (rc != OOP_OK) return rc;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_device_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return OOP_ERR_CUDA;
        g_device_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        if (g_device_ok[dev] == 1) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
                g_device_ok[dev] = 0;
                return OOP_ERR_CUDA;
            }
            g_status_ptr[dev] = static_cast<int *>(p);
        }
    }
    if (g_device_ok[dev] != 1) return OOP_ERR_DEVICE;
    *status = g_status_ptr[dev];
    return OOP_OK;
}

bool aligned(const void *p, uintptr_t n) { return reinterpret_cast<uintptr_t>(p) % n == 0; }

int64_t row_bytes(int type, int64_t n) {
    const int qk = type_block_elems(type);
    if (qk < 0) return -1;
    return n / qk * type_block_bytes(type);
}

// Shape checks shared by the size query and the call.
int check_out_prod_shape(int a_type, const int64_t ne_a[4], const int64_t ne_b[4],
                         OutProdShape *s) {
    if (!ne_a || !ne_b) return OOP_ERR_NULL;
    for (int i = 0; i < 4; ++i)
        if (ne_a[i] < 0 || ne_b[i] < 0) return OOP_ERR_SHAPE;
    if (type_block_elems(a_type) < 0) return OOP_ERR_TYPE;
    if (ne_a[1] != ne_b[1]) return OOP_ERR_SHAPE;
    if (ne_a[2] < 1 || ne_a[3] < 1) return OOP_ERR_BROADCAST;
    if (ne_b[2] % ne_a[2] != 0 || ne_b[3] % ne_a[3] != 0) return OOP_ERR_BROADCAST;
    if (ne_a[0] % type_block_elems(a_type) != 0) return OOP_ERR_SHAPE;
    // element counts must fit comfortably in int64 arithmetic
    const double big = 9.0e18;
    if (static_cast<double>(ne_a[0]) * ne_a[1] * ne_a[2] * ne_a[3] * 4.0 > big ||
        static_cast<double>(ne_b[0]) * ne_b[1] * ne_b[2] * ne_b[3] * 4.0 > big ||
        static_cast<double>(ne_a[0]) * ne_b[0] * ne_b[2] * ne_b[3] * 4.0 > big)
        return OOP_ERR_SHAPE;
    if (ne_b[2] * ne_b[3] > 65535) return OOP_ERR_SHAPE;   // slices ride grid.z
    s->M = ne_a[0];
    s->K = ne_a[1];
    s->N = ne_b[0];
    s->ne02 = ne_a[2];
    s->ne03 = ne_a[3];
    s->ne12 = ne_b[2];
    s->ne13 = ne_b[3];
    s->dps2 = s->ne12 / s->ne02;
    s->dps3 = s->ne13 / s->ne03;
    s->a_type = a_type;
    s->a_row_bytes = row_bytes(a_type, s->M);
    return OOP_OK;
}

bool skinny_ok(const OutProdShape &s) { return s.a_type == OOP_TYPE_F32 && s.N >= 1 && s.N <= 32; }

int choose_path(const OutProdShape &s, int path) {
    if (path == OOP_PATH_AUTO) return skinny_ok(s) ? OOP_PATH_SKINNY : OOP_PATH_TCGEN05;
    return path;
}

// The least workspace a path runs with (the tensor-core path runs its
// data-parallel schedule on this much; stream-K needs tc_workspace_bytes).
size_t workspace_min(const OutProdShape &s, int path) {
    if (path == OOP_PATH_TCGEN05) return tc_workspace_min_bytes(s);
    return 0;
}

thread_local cudaError_t g_last_cuda = cudaSuccess;

}  // namespace

int device_status_word(int **status) { return device_setup(status); }

int out_prod_check_shape(int a_type, const int64_t ne_a[4], const int64_t ne_b[4]) {
    OutProdShape s = {};
    return check_out_prod_shape(a_type, ne_a, ne_b, &s);
}

int out_prod_auto_workspace(int a_type, const int64_t ne_a[4], const int64_t ne_b[4],
                            size_t *min_bytes, size_t *full_bytes) {
    *min_bytes = *full_bytes = 0;
    OutProdShape s = {};
    const int rc = check_out_prod_shape(a_type, ne_a, ne_b, &s);
    if (rc != OOP_OK) return rc;
    if (choose_path(s, OOP_PATH_AUTO) == OOP_PATH_TCGEN05) {
        *min_bytes = tc_workspace_min_bytes(s);
        *full_bytes = tc_workspace_bytes(s);
    }
    return OOP_OK;
}

namespace {

int cuda_rc(cudaError_t e) {
    if (e == cudaSuccess) return OOP_OK;
    g_last_cuda = e;
    return OOP_ERR_CUDA;
}

// Byte strides of a src1 view: non-negative multiples of 4 (strides of size-1
// dimensions are ignored).  Sets s->b_strided unless the view is the dense
// layout, and s->bs to element strides.
int check_b_strides(const int64_t nb_b[4], OutProdShape *s) {
    s->b_strided = false;
    if (!nb_b) return OOP_OK;
    for (int i = 0; i < 4; ++i)
        if (nb_b[i] < 0 || nb_b[i] % 4 != 0) return OOP_ERR_SHAPE;
    const int64_t ne[4] = {s->N, s->K, s->ne12, s->ne13};
    const int64_t dense[4] = {1, s->N, s->N * s->K, s->N * s->K * s->ne12};
    for (int i = 0; i < 4; ++i) {
        s->bs[i] = ne[i] > 1 ? nb_b[i] / 4 : 0;
        if (ne[i] > 1 && s->bs[i] != dense[i]) s->b_strided = true;
    }
    return OOP_OK;
}

// The least workspace of a path; a strided src1 adds its gather into the
// dense layout for the CUDA-core kernels (the tensor-core split reads views).
size_t workspace_need(const OutProdShape &s, int path) {
    if (s.b_strided && path != OOP_PATH_TCGEN05) return strided_gather_bytes(s);
    return workspace_min(s, path);
}

}  // namespace

int cuda_status(cudaError_t e) { return cuda_rc(e); }

int run_out_prod(const void *a, int a_type, const float *b, const int64_t nb_b[4], float *dst,
                 const int64_t ne_a[4], const int64_t ne_b[4], const int64_t ne_dst[4],
                 void *workspace, size_t workspace_bytes, void *stream, int path,
                 bool check_only) {
    g_kernel_launches = 0;
    OutProdShape s = {};
    int rc = check_out_prod_shape(a_type, ne_a, ne_b, &s);
    if (rc != OOP_OK) return rc;
    rc = check_b_strides(nb_b, &s);
    if (rc != OOP_OK) return rc;
    if (!ne_dst) return OOP_ERR_NULL;
    if (ne_dst[0] != s.M || ne_dst[1] != s.N || ne_dst[2] != s.ne12 || ne_dst[3] != s.ne13)
        return OOP_ERR_SHAPE;
    if (path < OOP_PATH_AUTO || path > OOP_PATH_SIMT) return OOP_ERR_PATH;

    const int64_t n_dst = s.M * s.N * s.ne12 * s.ne13;
    if (n_dst == 0) return OOP_OK;
    if (!dst) return OOP_ERR_NULL;
    if (!aligned(dst, 4)) return OOP_ERR_ALIGN;
    if (s.K > 0) {
        if (!a || !b) return OOP_ERR_NULL;
        if (!aligned(b, 4)) return OOP_ERR_ALIGN;
        if (!aligned(a, a_type == OOP_TYPE_F32 ? 4 : 2)) return OOP_ERR_ALIGN;
    }
    int *status = nullptr;
    rc = device_setup(&status);
    if (rc != OOP_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    const int chosen = choose_path(s, path);
    if (chosen == OOP_PATH_SKINNY && !skinny_ok(s)) return OOP_ERR_PATH;
    const size_t need = workspace_need(s, chosen);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
        return OOP_ERR_WORKSPACE;
    if (check_only) return OOP_OK;

    if (s.K == 0)   // an empty sum
        return cuda_rc(cudaMemsetAsync(dst, 0, static_cast<size_t>(n_dst) * sizeof(float), st));

    cudaError_t e = cudaSuccess;
    if (s.b_strided && chosen != OOP_PATH_TCGEN05) {
        // the CUDA-core kernels read the dense layout: gather the view first
        float *dense = static_cast<float *>(workspace);
        e = launch_b_gather(b, s, dense, st);
        if (e != cudaSuccess) return cuda_rc(e);
        b = dense;
        s.b_strided = false;
    }
    const int gathered = g_kernel_launches;
    s.a_vec16 = aligned(a, 16) && (s.a_row_bytes % 16 == 0);
    s.b_vec16 = !s.b_strided && aligned(b, 16) && (s.N % 4 == 0);
    s.dst_vec16 = aligned(dst, 16) && (s.M % 4 == 0);

    switch (chosen) {
    case OOP_PATH_SKINNY:
        if (skinny_tma_ok(static_cast<const float *>(a), b, s))
            e = launch_skinny_tma(static_cast<const float *>(a), b, dst, s, status, st);
        else
            e = launch_skinny(static_cast<const float *>(a), b, dst, s, st);
        if (e == cudaSuccess) g_kernel_launches = gathered + 1;
        break;
    case OOP_PATH_TCGEN05:
        e = launch_dense_tc(a, b, dst, s, workspace, workspace_bytes, status, st);
        if (e == cudaErrorNotSupported) return OOP_ERR_PATH;
        break;
    case OOP_PATH_SIMT:
        e = launch_dense_simt(a, b, dst, s, st);
        if (e == cudaSuccess) g_kernel_launches = gathered + 1;
        break;
    default:
        return OOP_ERR_PATH;
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    return cuda_rc(e);
}

}  // namespace oop

using namespace oop;

extern "C" {

size_t oop_out_prod_workspace_size(int a_type, const int64_t ne_a[4], const int64_t ne_b[4]) {
    OutProdShape s = {};
    if (check_out_prod_shape(a_type, ne_a, ne_b, &s) != OOP_OK) return 0;
    // cover every path a caller may pick with oop_out_prod_ex
    return tc_workspace_bytes(s);
}

size_t oop_out_prod_workspace_min_size(int a_type, const int64_t ne_a[4], const int64_t ne_b[4]) {
    OutProdShape s = {};
    if (check_out_prod_shape(a_type, ne_a, ne_b, &s) != OOP_OK) return 0;
    return workspace_min(s, OOP_PATH_TCGEN05);
}

int oop_out_prod_ex(const void *a, int a_type, const float *b, float *dst, const int64_t ne_a[4],
                    const int64_t ne_b[4], const int64_t ne_dst[4], void *workspace,
                    size_t workspace_bytes, void *stream, int path) {
    return oop::run_out_prod(a, a_type, b, nullptr, dst, ne_a, ne_b, ne_dst, workspace,
                             workspace_bytes, stream, path);
}

size_t oop_out_prod_strided_workspace_size(int a_type, const int64_t ne_a[4],
                                           const int64_t ne_b[4], const int64_t nb_b[4]) {
    OutProdShape s = {};
    if (check_out_prod_shape(a_type, ne_a, ne_b, &s) != OOP_OK) return 0;
    if (check_b_strides(nb_b, &s) != OOP_OK) return 0;
    if (!s.b_strided) return tc_workspace_bytes(s);
    return std::max(tc_workspace_bytes(s), strided_gather_bytes(s));
}

int oop_out_prod_strided(const void *a, int a_type, const float *b, const int64_t nb_b[4],
                         float *dst, const int64_t ne_a[4], const int64_t ne_b[4],
                         const int64_t ne_dst[4], void *workspace, size_t workspace_bytes,
                         void *stream, int path) {
    if (!nb_b) {
        g_kernel_launches = 0;
        return OOP_ERR_NULL;
    }
    return oop::run_out_prod(a, a_type, b, nb_b, dst, ne_a, ne_b, ne_dst, workspace,
                             workspace_bytes, stream, path);
}

int oop_out_prod(const void *a, int a_type, const float *b, float *dst, const int64_t ne_a[4],
                 const int64_t ne_b[4], const int64_t ne_dst[4], void *workspace,
                 size_t workspace_bytes, void *stream) {
    return oop_out_prod_ex(a, a_type, b, dst, ne_a, ne_b, ne_dst, workspace, workspace_bytes,
                           stream, OOP_PATH_AUTO);
}

int oop_out_prod_plan(int a_type, const int64_t ne_a[4], const int64_t ne_b[4], int path, int sms,
                      size_t workspace_bytes, oop_plan *plan) {
    if (!plan) return OOP_ERR_NULL;
    *plan = oop_plan{};
    OutProdShape s = {};
    int rc = check_out_prod_shape(a_type, ne_a, ne_b, &s);
    if (rc != OOP_OK) return rc;
    if (path < OOP_PATH_AUTO || path > OOP_PATH_SIMT) return OOP_ERR_PATH;
    if (sms < 1) return OOP_ERR_DEVICE;
    if (s.M * s.N * s.ne12 * s.ne13 == 0) return OOP_OK;          // nothing to do
    const int chosen = choose_path(s, path);
    if (chosen == OOP_PATH_SKINNY && !skinny_ok(s)) return OOP_ERR_PATH;
    const size_t need = workspace_min(s, chosen);
    if (need > 0 && workspace_bytes < need) return OOP_ERR_WORKSPACE;
    plan->path = chosen;
    if (s.K == 0) return OOP_OK;                                   // one memset
    switch (chosen) {
    case OOP_PATH_SKINNY:
        if (skinny_tma_shape_ok(s, sms)) {
            plan->kernel = OOP_KERNEL_SKINNY_TMA;
            plan->item_m = static_cast<int>(skinny_tma_tile_m(s, sms));
        } else {
            plan->kernel = OOP_KERNEL_SKINNY;
        }
        plan->launches = 1;
        break;
    case OOP_PATH_TCGEN05:
        plan->ctas = tc_plan_ctas(s, sms, workspace_bytes);
        plan->kernel = plan->ctas > 0 ? OOP_KERNEL_TC_STREAM_K : OOP_KERNEL_TC_DATA_PARALLEL;
        plan->launches = plan->ctas > 0 ? 3 : 2;
        break;
    default:
        plan->kernel = OOP_KERNEL_SIMT;
        plan->launches = 1;
        break;
    }
    return OOP_OK;
}

}  // extern "C"

namespace oop {
namespace {

int check_mmid_shape(int w_type, const int64_t ne_w[3], const int64_t ne_ids[2], MmidShape *s) {
    if (!ne_w || !ne_ids) return OOP_ERR_NULL;
    if (type_block_elems(w_type) < 0) return OOP_ERR_TYPE;
    for (int i = 0; i < 3; ++i)
        if (ne_w[i] < 0) return OOP_ERR_SHAPE;
    if (ne_w[0] % type_block_elems(w_type) != 0) return OOP_ERR_SHAPE;   // blocks run along k
    if (ne_ids[0] < 0 || ne_ids[1] < 0) return OOP_ERR_SHAPE;
    *s = MmidShape{ne_w[0], ne_w[1], ne_w[2], ne_ids[0], ne_ids[1], w_type};
    const double big = 9.0e18;
    if (static_cast<double>(s->K) * s->N * s->E * 4.0 > big ||
        static_cast<double>(s->K) * s->n_used * s->n_tok * 4.0 > big ||
        static_cast<double>(s->N) * s->n_used * s->n_tok * 4.0 > big)
        return OOP_ERR_SHAPE;
    if (s->E > 6144) return OOP_ERR_SHAPE;        // routing keeps per-expert counts on chip
    if (s->n_used * s->n_tok > 0x7fffffffLL) return OOP_ERR_SHAPE;
    return OOP_OK;
}

}  // namespace
}  // namespace oop

extern "C" {

size_t oop_mul_mat_id_back_workspace_size(int w_type, const int64_t ne_w[3],
                                          const int64_t ne_ids[2]) {
    oop::MmidShape s = {};
    if (oop::check_mmid_shape(w_type, ne_w, ne_ids, &s) != OOP_OK) return 0;
    if (s.n_used * s.n_tok == 0 || s.K == 0 || s.E == 0) return 0;
    return oop::tc_mmid_workspace_bytes(s);
}

int oop_mul_mat_id_back_ex(const void *W, int w_type, const int32_t *ids, const float *g,
                           float *dx, const int64_t ne_w[3], const int64_t ne_ids[2],
                           void *workspace, size_t workspace_bytes, void *stream, int path) {
    oop::g_kernel_launches = 0;
    oop::MmidShape s = {};
    int rc = oop::check_mmid_shape(w_type, ne_w, ne_ids, &s);
    if (rc != OOP_OK) return rc;
    if (path != OOP_PATH_AUTO && path != OOP_PATH_TCGEN05 && path != OOP_PATH_SIMT)
        return OOP_ERR_PATH;
    const int64_t slots = s.n_used * s.n_tok;
    if (slots == 0 || s.K == 0) return OOP_OK;
    if (!dx || !ids) return OOP_ERR_NULL;
    if (!aligned(dx, 4) || !aligned(ids, 4)) return OOP_ERR_ALIGN;
    if (s.N > 0) {
        if (!W || !g) return OOP_ERR_NULL;
        if (!aligned(g, 4) || !aligned(W, w_type == OOP_TYPE_F32 ? 4 : 2)) return OOP_ERR_ALIGN;
    }
    // (W's rows are then 2-byte aligned too: every block size is even)
    int *status = nullptr;
    rc = device_setup(&status);
    if (rc != OOP_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool per_slot = path == OOP_PATH_SIMT || s.N == 0 || s.E == 0;
    if (!per_slot) {
        const size_t need = oop::tc_mmid_workspace_bytes(s);
        if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
            return OOP_ERR_WORKSPACE;
        cudaError_t e = oop::launch_mmid_tc(W, ids, g, dx, s, workspace, status, st);
        if (e == cudaSuccess) e = cudaGetLastError();
        return cuda_rc(e);
    }
    if (s.N > 48 * 1024) return OOP_ERR_SHAPE;   // g's slot column is staged on chip
    cudaError_t e = oop::launch_mmid_per_slot(W, ids, g, dx, s, status, st);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) oop::g_kernel_launches = 1;
    return cuda_rc(e);
}

int oop_mul_mat_id_back(const void *W, int w_type, const int32_t *ids, const float *g, float *dx,
                        const int64_t ne_w[3], const int64_t ne_ids[2], void *workspace,
                        size_t workspace_bytes, void *stream) {
    return oop_mul_mat_id_back_ex(W, w_type, ids, g, dx, ne_w, ne_ids, workspace,
                                  workspace_bytes, stream, OOP_PATH_AUTO);
}

size_t oop_mul_mat_id_weight_grad_workspace_size(const int64_t ne_x[3], const int64_t ne_dy[3],
                                                  int64_t n_expert) {
    if (!ne_x || !ne_dy) return 0;
    const oop::WgradShape s = {ne_x[0], ne_x[1], ne_dy[0], ne_dy[1], ne_x[2], n_expert};
    if (s.K < 0 || s.n_x < 1 || s.N < 0 || s.n_used < 0 || s.n_tok < 0 || ne_dy[2] != s.n_tok ||
        s.n_used % s.n_x != 0 || s.E < 1 || s.E > 6144)
        return 0;
    if (s.K == 0 || s.N == 0 || s.n_used * s.n_tok == 0) return 0;
    return oop::tc_wgrad_workspace_bytes(s);
}

int oop_mul_mat_id_weight_grad(const float *x, const int32_t *ids, const float *dy, float *dW,
                               const int64_t ne_x[3], const int64_t ne_dy[3], int64_t n_expert,
                               void *workspace, size_t workspace_bytes, void *stream) {
    oop::g_kernel_launches = 0;
    if (!ne_x || !ne_dy) return OOP_ERR_NULL;
    const oop::WgradShape s = {ne_x[0], ne_x[1], ne_dy[0], ne_dy[1], ne_x[2], n_expert};
    if (s.K < 0 || s.n_x < 1 || s.N < 0 || s.n_used < 0 || s.n_tok < 0) return OOP_ERR_SHAPE;
    if (ne_dy[2] != s.n_tok || s.n_used % s.n_x != 0) return OOP_ERR_SHAPE;
    if (s.E < 1 || s.E > 6144) return OOP_ERR_SHAPE;          // counts are kept on chip
    const double big = 9.0e18;
    if (static_cast<double>(s.K) * s.N * s.E * 4.0 > big ||
        static_cast<double>(s.K) * s.n_x * s.n_tok * 4.0 > big ||
        static_cast<double>(s.N) * s.n_used * s.n_tok * 4.0 > big ||
        s.n_used * s.n_tok > 0x3fffffffLL)
        return OOP_ERR_SHAPE;
    if (s.K == 0 || s.N == 0) return OOP_OK;                  // dW is empty
    if (!dW) return OOP_ERR_NULL;
    if (!aligned(dW, 4)) return OOP_ERR_ALIGN;
    const int64_t slots = s.n_used * s.n_tok;
    if (slots > 0) {
        if (!x || !ids || !dy) return OOP_ERR_NULL;
        if (!aligned(x, 4) || !aligned(ids, 4) || !aligned(dy, 4)) return OOP_ERR_ALIGN;
    }
    int *status = nullptr;
    int rc = device_setup(&status);
    if (rc != OOP_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (slots == 0)   // no slot routed anywhere: every expert's gradient is zero
        return cuda_rc(cudaMemsetAsync(dW, 0, static_cast<size_t>(s.K * s.N * s.E) * 4, st));
    const size_t need = oop::tc_wgrad_workspace_bytes(s);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return OOP_ERR_WORKSPACE;
    cudaError_t e = oop::launch_mmid_wgrad(x, ids, dy, dW, s, workspace, status, st);
    if (e == cudaSuccess) e = cudaGetLastError();
    return cuda_rc(e);
}

int oop_device_status(void *stream, int clear) {
    int *status = nullptr;
    int rc = device_setup(&status);
    if (rc != OOP_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return OOP_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return OOP_ERR_CUDA;
    if (clear && v != 0) {
        if (cudaMemset(status, 0, sizeof(int)) != cudaSuccess) return OOP_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return OOP_ERR_CUDA;
    }
    return v;
}

const char *oop_status_string(int status) {
    switch (status) {
    case OOP_OK: return "ok";
    case OOP_ERR_NULL: return "a required pointer is NULL";
    case OOP_ERR_TYPE: return "unsupported element type";
    case OOP_ERR_SHAPE: return "shape mismatch or unsupported size";
    case OOP_ERR_BROADCAST: return "b.ne2/b.ne3 not divisible by a.ne2/a.ne3";
    case OOP_ERR_ALIGN: return "pointer below its element alignment";
    case OOP_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
    case OOP_ERR_CUDA: return "CUDA runtime error";
    case OOP_ERR_BAD_ID: return "expert id out of range (slot zeroed)";
    case OOP_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out";
    case OOP_ERR_DEVICE: return "current device is not sm_103";
    case OOP_ERR_PATH: return "the requested kernel cannot take this call";
    case OOP_ERR_SCRATCH_LIMIT: return "needs more scratch than the library's fixed device array";
    default: return "unknown status";
    }
}

int oop_version(void) { return (0 << 16) | 1; }

const char *oop_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda); }

int oop_profile_main_kernel(void *before, void *after) {
    tc_set_profile_events(static_cast<cudaEvent_t>(before), static_cast<cudaEvent_t>(after));
    return OOP_OK;
}

int oop_debug_inject_timeout(int enable) {
    tc_set_inject(enable ? 1 : 0);
    return OOP_OK;
}

int oop_debug_set_tc_schedule(int mode) {
    if (mode < 0 || mode > 2) return OOP_ERR_PATH;
    tc_set_schedule(mode);
    return OOP_OK;
}

int oop_last_launch_count(void) { return g_kernel_launches; }

}  // extern "C"
