// oop_internal.cuh -- shared declarations of the CUDA library (not part of
// the public C ABI; the public header is include/oop.h).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "oop.h"

namespace oop {

// dst columns (src1 rows n) per tile of the tensor-core kernel
constexpr int kTcTileN = 128;

// Elements and bytes per block of a src0 type (1 and the element size for the
// plain types), -1 for an unknown type.  Host and device.
__host__ __device__ constexpr int type_block_elems(int type) {
    switch (type) {
    case OOP_TYPE_F32: case OOP_TYPE_F16: case OOP_TYPE_BF16: return 1;
    case OOP_TYPE_Q4_0: case OOP_TYPE_Q4_1: case OOP_TYPE_Q5_0: case OOP_TYPE_Q5_1:
    case OOP_TYPE_Q8_0: return 32;
    case OOP_TYPE_Q2_K: case OOP_TYPE_Q3_K: case OOP_TYPE_Q4_K: case OOP_TYPE_Q5_K:
    case OOP_TYPE_Q6_K: return 256;
    default: return -1;
    }
}
__host__ __device__ constexpr int type_block_bytes(int type) {
    switch (type) {
    case OOP_TYPE_F32: return 4;
    case OOP_TYPE_F16: case OOP_TYPE_BF16: return 2;
    case OOP_TYPE_Q4_0: return 18;
    case OOP_TYPE_Q4_1: return 20;
    case OOP_TYPE_Q5_0: return 22;
    case OOP_TYPE_Q5_1: return 24;
    case OOP_TYPE_Q8_0: return 34;
    case OOP_TYPE_Q2_K: return 84;
    case OOP_TYPE_Q3_K: return 110;
    case OOP_TYPE_Q4_K: return 144;
    case OOP_TYPE_Q5_K: return 176;
    case OOP_TYPE_Q6_K: return 210;
    default: return -1;
    }
}

// One OUT_PROD call after validation.  Slice (i2, i3) of dst reads src0
// slice (i2/dps2, i3/dps3): the CPU backend's broadcast map ("metal: OUT_PROD
// runs batched, broadcast and narrow shapes on the GPU", review comment).
struct OutProdShape {
    int64_t M, K, N;
    int64_t ne02, ne03, ne12, ne13;
    int64_t dps2, dps3;
    int64_t a_row_bytes;          // bytes of one src0 row of M elements
    int a_type;
    bool a_vec16;                 // a base and row stride 16-byte aligned
    bool b_vec16;                 // b base and row stride 16-byte aligned
    bool dst_vec16;               // dst base and row stride 16-byte aligned
    // src1 as a strided view: element (n, k, i2, i3) at
    // n*bs[0] + k*bs[1] + i2*bs[2] + i3*bs[3] floats from b.  Only the
    // tensor-core split reads such a view; b_strided false means the dense
    // layout ((i3*ne12 + i2)*K + k)*N + n.
    bool b_strided;
    int64_t bs[4];
};

struct MmidShape {
    int64_t K, N, E, n_used, n_tok;
    int w_type;
};

// MUL_MAT_ID's expert-weight gradient: x {K, n_x, n_tok}, dy {N, n_used,
// n_tok}, dW {K, N, E}.
struct WgradShape {
    int64_t K, n_x, N, n_used, n_tok, E;
};

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// First error wins; later errors do not overwrite it.
__device__ __forceinline__ void record_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ---- kernels (each .cu file owns its launcher) ----------------------------

// cuTensorMapEncodeTiled through the runtime's driver entry point, looked up
// once (nullptr when the driver does not offer it).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Skinny-N OUT_PROD: f32 src0, N <= 32.
cudaError_t launch_skinny(const float *a, const float *b, float *dst,
                          const OutProdShape &s, cudaStream_t stream);
// Its persistent TMA-fed form for large problems (N % 4 == 0, M % 4 == 0,
// 16-byte aligned a and b, at least two m-tile x slice items per SM).
bool skinny_tma_ok(const float *a, const float *b, const OutProdShape &s);
// The shape part of that rule on a GPU with `sms` SMs (no device calls), and
// the m-width of its items: 128, 64, or 0 when the form does not apply.
bool skinny_tma_shape_ok(const OutProdShape &s, int sms);
int64_t skinny_tma_tile_m(const OutProdShape &s, int sms);
cudaError_t launch_skinny_tma(const float *a, const float *b, float *dst,
                              const OutProdShape &s, int *status, cudaStream_t stream);

// A list of single-slice f32 problems with the same N in one persistent
// launch (at most skinny_batch_max() per launch; each must pass
// skinny_batch_ok).
bool skinny_batch_ok(const oop_out_prod_problem &q, int64_t N);
int skinny_batch_max();
cudaError_t launch_skinny_batch(const oop_out_prod_problem *probs, int count, int64_t N,
                                int *status, cudaStream_t stream);

// CUDA-core tiled OUT_PROD, any src0 type.
cudaError_t launch_dense_simt(const void *a, const float *b, float *dst,
                              const OutProdShape &s, cudaStream_t stream);

// Kernels enqueued by the current API call on this thread (each launcher
// adds its own).
extern thread_local int g_kernel_launches;

// The current device's status-word address, after checking it is sm_103
// (OOP_OK or the status the entry points return).
int device_status_word(int **status);
// OOP_OK for cudaSuccess; otherwise OOP_ERR_CUDA, recording the error for
// oop_last_cuda_error.
int cuda_status(cudaError_t e);

// SM count of the current device, queried once per device (0 on failure).
// Safe to call from several host threads at once.
int device_sm_count();

// The OUT_PROD shape contract as oop_out_prod checks it (OOP_OK or the
// status it would return for these sizes and type).
int out_prod_check_shape(int a_type, const int64_t ne_a[4], const int64_t ne_b[4]);

// The workspace of the kernel oop_out_prod would choose for these sizes: the
// least it runs with and the size that lets it pick its fastest schedule
// (both 0 for the skinny-N kernel, which needs none).  Returns the shape
// check's status.
int out_prod_auto_workspace(int a_type, const int64_t ne_a[4], const int64_t ne_b[4],
                            size_t *min_bytes, size_t *full_bytes);

// Every OUT_PROD entry point ends here: host checks, kernel choice, launch.
// nb_b: byte strides of a src1 view, or NULL for the dense layout.  With
// check_only the call returns after the host checks, having enqueued nothing.
int run_out_prod(const void *a, int a_type, const float *b, const int64_t nb_b[4], float *dst,
                 const int64_t ne_a[4], const int64_t ne_b[4], const int64_t ne_dst[4],
                 void *workspace, size_t workspace_bytes, void *stream, int path,
                 bool check_only = false);

// A strided src1 view gathered into the dense layout [slice][k][n] (for the
// CUDA-core kernels), and the bytes that takes.
size_t strided_gather_bytes(const OutProdShape &s);
cudaError_t launch_b_gather(const float *b, const OutProdShape &s, float *out,
                            cudaStream_t stream);

// Tensor-core OUT_PROD (tcgen05, 3xTF32).  The workspace holds the TF32 split
// of src1 (the minimum) and, after it, the stream-K partial slots; with less
// than tc_workspace_bytes the data-parallel schedule is used.
size_t tc_workspace_bytes(const OutProdShape &s);
size_t tc_workspace_min_bytes(const OutProdShape &s);
void tc_set_inject(int v);   // test hook: the next tensor-core launch drops one TMA stage
void tc_set_schedule(int v); // test hook: 0 automatic, 1 data-parallel, 2 stream-K
void tc_set_profile_events(cudaEvent_t before, cudaEvent_t after);
// The tile kernel's schedule on a GPU with `sms` SMs and this much workspace
// (no device calls): the stream-K CTA count, 0 for data-parallel.
int tc_plan_ctas(const OutProdShape &s, int sms, size_t workspace_bytes);
cudaError_t launch_dense_tc(const void *a, const float *b, float *dst,
                            const OutProdShape &s, void *workspace, size_t workspace_bytes,
                            int *status, cudaStream_t stream);

// MUL_MAT_ID_BACK as a grouped tensor-core product (slots sorted by expert).
size_t tc_mmid_workspace_bytes(const MmidShape &s);
cudaError_t launch_mmid_tc(const void *W, const int32_t *ids, const float *g, float *dx,
                           const MmidShape &s, void *workspace, int *status,
                           cudaStream_t stream);

// MUL_MAT_ID's expert-weight gradient as a segmented tensor-core product.
size_t tc_wgrad_workspace_bytes(const WgradShape &s);
cudaError_t launch_mmid_wgrad(const float *x, const int32_t *ids, const float *dy, float *dW,
                              const WgradShape &s, void *workspace, int *status,
                              cudaStream_t stream);

// MUL_MAT_ID_BACK, one CTA per routed slot.
cudaError_t launch_mmid_per_slot(const void *W, const int32_t *ids,
                                 const float *g, float *dx, const MmidShape &s,
                                 int *status, cudaStream_t stream);

}  // namespace oop
