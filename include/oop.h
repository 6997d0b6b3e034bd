/*
 * oop.h -- GB300 (sm_103a) OUT_PROD and MUL_MAT_ID_BACK, C ABI.
 *
 * OUT_PROD is the operation that carries the whole matmul backward in ggml
 * training: both gradients of a MUL_MAT are out-products ("metal: OUT_PROD
 * multiplies in float staging; a training gradient overflowed half", scope
 * paragraph: src0's gradient is out_prod(src1, grad), src1's is
 * out_prod(src0, grad^T)).  MUL_MAT_ID_BACK is the MoE input gradient ("Metal
 * kernel_mul_mat_id_back", first bullet).
 *
 * Layout (ggml's): ne[0] is the fastest dimension; every tensor is dense and
 * contiguous.  M = a.ne0, K = a.ne1 = b.ne1, N = b.ne0.
 *
 * Memory: every pointer passed to a compute entry point is a DEVICE pointer
 * on the current CUDA device, owned by the caller and left owned by the
 * caller.  The library allocates nothing per call and keeps no state except
 * one status word per device (see oop_device_status).
 *
 * Device reset: the library looks up the device addresses of its own device
 * variables (the status word, the scratch of oop_out_prod_noalloc) once per
 * device and keeps them for the life of the process.  A cudaDeviceReset (or
 * anything else that destroys the device's primary context) makes those
 * addresses stale: do not call the library on that device afterwards.
 *
 * Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 * work is enqueued on it in order; no entry point synchronises except
 * oop_device_status.
 *
 * Errors: arguments are checked on the host before anything is enqueued; a
 * failed check returns a negative oop_status and enqueues nothing.  Faults the
 * device detects while running (an expert id out of range, a bounded wait that
 * ran out) are recorded in the device status word and never trap.
 */
#ifndef OOP_H
#define OOP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  The numbers are ggml's public type ids, so a ggml caller
 * passes its own tensor type unchanged; the block layouts are ggml's
 * published formats ("Metal kernel_mul_mat_id_back", first bullet: out_prod
 * is instantiated for all of these).  Blocks run along ne0, so a quantised
 * src0 needs ne0 % 32 == 0 (% 256 for the K-quants).  Little-endian fields;
 * d, m, dmin are binary16. */
typedef enum {
    OOP_TYPE_F32 = 0,
    OOP_TYPE_F16 = 1,
    OOP_TYPE_Q4_0 = 2,  /* 18-byte blocks of 32: d, 16 bytes; byte j holds
                           element j (low nibble) and j+16 (high nibble);
                           value = d * (nibble - 8) */
    OOP_TYPE_Q4_1 = 3,  /* 20-byte blocks of 32: d, m, nibbles as q4_0;
                           value = d * nibble + m */
    OOP_TYPE_Q5_0 = 6,  /* 22-byte blocks of 32: d, a 32-bit word whose bit j is
                           element j's fifth bit, nibbles as q4_0;
                           value = d * (v - 16), v = nibble | fifth << 4 */
    OOP_TYPE_Q5_1 = 7,  /* 24-byte blocks of 32: d, m, fifth bits, nibbles;
                           value = d * v + m */
    OOP_TYPE_Q8_0 = 8,  /* 34-byte blocks of 32: d, 32 int8 q; value = d*q */
    OOP_TYPE_Q2_K = 10, /* 84-byte blocks of 256: 16 bytes of 4-bit scale and
                           offset per 16 elements, 64 bytes of 2-bit codes, d, dmin */
    OOP_TYPE_Q3_K = 11, /* 110-byte blocks of 256: 32 bytes of third bits, 64 bytes
                           of 2-bit codes, 12 bytes of 6-bit scales, d */
    OOP_TYPE_Q4_K = 12, /* 144-byte blocks of 256: d, dmin, 12 bytes of 6-bit scales
                           and offsets per 32 elements, 128 bytes of 4-bit codes;
                           value = d * scale * code - dmin * offset */
    OOP_TYPE_Q5_K = 13, /* 176-byte blocks of 256: as q4_K plus 32 bytes of fifth bits */
    OOP_TYPE_Q6_K = 14, /* 210-byte blocks of 256: 128 bytes of low nibbles, 64 of
                           2-bit high parts, 16 int8 scales per 16 elements, d;
                           value = d * scale * (code - 32) */
    OOP_TYPE_BF16 = 30
} oop_type;

typedef enum {
    OOP_OK = 0,
    OOP_ERR_NULL = -1,           /* a required pointer is NULL */
    OOP_ERR_TYPE = -2,           /* unsupported element type for this operand */
    OOP_ERR_SHAPE = -3,          /* negative size, K mismatch, wrong dst ne, M % 32 */
    OOP_ERR_BROADCAST = -4,      /* b.ne2 % a.ne2 or b.ne3 % a.ne3 non-zero */
    OOP_ERR_ALIGN = -5,          /* a pointer below its element's alignment */
    OOP_ERR_WORKSPACE = -6,      /* workspace NULL or smaller than required */
    OOP_ERR_CUDA = -7,           /* a CUDA runtime call or launch failed */
    OOP_ERR_BAD_ID = -8,         /* device: an expert id outside [0, E) */
    OOP_ERR_DEVICE_TIMEOUT = -9, /* device: a bounded wait ran out */
    OOP_ERR_DEVICE = -10,        /* the current device is not sm_103 */
    OOP_ERR_PATH = -11,          /* oop_out_prod_ex: that kernel cannot take this call */
    OOP_ERR_SCRATCH_LIMIT = -12  /* oop_out_prod_noalloc: the call needs more scratch
                                    than the library's fixed device array holds */
} oop_status;

/* Kernel selection for oop_out_prod_ex. */
typedef enum {
    OOP_PATH_AUTO = 0,    /* what oop_out_prod does */
    OOP_PATH_SKINNY = 1,  /* CUDA-core skinny-N kernel: f32 src0, N <= 32 */
    OOP_PATH_TCGEN05 = 2, /* tensor-core kernel (3xTF32 split), any src0 type */
    OOP_PATH_SIMT = 3     /* CUDA-core tiled kernel, any src0 type (for checks) */
} oop_path;

/*
 * OUT_PROD.  The operation of "metal: OUT_PROD runs batched, broadcast and
 * narrow shapes on the GPU" (review comment, first bullet):
 *
 *   dst[m, n, i2, i3] = sum_k a[m, k, i2/dps2, i3/dps3] * b[n, k, i2, i3]
 *
 *   ne_a   = {M, K, ne02, ne03}   a (src0): any oop_type
 *   ne_b   = {N, K, ne12, ne13}   b (src1): f32
 *   ne_dst = {M, N, ne12, ne13}   dst: f32, OVERWRITTEN (not accumulated)
 *   dps2 = ne12/ne02 and dps3 = ne13/ne03 must divide exactly.
 *
 * Quantised a needs M % 32 == 0 (M % 256 for the K-quants: its blocks run
 * along ne0).  Alignment: f32 pointers 4 bytes, any other a 2 bytes; 16-byte
 * alignment of a and of its rows enables the TMA-fed paths.  The skinny-N
 * kernel takes f32 src0 only; every other type runs on the tensor-core (or
 * CUDA-core) kernel.  K == 0 writes zeros (an empty sum); any other zero size is a no-op.
 * b may hold values far beyond binary16's range: no operand is ever rounded to
 * fp16.  Precision: every finite input gives a finite result within
 * 2e-6 * sum_k |a*b| of the exact sum.
 *
 * workspace: device scratch, 256-byte aligned, of
 * oop_out_prod_workspace_size(...) bytes (NULL allowed when that size is 0).
 * The tensor-core path holds the TF32 split of src1 there and, after it, the
 * k-partials of its stream-K schedule; it runs with as little as
 * oop_out_prod_workspace_min_size(...) bytes, then on its data-parallel
 * schedule only (same results up to rounding order, maybe slower).  Less
 * than the minimum returns OOP_ERR_WORKSPACE.  Its contents on entry do not
 * matter; the call may overwrite all of it.  Two calls in flight at once must
 * not share one workspace.  Both sizes are 0 for an invalid shape.
 */
size_t oop_out_prod_workspace_size(int a_type, const int64_t ne_a[4],
                                   const int64_t ne_b[4]);
size_t oop_out_prod_workspace_min_size(int a_type, const int64_t ne_a[4],
                                       const int64_t ne_b[4]);

int oop_out_prod(const void *a, int a_type, const float *b, float *dst,
                 const int64_t ne_a[4], const int64_t ne_b[4],
                 const int64_t ne_dst[4], void *workspace,
                 size_t workspace_bytes, void *stream);

/* oop_out_prod with the kernel chosen by the caller (oop_path); a path that
 * cannot take the call returns OOP_ERR_PATH.  The workspace rule is the same
 * (oop_out_prod_workspace_size covers every path). */
int oop_out_prod_ex(const void *a, int a_type, const float *b, float *dst,
                    const int64_t ne_a[4], const int64_t ne_b[4],
                    const int64_t ne_dst[4], void *workspace,
                    size_t workspace_bytes, void *stream, int path);

/*
 * OUT_PROD with src1 given as a strided view: element b[n, k, i2, i3] is the
 * f32 at byte offset n*nb_b[0] + k*nb_b[1] + i2*nb_b[2] + i3*nb_b[3] from b.
 * The gradient of a MUL_MAT's src1 is out_prod(src0, grad^T) ("metal:
 * OUT_PROD multiplies in float staging; a training gradient overflowed half",
 * scope paragraph); with nb_b = {4*R, 4, 4*R*T, 4*R*T*ne12} for a grad of
 * {R, T, ne12, ne13}, grad^T is read in place, never materialised.
 *
 * Strides: non-negative multiples of 4 (any order, repeats allowed; a stride
 * of a size-1 dimension is ignored); anything else returns OOP_ERR_SHAPE.
 * The operation, the other arguments, dst, path and errors are those of
 * oop_out_prod_ex.  workspace: oop_out_prod_strided_workspace_size(...)
 * bytes (which covers every path): the tensor-core kernel's split pre-pass
 * reads the view itself; the CUDA-core kernels first gather it into the dense
 * layout in the workspace (4*N*K bytes per slice), so with a strided view
 * they need a workspace too.  A view that is the dense layout is exactly
 * oop_out_prod_ex.
 */
size_t oop_out_prod_strided_workspace_size(int a_type, const int64_t ne_a[4],
                                           const int64_t ne_b[4], const int64_t nb_b[4]);

int oop_out_prod_strided(const void *a, int a_type, const float *b, const int64_t nb_b[4],
                         float *dst, const int64_t ne_a[4], const int64_t ne_b[4],
                         const int64_t ne_dst[4], void *workspace, size_t workspace_bytes,
                         void *stream, int path);

/*
 * Both gradients of a MUL_MAT, in one call ("metal: OUT_PROD multiplies in
 * float staging", scope paragraph: src0's gradient is out_prod(src1, grad),
 * src1's is out_prod(src0, grad^T)).  Forward, with ggml's broadcast:
 *
 *   y[r, t, i2, i3] = sum_k W[k, r, i2/dps2, i3/dps3] * x[k, t, i2, i3]
 *
 *   ne_w = {K, R, ne02, ne03}   W: any oop_type
 *   ne_x = {K, T, ne12, ne13}   x: f32;  dy: f32 {R, T, ne12, ne13}
 *
 *   dx[k, t, i2, i3] = sum_r W[k, r, i2/dps2, i3/dps3] * dy[r, t, i2, i3]
 *                      (OUT_PROD(W, dy^T), dy^T read in place);  dx like x
 *   dW[k, r, j2, j3] = sum of x[k, t, i2, i3] * dy[r, t, i2, i3] over t and
 *                      over the slices (i2, i3) of broadcast group (j2, j3)
 *                      (OUT_PROD(x, dy) with each group's rows as one longer
 *                      reduction);  dW {K, R, ne02, ne03}, f32
 *
 * Either output may be NULL (not computed); both are OVERWRITTEN.  dW needs
 * each group's slices adjacent in memory (dps3 == 1 or ne02 == 1), else
 * OOP_ERR_BROADCAST.  Precision as oop_out_prod.  workspace: at least
 * oop_mul_mat_back_workspace_size(...) bytes, 256-byte aligned; the two
 * products run one after the other on `stream` and share it.  Every check of
 * both products runs before anything is enqueued.
 */
size_t oop_mul_mat_back_workspace_size(int w_type, const int64_t ne_w[4],
                                       const int64_t ne_x[4]);

int oop_mul_mat_back(const void *W, int w_type, const float *x, const float *dy, float *dW,
                     float *dx, const int64_t ne_w[4], const int64_t ne_x[4], void *workspace,
                     size_t workspace_bytes, void *stream);

/*
 * A list of narrow OUT_PRODs in as few launches as possible (no counterpart
 * on the pages' API; the workload is theirs: "metal: OUT_PROD runs batched,
 * broadcast and narrow shapes on the GPU", opening list item 2 -- the rank-r
 * gradients of LoRA fine-tuning).  Each problem is one slice:
 *
 *   dst[m, n] = sum_k a[m, k] * b[n, k]     a {M, K} f32, b {N, K} f32
 *
 * with dst {M, N} f32 OVERWRITTEN, or, with dst_transposed != 0, stored as
 * {N, M} (element (m, n) at m * N + n).  N (1..32) is the
 * same for every problem of the call.  Problems whose a and b are 16-byte
 * aligned with M % 4 == 0, N % 4 == 0 and K > 0 are streamed together by one
 * persistent kernel, up to oop_out_prod_batch_max() per launch (each with its
 * own tensor map); any other problem runs as its own skinny-N launch.  No
 * workspace.  Precision and errors as oop_out_prod; every problem is checked
 * before anything is enqueued.  K == 0 zero-fills that dst.
 */
typedef struct {
    const float *a;       /* {M, K}: device, f32 */
    const float *b;       /* {N, K}: device, f32 */
    float *dst;           /* {M, N}, or {N, M} when dst_transposed: device, f32 */
    int64_t M, K;
    int dst_transposed;
} oop_out_prod_problem;

int oop_out_prod_batch_max(void);

int oop_out_prod_batch(const oop_out_prod_problem *problems, int count, int64_t N, void *stream);

/*
 * Both LoRA adapter gradients of one projection in one launch.  With the
 * adapter y += B (A x) (ggml: A {K_in, r}, B {r, N_out}), the forward's
 * h = A x {r, T} and the backward's dh = B^T dz {r, T} for the output
 * gradient dz {N_out, T} and input x {K_in, T}:
 *
 *   dA = OUT_PROD(x, dh)   {K_in, r}      dA[k, j] = sum_t x[k, t] * dh[j, t]
 *   dB = OUT_PROD(h, dz)   {r, N_out}     dB[j, o] = sum_t h[j, t] * dz[o, t]
 *
 * (dB as the narrow product OUT_PROD(dz, h) written transposed.)  All f32,
 * device pointers, dense; r in 1..32; dA and dB OVERWRITTEN.  Errors and
 * precision as oop_out_prod_batch.
 */
int oop_lora_backward(const float *x, const float *h, const float *dz, const float *dh, float *dA,
                      float *dB, int64_t K_in, int64_t N_out, int64_t T, int64_t r,
                      void *stream);

/*
 * OUT_PROD from HOST buffers (no counterpart on the pages; the benchmark's
 * end-to-end figure goes through it): enqueues on `stream` the copies of a
 * and b into `device_buffer`, the product, and the copy of dst back into
 * dst_host; returns once everything is enqueued.  Synchronise `stream`
 * before reading dst_host.  Pinned (page-locked) host memory makes the copies
 * asynchronous; pageable memory works but blocks the host in the copies.
 *
 * device_buffer: device memory of at least
 * oop_out_prod_host_buffer_size(...) bytes (0 for an invalid shape),
 * 256-byte aligned, holding the device copies of a, b and dst, the
 * workspace and, for the pipelined form, one dst-sized partial per k chunk
 * after the first.  For a single slice with K >= 512 (and not the skinny-N
 * f32 case) the call pipelines up to four chunks of k: a chunk's a and b rows
 * (contiguous host memory) are copied in while the previous chunk's product
 * runs; the chunk results are then summed in k order with a Kahan
 * compensation, in four pieces of dst, each copied out while the next one is
 * summed.  Those copies run on a copy stream the library creates once per
 * device and are ordered against `stream` by events, so the call returns with
 * `stream` waiting for its last copy.  Calls on one device are enqueued one
 * at a time (a library lock).  Errors: as oop_out_prod; OOP_ERR_WORKSPACE for
 * a missing, small or misaligned device_buffer.
 */
size_t oop_out_prod_host_buffer_size(int a_type, const int64_t ne_a[4],
                                     const int64_t ne_b[4]);

int oop_out_prod_host(const void *a_host, int a_type, const float *b_host, float *dst_host,
                      const int64_t ne_a[4], const int64_t ne_b[4],
                      const int64_t ne_dst[4], void *device_buffer,
                      size_t device_bytes, void *stream);

/*
 * OUT_PROD without any device allocation (no counterpart on the pages: the
 * Metal op takes its scratch from the ggml graph).  For callers that cannot
 * allocate device memory or hand the library a scratch buffer -- code inside
 * a framework whose allocator owns all device memory, plug-ins that only get
 * fixed pre-sized tensors, loops where a cudaMalloc would synchronise the
 * device or break a fixed memory budget.
 *
 * Same operation, arguments, errors and precision as oop_out_prod, minus the
 * workspace: the scratch is a 64 MiB device array inside this library
 * (oop_out_prod_noalloc_scratch_bytes()), present on every GPU that loads the
 * library until the process exits.  The scratch a call needs is that of the
 * kernel oop_out_prod picks for it: none for the skinny-N kernel (f32 src0,
 * N <= 32, any K and slice count), otherwise the tensor-core kernel's
 * minimum (oop_out_prod_workspace_min_size).  A call needing more than the
 * array returns OOP_ERR_SCRATCH_LIMIT and enqueues nothing; scratch beyond
 * the minimum only widens the tensor-core kernel's choice of schedule.  The
 * call allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine.
 *
 * The first call on a device that needs scratch looks up that array's
 * device address (once per device, with the device current); make that first
 * call before any stream capture begins.  Every call on a device shares the
 * one array, and each call rewrites all of the scratch it reads, so nothing
 * needs clearing between calls; but two calls that overlap on the GPU (other
 * streams, or another host thread) race on it -- order them on one stream.
 */
size_t oop_out_prod_noalloc_scratch_bytes(void);

int oop_out_prod_noalloc(const void *a, int a_type, const float *b, float *dst,
                         const int64_t ne_a[4], const int64_t ne_b[4],
                         const int64_t ne_dst[4], void *stream);

/*
 * MUL_MAT_ID_BACK, the MoE input gradient ("Metal kernel_mul_mat_id_back",
 * first bullet): for every routed slot (i, t) with expert e = ids[i, t],
 *
 *   dx[k, i, t] = sum_r W[k, r, e] * g[r, i, t]
 *
 *   ne_w   = {K, N, E}             W: any oop_type (out_prod's set), k fastest;
 *                                  rows (e, r) of K elements, quantised blocks
 *                                  along k (K % 32, or % 256 for the K-quants)
 *   ne_ids = {n_used, n_tokens}    ids: int32, slot i fastest
 *   g:  f32 {N, n_used, n_tokens}
 *   dx: f32 {K, n_used, n_tokens}, OVERWRITTEN; one writer per element.
 *
 * The default kernel sorts the slots by expert on the device and runs the
 * tensor-core product per expert (same 3xTF32 scheme and bound as OUT_PROD);
 * it needs oop_mul_mat_id_back_workspace_size(...) bytes of workspace.
 * An id outside [0, E) zeroes that slot's dx and records OOP_ERR_BAD_ID in the
 * device status word.  E <= 6144.
 */
size_t oop_mul_mat_id_back_workspace_size(int w_type, const int64_t ne_w[3],
                                          const int64_t ne_ids[2]);

int oop_mul_mat_id_back(const void *W, int w_type, const int32_t *ids,
                        const float *g, float *dx, const int64_t ne_w[3],
                        const int64_t ne_ids[2], void *workspace,
                        size_t workspace_bytes, void *stream);

/* oop_mul_mat_id_back with the kernel chosen by the caller: OOP_PATH_AUTO or
 * OOP_PATH_TCGEN05 (grouped tensor-core product, needs the workspace) or
 * OOP_PATH_SIMT (one CTA per routed slot, CUDA cores, no workspace). */
int oop_mul_mat_id_back_ex(const void *W, int w_type, const int32_t *ids,
                           const float *g, float *dx, const int64_t ne_w[3],
                           const int64_t ne_ids[2], void *workspace,
                           size_t workspace_bytes, void *stream, int path);

/*
 * The expert-weight gradient of MUL_MAT_ID, the op whose input gradient is
 * MUL_MAT_ID_BACK ("Metal kernel_mul_mat_id_back": its proof is the gradient
 * check of MUL_MAT_ID).  Forward, per routed slot (i, t):
 *
 *   y[r, i, t] = sum_k W[k, r, ids[i, t]] * x[k, i % n_x, t]
 *
 *   ne_x  = {K, n_x, n_tokens}      x: f32; n_x = 1 (one row per token, shared
 *                                   by its slots) or n_used (one per slot),
 *                                   any n_x dividing n_used
 *   ids:  int32 {n_used, n_tokens}  slot i fastest
 *   ne_dy = {N, n_used, n_tokens}   dy: f32, the gradient of y
 *   dW:   f32 {K, N, n_expert}, OVERWRITTEN:
 *
 *   dW[k, r, e] = sum over the slots (i, t) with ids[i, t] == e of
 *                 x[k, i % n_x, t] * dy[r, i, t]      (zero if no slot is routed to e)
 *
 * Per expert an OUT_PROD whose reduction runs over that expert's routed
 * slots, on the tensor cores (same 3xTF32 scheme and bound as oop_out_prod).
 * An id outside [0, n_expert) takes part in no sum and records OOP_ERR_BAD_ID
 * in the device status word.  n_expert <= 6144.  workspace:
 * oop_mul_mat_id_weight_grad_workspace_size(...) bytes, 256-byte aligned (0
 * and NULL allowed for an empty call).
 */
size_t oop_mul_mat_id_weight_grad_workspace_size(const int64_t ne_x[3], const int64_t ne_dy[3],
                                                  int64_t n_expert);

int oop_mul_mat_id_weight_grad(const float *x, const int32_t *ids, const float *dy, float *dW,
                               const int64_t ne_x[3], const int64_t ne_dy[3], int64_t n_expert,
                               void *workspace, size_t workspace_bytes, void *stream);

/* Synchronises `stream`, then returns the current device's status word
 * (OOP_OK, or the first device-side error recorded since it was last
 * cleared); clears it when `clear` is non-zero.  Returns OOP_ERR_CUDA if the
 * synchronisation itself fails. */
int oop_device_status(void *stream, int clear);

/* A static English description of a status code. */
const char *oop_status_string(int status);

/* The CUDA runtime's description of the error behind the calling thread's
 * most recent OOP_ERR_CUDA ("no error" if there was none).  Static string. */
const char *oop_last_cuda_error(void);

/* Library version, (major << 16) | minor. */
int oop_version(void);

/* Measurement hook (no counterpart on the pages): the next tensor-core launch
 * made by the calling thread (OUT_PROD or MUL_MAT_ID_BACK) records the
 * cudaEvent_t `before` on its stream just before its main tile kernel and
 * `after` just after it, so a caller can time that kernel alone, without the
 * src1 split pre-pass.  The events are used once.  Returns OOP_OK. */
int oop_profile_main_kernel(void *before, void *after);

/* Test hook for the device-side failure path (no counterpart on the pages).
 * With enable != 0, the NEXT tensor-core OUT_PROD launch on this process
 * skips one of its TMA copies, so its MMA thread's bounded wait runs out
 * (after about one second); the kernel then records OOP_ERR_DEVICE_TIMEOUT in
 * the device status word, releases its tensor memory and returns without
 * trapping.  dst is left unspecified by that call.  The flag is consumed by
 * that one launch.  Returns OOP_OK. */
int oop_debug_inject_timeout(int enable);

/* The kernels an OUT_PROD call would enqueue, decided by the same host rules
 * as oop_out_prod_ex (no counterpart on the pages; nothing runs and no device
 * is needed): for a GPU with `sms` SMs, `workspace_bytes` of workspace and
 * 16-byte aligned a and b.  The tile schedule follows
 * oop_debug_set_tc_schedule like the calls do. */
typedef enum {
    OOP_KERNEL_NONE = 0,             /* empty dst: nothing; K == 0: one memset of dst */
    OOP_KERNEL_SKINNY = 1,           /* register-pipelined skinny-N kernel */
    OOP_KERNEL_SKINNY_TMA = 2,       /* persistent, TMA-fed skinny-N kernel */
    OOP_KERNEL_TC_DATA_PARALLEL = 3, /* split of src1, then one 128 x 96 dst tile per CTA */
    OOP_KERNEL_TC_STREAM_K = 4,      /* split of src1, stream-K tile kernel, fix-up */
    OOP_KERNEL_SIMT = 5              /* CUDA-core tiled kernel */
} oop_kernel;

typedef struct {
    int path;     /* OOP_PATH_SKINNY / _TCGEN05 / _SIMT; 0 (AUTO) when dst is empty */
    int kernel;   /* an oop_kernel */
    int item_m;   /* OOP_KERNEL_SKINNY_TMA: m columns per work item (128 or 64), else 0 */
    int ctas;     /* OOP_KERNEL_TC_STREAM_K: CTAs sharing the tile x k-block iterations, else 0 */
    int launches; /* kernels the call enqueues (as oop_last_launch_count reports) */
} oop_plan;

/* Fills *plan.  Returns OOP_OK, the argument errors of oop_out_prod_ex (shape,
 * type, broadcast, path, OOP_ERR_WORKSPACE when workspace_bytes is below the
 * chosen path's minimum), OOP_ERR_NULL for a NULL plan, or OOP_ERR_DEVICE
 * when sms < 1. */
int oop_out_prod_plan(int a_type, const int64_t ne_a[4], const int64_t ne_b[4], int path,
                      int sms, size_t workspace_bytes, oop_plan *plan);

/* Test hook (no counterpart on the pages): the schedule of the tensor-core
 * OUT_PROD tile kernel for the calls that follow on this process.  mode 0 =
 * automatic (the default: stream-K when an even share of the tile x k-block
 * iterations per SM, plus the cost of the partials and the fix-up, beats the
 * data-parallel waves by 10%, and the workspace holds the partials), 1 = always
 * data-parallel (one 128 x 96 dst tile per CTA), 2 = always stream-K (one
 * CTA per SM sharing the tile x k-block iterations, then a fix-up kernel),
 * when the workspace allows.  MUL_MAT_ID_BACK's grouped product (its tile
 * count is known on the device only) runs one CTA per SM taking whole tiles
 * round-robin in mode 0, stream-K in mode 2 and data-parallel in mode 1.
 * Results agree to rounding order either way.
 * Returns OOP_OK, or OOP_ERR_PATH for another mode. */
int oop_debug_set_tc_schedule(int mode);

/* How many kernels the last OUT_PROD or MUL_MAT_ID_BACK call made on this
 * host thread enqueued (0 after a rejected call or an empty one; memsets are
 * not kernels).  No counterpart on the pages; for benchmarks that report
 * their launch count. */
int oop_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* OOP_H */
