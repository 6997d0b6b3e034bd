// noalloc.cu -- OUT_PROD for callers that cannot allocate device memory.
//
// The tensor-core OUT_PROD needs scratch for its TF32 split of src1 (two
// words per element of b).  oop_out_prod takes that scratch from the caller.
// Some callers cannot hand it over: code that runs inside a framework whose
// allocator owns all device memory and offers no way to request a temporary
// buffer, plug-ins called with fixed, pre-sized tensors only, and code paths
// where a cudaMalloc would synchronise the device or fail (real-time loops,
// memory budgets fixed at start-up).  oop_out_prod_noalloc serves them: its
// scratch is a file-scope device array of a fixed size that is part of this
// library's image, so it exists on every GPU that loads the library and
// stays there until the process exits.  Nothing here calls cudaMalloc,
// cudaFree or any allocating routine.
#include <mutex>

#include "oop_internal.cuh"

namespace oop {
namespace {

// 64 MiB: the TF32 split of a gradient of up to 8 Mi elements (for example
// N = 1024, K = 8192, one slice).
constexpr size_t kScratchBytes = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];

// Once per device, with that device current: the device address of the
// array.  (In host code the array's name is only a host-side stand-in.)
int scratch_for_current_device(void **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return OOP_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return OOP_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return OOP_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return OOP_OK;
}

}  // namespace
}  // namespace oop

extern "C" {

size_t oop_out_prod_noalloc_scratch_bytes(void) { return oop::kScratchBytes; }

int oop_out_prod_noalloc(const void *a, int a_type, const float *b, float *dst,
                         const int64_t ne_a[4], const int64_t ne_b[4], const int64_t ne_dst[4],
                         void *stream) {
    // The scratch the kernel oop_out_prod chooses needs: none for the skinny-N
    // kernel (f32 src0, N <= 32), else the tensor-core minimum, with whatever
    // of the array lies beyond it letting that kernel pick its stream-K
    // schedule.  Shape errors are left to oop_out_prod, which reports them
    // exactly as it always does.
    size_t need = 0, full = 0;
    if (oop::out_prod_auto_workspace(a_type, ne_a, ne_b, &need, &full) != OOP_OK)
        return oop_out_prod(a, a_type, b, dst, ne_a, ne_b, ne_dst, nullptr, 0, stream);
    if (need > oop::kScratchBytes) return OOP_ERR_SCRATCH_LIMIT;
    const size_t give = full < oop::kScratchBytes ? full : oop::kScratchBytes;
    void *scratch = nullptr;
    if (give > 0) {
        const int rc = oop::scratch_for_current_device(&scratch);
        if (rc != OOP_OK) return rc;
    }
    return oop_out_prod(a, a_type, b, dst, ne_a, ne_b, ne_dst, scratch, give, stream);
}

}  // extern "C"
