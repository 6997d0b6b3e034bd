// host.cu -- OUT_PROD from host buffers: the copies in, the product, the copy
// of dst out, enqueued as one call.
//
// For a single slice long enough in k (tensor-core shapes), the work is
// pipelined over up to four chunks of k: chunk c's src0 rows and src1 rows --
// contiguous host memory, so every copy runs at full speed -- go in while
// chunk c-1's product runs; chunk 0's product writes dst, the others a
// dst-sized partial each; then dst = the chunk results summed in k order with
// a Kahan compensation, in four pieces, each copied out while the next is
// summed.  The copies run on a library-owned copy stream (one per device,
// created on first use) ordered against the caller's stream by events;
// everything is enqueued before the call returns and the caller's stream is
// made to wait for the last copy, so synchronising that stream is enough.
// Otherwise the copies and the product run in order on the caller's stream.
#include <algorithm>
#include <mutex>

#include "oop_internal.cuh"

namespace oop {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 4;                 // chunks of k
constexpr int kPieces = 4;                    // pieces of dst summed and copied out
constexpr int64_t kMinChunkK = 256;           // k rows per chunk, at least
constexpr int kEvents = kMaxChunks + kPieces + 2;

struct HostPipe {
    cudaStream_t copy = nullptr;
    cudaEvent_t ev[kEvents] = {};
};

std::mutex g_host_mu;
HostPipe g_pipe[kMaxDevices];

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct HostLayout {
    size_t a_bytes, b_bytes, dst_bytes;
    size_t off_a, off_b, off_dst, off_ws, ws_bytes, off_parts, part_bytes, total;
    int chunks;                               // chunks of k (1: no pipelining)
};

int64_t src0_bytes(int a_type, const int64_t ne_a[4]) {
    const int64_t rows = ne_a[1] * ne_a[2] * ne_a[3];
    const int qk = type_block_elems(a_type);
    if (qk < 0) return -1;
    return ne_a[0] / qk * type_block_bytes(a_type) * rows;
}

// Chunks of k for the pipelined form: one slice, a tensor-core shape (the
// skinny-N kernel, f32 with N <= 32, is one memory-bound pass), at least
// kMinChunkK rows a chunk.
int host_k_chunks(int a_type, const int64_t ne_a[4], const int64_t ne_b[4]) {
    const bool single = ne_b[2] * ne_b[3] == 1 && ne_a[2] * ne_a[3] == 1;
    if (!single || (a_type == OOP_TYPE_F32 && ne_b[0] <= 32)) return 1;
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(kMaxChunks, ne_a[1] / kMinChunkK)));
}

bool plan_host(int a_type, const int64_t ne_a[4], const int64_t ne_b[4], HostLayout *L) {
    const size_t ws = oop_out_prod_workspace_size(a_type, ne_a, ne_b);
    const int64_t ab = src0_bytes(a_type, ne_a);
    if (ab < 0) return false;
    L->a_bytes = static_cast<size_t>(ab);
    L->b_bytes = 4 * static_cast<size_t>(ne_b[0] * ne_b[1] * ne_b[2] * ne_b[3]);
    L->dst_bytes = 4 * static_cast<size_t>(ne_a[0] * ne_b[0] * ne_b[2] * ne_b[3]);
    size_t o = 0;
    L->off_a = o;
    o += align256(L->a_bytes);
    L->off_b = o;
    o += align256(L->b_bytes);
    L->off_dst = o;
    o += align256(L->dst_bytes);
    L->off_ws = o;
    L->ws_bytes = ws;
    o += align256(ws);
    L->chunks = host_k_chunks(a_type, ne_a, ne_b);
    L->off_parts = o;
    L->part_bytes = align256(L->dst_bytes);
    o += static_cast<size_t>(L->chunks - 1) * L->part_bytes;   // chunks 1.. write partials
    L->total = o;
    return true;
}

// dst[i] = dst[i] + parts[0][i] + ... + parts[nparts-1][i], added in that
// (k) order with a Kahan compensation, for i in [i0, i1).
__global__ void __launch_bounds__(256) chunk_sum_kernel(float *__restrict__ dst,
                                                        const float *__restrict__ parts,
                                                        int64_t part_stride, int nparts,
                                                        int64_t i0, int64_t i1) {
    for (int64_t i = i0 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < i1;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float s = dst[i], c = 0.f;
        for (int q = 0; q < nparts; ++q) {
            const float y = parts[q * part_stride + i] - c;
            const float t = s + y;
            c = (t - s) - y;
            s = t;
        }
        dst[i] = s - c;
    }
}

int pipe_for_device(HostPipe **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return OOP_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return OOP_ERR_DEVICE;
    HostPipe &p = g_pipe[dev];
    if (!p.copy) {
        if (cudaStreamCreateWithFlags(&p.copy, cudaStreamNonBlocking) != cudaSuccess)
            return OOP_ERR_CUDA;
        for (int i = 0; i < kEvents; ++i)
            if (cudaEventCreateWithFlags(&p.ev[i], cudaEventDisableTiming) != cudaSuccess)
                return OOP_ERR_CUDA;
    }
    *out = &p;
    return OOP_OK;
}

int rc_of(cudaError_t e) { return e == cudaSuccess ? OOP_OK : OOP_ERR_CUDA; }

}  // namespace
}  // namespace oop

using namespace oop;

extern "C" {

size_t oop_out_prod_host_buffer_size(int a_type, const int64_t ne_a[4], const int64_t ne_b[4]) {
    if (!ne_a || !ne_b) return 0;
    HostLayout L;
    if (out_prod_check_shape(a_type, ne_a, ne_b) != OOP_OK || !plan_host(a_type, ne_a, ne_b, &L))
        return 0;
    return L.total;
}

int oop_out_prod_host(const void *a_host, int a_type, const float *b_host, float *dst_host,
                      const int64_t ne_a[4], const int64_t ne_b[4], const int64_t ne_dst[4],
                      void *device_buffer, size_t device_bytes, void *stream) {
    if (!ne_a || !ne_b || !ne_dst) return OOP_ERR_NULL;
    // The shape contract exactly as oop_out_prod reports it: called with no
    // buffers it returns a shape error, OOP_OK for an empty dst (nothing to
    // do), and otherwise OOP_ERR_NULL, having enqueued nothing.
    int rc = oop_out_prod(nullptr, a_type, nullptr, nullptr, ne_a, ne_b, ne_dst, nullptr, 0,
                          stream);
    g_kernel_launches = 0;
    if (rc != OOP_ERR_NULL) return rc;
    HostLayout L;
    if (!plan_host(a_type, ne_a, ne_b, &L)) return OOP_ERR_TYPE;
    if (!a_host || !b_host || !dst_host || !device_buffer) return OOP_ERR_NULL;
    if (device_bytes < L.total || reinterpret_cast<uintptr_t>(device_buffer) % 256)
        return OOP_ERR_WORKSPACE;
    uint8_t *dbuf = static_cast<uint8_t *>(device_buffer);
    void *a_dev = dbuf + L.off_a;
    float *b_dev = reinterpret_cast<float *>(dbuf + L.off_b);
    float *dst_dev = reinterpret_cast<float *>(dbuf + L.off_dst);
    void *ws = dbuf + L.off_ws;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    const int64_t M = ne_a[0], K = ne_a[1], N = ne_b[0];
    const int chunks = K > 0 ? L.chunks : 1;
    if (chunks < 2) {
        rc = rc_of(cudaMemcpyAsync(a_dev, a_host, L.a_bytes, cudaMemcpyHostToDevice, st));
        if (rc == OOP_OK)
            rc = rc_of(cudaMemcpyAsync(b_dev, b_host, L.b_bytes, cudaMemcpyHostToDevice, st));
        if (rc == OOP_OK)
            rc = oop_out_prod(a_dev, a_type, b_dev, dst_dev, ne_a, ne_b, ne_dst, ws, L.ws_bytes,
                              stream);
        if (rc == OOP_OK)
            rc = rc_of(cudaMemcpyAsync(dst_host, dst_dev, L.dst_bytes, cudaMemcpyDeviceToHost, st));
        return rc;
    }

    std::lock_guard<std::mutex> lock(g_host_mu);
    HostPipe *pp = nullptr;
    rc = pipe_for_device(&pp);
    if (rc != OOP_OK) return rc;
    cudaStream_t cs = pp->copy;
    cudaEvent_t *ev = pp->ev;
    // chunk c: src0 / src1 rows [kb[c], kb[c+1]), boundaries on 32-row k-blocks;
    // the first chunk's copy is the one nothing overlaps, so it is half the
    // others (the copies then stay ahead of the products: ~200 GB/s of pinned
    // copies bring rows faster than the product consumes them)
    int64_t kb[kMaxChunks + 1];
    kb[0] = 0;
    kb[1] = std::min<int64_t>(K, (K / (2 * chunks - 1) + 31) / 32 * 32);
    const int64_t step = ((K - kb[1] + chunks - 2) / (chunks - 1) + 31) / 32 * 32;
    for (int c = 2; c <= chunks; ++c) kb[c] = std::min<int64_t>(K, kb[1] + (c - 1) * step);
    const size_t a_row = L.a_bytes / static_cast<size_t>(K);          // src0 bytes per k row
    const uint8_t *a_h = static_cast<const uint8_t *>(a_host);
    uint8_t *a_d = static_cast<uint8_t *>(a_dev);
    float *parts = reinterpret_cast<float *>(dbuf + L.off_parts);
    const int64_t part_stride = static_cast<int64_t>(L.part_bytes / 4);
    cudaError_t e = cudaEventRecord(ev[0], st);                // after the caller's prior work
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev[0], 0);
    // copy stream: chunk c's src0 rows and src1 rows in
    for (int c = 0; c < chunks && e == cudaSuccess; ++c) {
        const int64_t k0 = kb[c], kc = kb[c + 1] - kb[c];
        e = cudaMemcpyAsync(a_d + k0 * a_row, a_h + k0 * a_row, static_cast<size_t>(kc) * a_row,
                            cudaMemcpyHostToDevice, cs);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(b_dev + k0 * N, b_host + k0 * N, static_cast<size_t>(kc * N) * 4,
                                cudaMemcpyHostToDevice, cs);
        if (e == cudaSuccess) e = cudaEventRecord(ev[1 + c], cs);
    }
    // compute (caller's) stream: product c once its rows are in; chunk 0 into
    // dst, chunk c > 0 into partial c - 1
    int launches = 0;
    for (int c = 0; c < chunks && e == cudaSuccess && rc == OOP_OK; ++c) {
        e = cudaStreamWaitEvent(st, ev[1 + c], 0);
        if (e != cudaSuccess) break;
        const int64_t k0 = kb[c], kc = kb[c + 1] - kb[c];
        const int64_t ne_ac[4] = {M, kc, 1, 1}, ne_bc[4] = {N, kc, 1, 1};
        float *out = c == 0 ? dst_dev : parts + (c - 1) * part_stride;
        rc = oop_out_prod(a_d + k0 * a_row, a_type, b_dev + k0 * N, out, ne_ac, ne_bc, ne_dst, ws,
                          L.ws_bytes, stream);
        launches += g_kernel_launches;
    }
    // dst = the chunks summed in k order, a piece at a time, each piece copied
    // out (copy stream) while the next one is summed
    const int64_t elems = M * N;
    for (int q = 0; q < kPieces && e == cudaSuccess && rc == OOP_OK; ++q) {
        const int64_t i0 = elems * q / kPieces, i1 = elems * (q + 1) / kPieces;
        if (i1 > i0) {
            const int64_t blocks = std::min<int64_t>(4 * 152, (i1 - i0 + 255) / 256);
            chunk_sum_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
                dst_dev, parts, part_stride, chunks - 1, i0, i1);
            e = cudaGetLastError();
            if (e != cudaSuccess) break;
            ++launches;
        }
        e = cudaEventRecord(ev[1 + kMaxChunks + q], st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev[1 + kMaxChunks + q], 0);
        if (e == cudaSuccess && i1 > i0)
            e = cudaMemcpyAsync(dst_host + i0, dst_dev + i0, static_cast<size_t>(i1 - i0) * 4,
                                cudaMemcpyDeviceToHost, cs);
    }
    // Whatever failed, the caller's stream is made to wait for every copy
    // already enqueued on the copy stream, so that synchronising it still
    // means no copy touches the caller's buffers any more.
    cudaError_t j = cudaEventRecord(ev[kMaxChunks + kPieces + 1], cs);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(st, ev[kMaxChunks + kPieces + 1], 0);
    g_kernel_launches = rc == OOP_OK && e == cudaSuccess ? launches : 0;
    if (rc != OOP_OK) return rc;
    if (e == cudaSuccess) e = j;
    return rc_of(e);
}

}  // extern "C"
