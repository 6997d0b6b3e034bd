// host.cu -- OUT_PROD from host buffers: the copies in, the product, the copy
// of dst out, enqueued as one call.
//
// For a single slice with N wide enough, the work is pipelined over up to four
// chunks of dst columns n (boundaries on tile edges): src0 and the
// first chunk's src1 columns go in, then each product runs while the next
// chunk's src1 columns are copied in and the previous chunk of dst is copied
// out.  The copies run on a library-owned copy stream (one per
// device, created on first use) ordered against the caller's stream by
// events; everything is enqueued before the call returns and the caller's
// stream is made to wait for the last copy, so synchronising that stream is
// enough.  Otherwise the copies and the product run in order on the caller's
// stream.
#include <algorithm>
#include <mutex>

#include "oop_internal.cuh"

namespace oop {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 4;
constexpr int kEvents = 2 * kMaxChunks + 2;

struct HostPipe {
    cudaStream_t copy = nullptr;
    cudaEvent_t ev[kEvents] = {};
};

std::mutex g_host_mu;
HostPipe g_pipe[kMaxDevices];

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct HostLayout {
    size_t a_bytes, b_bytes, dst_bytes;
    size_t off_a, off_b, off_dst, off_ws, ws_bytes, total;
};

int64_t src0_bytes(int a_type, const int64_t ne_a[4]) {
    const int64_t rows = ne_a[1] * ne_a[2] * ne_a[3];
    const int qk = type_block_elems(a_type);
    if (qk < 0) return -1;
    return ne_a[0] / qk * type_block_bytes(a_type) * rows;
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
    L->total = o;
    return true;
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
    const bool single = ne_b[2] * ne_b[3] == 1 && ne_a[2] * ne_a[3] == 1;
    // chunks of at least two tiles, boundaries on tile edges
    const int64_t tiles_n = (N + oop::kTcTileN - 1) / oop::kTcTileN;
    const int chunks = single && K > 0 ? static_cast<int>(std::min<int64_t>(kMaxChunks, tiles_n / 2)) : 1;
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
    int64_t nb[kMaxChunks + 1];                                // chunk c: columns [nb[c], nb[c+1])
    for (int c = 0; c <= chunks; ++c)
        nb[c] = std::min<int64_t>(N, (tiles_n * c + chunks - 1) / chunks * oop::kTcTileN);
    cudaError_t e = cudaEventRecord(ev[0], st);                // after the caller's prior work
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev[0], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(a_dev, a_host, L.a_bytes, cudaMemcpyHostToDevice, cs);
    // copy stream: src1 chunk c in, then (once product c is done) dst chunk c out
    // compute (caller's) stream: product c once its src1 chunk is in
    int launches = 0;
    for (int c = 0; c < chunks && e == cudaSuccess && rc == OOP_OK; ++c) {
        const int64_t nc = nb[c + 1] - nb[c];
        float *bc = b_dev + K * nb[c];                          // [K][nc] contiguous
        e = cudaMemcpy2DAsync(bc, nc * 4, b_host + nb[c], N * 4, nc * 4, K,
                              cudaMemcpyHostToDevice, cs);
        if (e == cudaSuccess) e = cudaEventRecord(ev[1 + c], cs);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev[1 + c], 0);
        if (e != cudaSuccess) break;
        const int64_t ne_bc[4] = {nc, K, 1, 1};
        const int64_t ne_dc[4] = {M, nc, 1, 1};
        rc = oop_out_prod(a_dev, a_type, bc, dst_dev + nb[c] * M, ne_a, ne_bc, ne_dc, ws,
                          L.ws_bytes, stream);
        if (rc != OOP_OK) break;
        launches += g_kernel_launches;
        e = cudaEventRecord(ev[1 + kMaxChunks + c], st);
    }
    for (int c = 0; c < chunks && e == cudaSuccess && rc == OOP_OK; ++c) {
        e = cudaStreamWaitEvent(cs, ev[1 + kMaxChunks + c], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dst_host + nb[c] * M, dst_dev + nb[c] * M,
                                static_cast<size_t>((nb[c + 1] - nb[c]) * M) * 4,
                                cudaMemcpyDeviceToHost, cs);
    }
    // Whatever failed, the caller's stream is made to wait for every copy
    // already enqueued on the copy stream, so that synchronising it still
    // means no copy touches the caller's buffers any more.
    cudaError_t j = cudaEventRecord(ev[2 * kMaxChunks + 1], cs);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(st, ev[2 * kMaxChunks + 1], 0);
    g_kernel_launches = rc == OOP_OK && e == cudaSuccess ? launches : 0;
    if (rc != OOP_OK) return rc;
    if (e == cudaSuccess) e = j;
    return rc_of(e);
}

}  // extern "C"
