// trsm_llnn_strided_batched_host: the strided-batched solve on HOST buffers.
// The batch is cut into chunks that flow through a three-stage pipeline on
// three internal streams -- copy in, solve, copy out -- over a ring of three
// device buffer sets, so the host->device copy of chunk i+1, the solve of
// chunk i and the device->host copy of chunk i-1 run at the same time (both
// copy directions and the SMs).  The internal streams are forked from and
// joined back to the caller's stream with events, so the call keeps the
// library's stream-ordered semantics; each caller stream has its own set of
// internal streams, so calls on different streams overlap.
#include <map>
#include <mutex>
#include <utility>

#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace {

int elem_size(int dtype) {
    switch (dtype) {
        case TRSM_F32: return 4;
        case TRSM_F64: return 8;
        case TRSM_C64: return 8;
        case TRSM_C128: return 16;
        default: return 0;
    }
}

bool alpha_zero(int dtype, const void *alpha) {
    const int parts = (dtype == TRSM_C64 || dtype == TRSM_C128) ? 2 : 1;
    for (int q = 0; q < parts; ++q) {
        const bool z = (dtype == TRSM_F32 || dtype == TRSM_C64) ? static_cast<const float *>(alpha)[q] == 0.f
                                                                 : static_cast<const double *>(alpha)[q] == 0.0;
        if (!z) return false;
    }
    return true;
}

constexpr int64_t kChunks = 8;
constexpr int kRing = 3;  // buffer sets in flight
std::mutex g_mu;
// Internal streams and a ring of device buffer sets, one per (device,
// caller stream), kept for the life of the process: the buffers only grow,
// so steady-state calls allocate nothing.  Work of successive calls on one
// caller stream is ordered by that stream, which makes the reuse safe.
struct Pipe {
    cudaStream_t in = nullptr, solve = nullptr, out = nullptr;
    void *dA[kRing] = {}, *dB[kRing] = {};
    size_t a_cap = 0, b_cap = 0;
    cudaEvent_t freed[kRing] = {};  // buffer set k read back by the out stream
};
std::map<std::pair<int, cudaStream_t>, Pipe *> g_pipes;

int pipe_for(cudaStream_t user, size_t a_bytes, size_t b_bytes, Pipe **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return trsm::cuda_status(e);
    std::lock_guard<std::mutex> lock(g_mu);
    Pipe *&p = g_pipes[{dev, user}];
    if (!p) {
        p = new Pipe;
        cudaStream_t *s[3] = {&p->in, &p->solve, &p->out};
        for (auto *q : s)
            if ((e = cudaStreamCreateWithFlags(q, cudaStreamNonBlocking)) != cudaSuccess) return trsm::cuda_status(e);
        for (auto &ev : p->freed)
            if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) return trsm::cuda_status(e);
    }
    if (a_bytes > p->a_cap || b_bytes > p->b_cap) {
        // growing: the old buffers may still be in use by earlier calls on
        // `user`; cudaFree waits for the device first
        for (int k = 0; k < kRing; ++k) {
            if (p->dA[k]) cudaFree(p->dA[k]);
            if (p->dB[k]) cudaFree(p->dB[k]);
            p->dA[k] = p->dB[k] = nullptr;
        }
        p->a_cap = a_bytes > p->a_cap ? a_bytes : p->a_cap;
        p->b_cap = b_bytes > p->b_cap ? b_bytes : p->b_cap;
        for (int k = 0; k < kRing; ++k) {
            if ((e = cudaMalloc(&p->dA[k], p->a_cap ? p->a_cap : 16)) != cudaSuccess ||
                (e = cudaMalloc(&p->dB[k], p->b_cap)) != cudaSuccess) {
                p->a_cap = p->b_cap = 0;
                return trsm::cuda_status(e);
            }
        }
    }
    *out = p;
    return TRSM_SUCCESS;
}

// `waiter` waits for the work enqueued so far on `from`.
int link(cudaStream_t from, cudaStream_t waiter) {
    cudaEvent_t ev;
    cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(ev, from);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(waiter, ev, 0);
    cudaEventDestroy(ev);  // released once the recorded work completes
    return e == cudaSuccess ? TRSM_SUCCESS : trsm::cuda_status(e);
}

}  // namespace

extern "C" int trsm_llnn_strided_batched_host(trsm_dtype_t dtype, trsm_layout_t layout, int64_t m, int64_t n,
                                              const void *alpha, const void *A, int64_t lda, int64_t strideA,
                                              void *B, int64_t ldb, int64_t strideB, int64_t batch, void *stream) {
    using trsm::cuda_status;
    const int eb = elem_size(dtype);
    if (!eb) return -1;
    if (layout != TRSM_COL_MAJOR && layout != TRSM_ROW_MAJOR) return -2;
    if (m < 0) return -3;
    if (n < 0) return -4;
    if (!alpha) return -5;
    if (lda < (m > 1 ? m : 1)) return -7;
    if (strideA < 0) return -8;
    const int64_t minor = layout == TRSM_COL_MAJOR ? m : n;
    if (ldb < (minor > 1 ? minor : 1)) return -10;
    if (batch < 0) return -12;
    if (batch > 1 && strideB < (layout == TRSM_COL_MAJOR ? ldb * n : ldb * m)) return -11;
    if (m == 0 || n == 0 || batch == 0) return TRSM_SUCCESS;
    const bool zero = alpha_zero(dtype, alpha);
    if (!zero && !A) return -6;
    if (!B) return -9;

    // elements spanned by `cnt` consecutive systems
    const int64_t a_ext = (m - 1) * lda + m;
    const int64_t b_ext = layout == TRSM_COL_MAJOR ? (n - 1) * ldb + m : (m - 1) * ldb + n;
    auto span = [](int64_t cnt, int64_t stride, int64_t ext) { return (cnt - 1) * stride + ext; };
    const int64_t chunks = batch < kChunks ? batch : kChunks;
    const int64_t cb = (batch + chunks - 1) / chunks;
    const bool share_a = strideA == 0 || batch == 1;  // one A for every system
    const size_t a_bytes = (size_t)(share_a ? a_ext : span(cb, strideA, a_ext)) * eb;
    const size_t b_bytes = (size_t)span(cb, strideB, b_ext) * eb;

    cudaStream_t user = static_cast<cudaStream_t>(stream);
    Pipe *pp = nullptr;
    int rc = pipe_for(user, zero ? 0 : a_bytes, b_bytes, &pp);
    if (rc) return rc;
    Pipe &p = *pp;
    const int nbuf = chunks < kRing ? (int)chunks : kRing;
    cudaError_t e = cudaSuccess;
    if (share_a && !zero) e = cudaMemcpyAsync(p.dA[0], A, (size_t)a_ext * eb, cudaMemcpyHostToDevice, user);
    rc = e == cudaSuccess ? TRSM_SUCCESS : cuda_status(e);
    if (!rc) rc = link(user, p.in);
    if (!rc) rc = link(user, p.solve);
    if (!rc) rc = link(user, p.out);
    for (int64_t c = 0; !rc && c * cb < batch; ++c) {
        const int64_t s0 = c * cb, cnt = (batch - s0 < cb) ? batch - s0 : cb;
        const int k = (int)(c % nbuf);
        const char *ha = static_cast<const char *>(A) + (size_t)(s0 * strideA) * eb;
        char *hb = static_cast<char *>(B) + (size_t)(s0 * strideB) * eb;
        const void *da = share_a ? p.dA[0] : p.dA[k];
        const size_t bb = (size_t)span(cnt, strideB, b_ext) * eb;
        // copy in, once the chunk that used buffer set k last has been copied out
        if (c >= nbuf) e = cudaStreamWaitEvent(p.in, p.freed[k], 0);
        if (e == cudaSuccess && !share_a && !zero)
            e = cudaMemcpyAsync(p.dA[k], ha, (size_t)span(cnt, strideA, a_ext) * eb, cudaMemcpyHostToDevice, p.in);
        if (e == cudaSuccess) e = cudaMemcpyAsync(p.dB[k], hb, bb, cudaMemcpyHostToDevice, p.in);
        if (e != cudaSuccess) {
            rc = cuda_status(e);
            break;
        }
        if ((rc = link(p.in, p.solve))) break;
        rc = trsm_llnn_strided_batched(dtype, layout, m, n, alpha, da, lda, share_a ? 0 : strideA, p.dB[k], ldb,
                                       strideB, cnt, p.solve);
        if (rc || (rc = link(p.solve, p.out))) break;
        e = cudaMemcpyAsync(hb, p.dB[k], bb, cudaMemcpyDeviceToHost, p.out);
        if (e == cudaSuccess) e = cudaEventRecord(p.freed[k], p.out);
        if (e != cudaSuccess) rc = cuda_status(e);
    }
    // join (also after a failure)
    const int j0 = link(p.in, user), j1 = link(p.solve, user), j2 = link(p.out, user);
    const int jr = j0 ? j0 : (j1 ? j1 : j2);
    return rc ? rc : jr;
}
