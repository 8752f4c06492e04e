// gemm_relu_host: C = ReLU(A . B) on host buffers -- copies in, GEMM on
// the device, copies out -- with large problems pipelined in row blocks
// over side streams so that the host-link copies and the GEMMs overlap.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include <mutex>

#include "gemm_relu.h"
#include "runtime.h"

namespace gr {
namespace rt {

// Streams and events of the pipelined host-buffer entry point.
int pipe_setup_locked(StreamBuffers& sb) {
    if (sb.pipe_ready) return GEMM_OK;
    bool ok = cudaStreamCreateWithFlags(&sb.cin, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&sb.cout, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&sb.ev_start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&sb.ev_done, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < kMaxHostChunks; ++i)
        ok = cudaEventCreateWithFlags(&sb.ev_a[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&sb.ev_c[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    sb.pipe_ready = true;
    return GEMM_OK;
}

void pipe_release(StreamBuffers& sb) {
    if (!sb.pipe_ready) return;
    cudaStreamDestroy(sb.cin);
    cudaStreamDestroy(sb.cout);
    cudaEventDestroy(sb.ev_start);
    cudaEventDestroy(sb.ev_done);
    for (int i = 0; i < kMaxHostChunks; ++i) {
        cudaEventDestroy(sb.ev_a[i]);
        cudaEventDestroy(sb.ev_c[i]);
    }
    sb.pipe_ready = false;
}

// Row blocks for the host-buffer entry point: with at least 16 MiB of A, B
// and C together, up to kMaxHostChunks blocks of a multiple of 256 rows (at
// least 512), so that the copy of block i + 1 in, the GEMM of block i and
// the copy of block i - 1 out overlap; else one block.
int64_t host_chunk_rows(int64_t M, int64_t N, int64_t K) {
    // tuning override: GEMM_RELU_HOST_BLOCK_ROWS=r (0: one block)
    const char* force = getenv("GEMM_RELU_HOST_BLOCK_ROWS");
    if (force && *force) {
        const long r = strtol(force, nullptr, 10);
        if (r <= 0 || K == 0 || r >= M) return M;
        // at most kMaxHostChunks blocks
        const int64_t least = (M + kMaxHostChunks - 1) / kMaxHostChunks;
        return (int64_t)r < least ? least : (int64_t)r;
    }
    const double bytes = 2.0 * ((double)M * K + (double)K * N + (double)M * N);
    if (K == 0 || bytes < 16.0 * 1024 * 1024 || M < 1024) return M;
    int64_t rows = (M + kMaxHostChunks - 1) / kMaxHostChunks;
    rows = (rows + 255) / 256 * 256;
    if (rows < 512) rows = 512;
    return rows >= M ? M : rows;
}

}  // namespace rt
}  // namespace gr

using namespace gr::rt;

extern "C" int gemm_relu_host(const void* A_host, const void* B_host, void* C_host, int64_t M,
                              int64_t N, int64_t K, int apply_relu, void* stream) {
    int rc = check_args(A_host, B_host, C_host, M, N, K, false);
    if (rc != GEMM_OK) return rc;
    if (M == 0 || N == 0) return GEMM_OK;
    int dev;
    if ((rc = current_device(&dev)) != GEMM_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int32_t* h_err = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if ((rc = init_device_locked(dev)) != GEMM_OK) return rc;
        DeviceState& d = g_dev[dev];
        StreamBuffers& sb = buffers_for_locked(d, stream);
        const size_t a_bytes = (size_t)M * K * 2, b_bytes = (size_t)K * N * 2, c_bytes = (size_t)M * N * 2;
        if ((rc = grow(&sb.hA, &sb.hA_bytes, a_bytes > 16 ? a_bytes : 16, st, false)) != GEMM_OK) return rc;
        if ((rc = grow(&sb.hB, &sb.hB_bytes, b_bytes > 16 ? b_bytes : 16, st, false)) != GEMM_OK) return rc;
        if ((rc = grow(&sb.hC, &sb.hC_bytes, c_bytes, st, false)) != GEMM_OK) return rc;
        if (!sb.h_err && cudaHostAlloc(&sb.h_err, sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess) {
            cudaGetLastError();
            sb.h_err = nullptr;
            return GEMM_ERR_OUT_OF_MEMORY;
        }
        const int64_t rows = host_chunk_rows(M, N, K);
        if (rows >= M) {
            // one block: copies in, GEMM, copies out, all on `stream`
            if (a_bytes && cudaMemcpyAsync(sb.hA, A_host, a_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
                rc = GEMM_ERR_CUDA;
            if (rc == GEMM_OK && b_bytes &&
                cudaMemcpyAsync(sb.hB, B_host, b_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
                rc = GEMM_ERR_CUDA;
            if (rc == GEMM_OK) rc = run_device(sb.hA, sb.hB, sb.hC, M, N, K, apply_relu, false, false, st, dev);
            if (rc == GEMM_OK &&
                cudaMemcpyAsync(C_host, sb.hC, c_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
                rc = GEMM_ERR_CUDA;
            // the error word comes back in the same stream, so one
            // synchronize covers the copies, the kernel and the check
            if (rc == GEMM_OK &&
                cudaMemcpyAsync(sb.h_err, d.d_err, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
                rc = GEMM_ERR_CUDA;
        } else {
            // Row blocks, pipelined over three streams: B and the blocks of
            // A go in on `cin`, block i's GEMM runs on `stream` once its rows
            // are in, and its C rows go out on `cout` once it is done; the
            // copy in of block i + 1, the GEMM of block i and the copy out of
            // block i - 1 overlap (the host link carries both directions at
            // once).  Everything starts after the work already queued on
            // `stream`, and `stream` waits for the last copy out.
            if ((rc = pipe_setup_locked(sb)) != GEMM_OK) return rc;
            const int nblk = (int)((M + rows - 1) / rows);
            const char* ah = static_cast<const char*>(A_host);
            char* ch = static_cast<char*>(C_host);
            char* ad = static_cast<char*>(sb.hA);
            char* cd = static_cast<char*>(sb.hC);
            bool ok = cudaEventRecord(sb.ev_start, st) == cudaSuccess &&
                      cudaStreamWaitEvent(sb.cin, sb.ev_start, 0) == cudaSuccess &&
                      cudaStreamWaitEvent(sb.cout, sb.ev_start, 0) == cudaSuccess &&
                      cudaMemcpyAsync(sb.hB, B_host, b_bytes, cudaMemcpyHostToDevice, sb.cin) == cudaSuccess;
            for (int i = 0; ok && i < nblk; ++i) {
                const int64_t r0 = (int64_t)i * rows, m = (M - r0) < rows ? (M - r0) : rows;
                ok = cudaMemcpyAsync(ad + r0 * K * 2, ah + r0 * K * 2, (size_t)m * K * 2, cudaMemcpyHostToDevice,
                                     sb.cin) == cudaSuccess &&
                     cudaEventRecord(sb.ev_a[i], sb.cin) == cudaSuccess;
            }
            for (int i = 0; ok && i < nblk && rc == GEMM_OK; ++i) {
                const int64_t r0 = (int64_t)i * rows, m = (M - r0) < rows ? (M - r0) : rows;
                ok = cudaStreamWaitEvent(st, sb.ev_a[i], 0) == cudaSuccess;
                if (ok) rc = run_device(ad + r0 * K * 2, sb.hB, cd + r0 * N * 2, m, N, K, apply_relu, false, false, st, dev);
                ok = ok && rc == GEMM_OK && cudaEventRecord(sb.ev_c[i], st) == cudaSuccess &&
                     cudaStreamWaitEvent(sb.cout, sb.ev_c[i], 0) == cudaSuccess &&
                     cudaMemcpyAsync(ch + r0 * N * 2, cd + r0 * N * 2, (size_t)m * N * 2, cudaMemcpyDeviceToHost,
                                     sb.cout) == cudaSuccess;
            }
            // (cout has waited for every GEMM: the error word is final)
            ok = ok && rc == GEMM_OK &&
                 cudaMemcpyAsync(sb.h_err, d.d_err, sizeof(int32_t), cudaMemcpyDeviceToHost, sb.cout) == cudaSuccess &&
                 cudaEventRecord(sb.ev_done, sb.cout) == cudaSuccess &&
                 cudaStreamWaitEvent(st, sb.ev_done, 0) == cudaSuccess;
            if (!ok && rc == GEMM_OK) rc = GEMM_ERR_CUDA;
            if (rc != GEMM_OK) {
                // leave nothing of this call running on the side streams
                cudaStreamSynchronize(sb.cin);
                cudaStreamSynchronize(sb.cout);
            }
        }
        if (rc != GEMM_OK) {
            cudaGetLastError();
            return rc;
        }
        h_err = sb.h_err;
    }
    if (cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (*(volatile int32_t*)h_err == 0) return GEMM_OK;
    std::lock_guard<std::mutex> lock(g_mu);
    return reset_after_error_locked(g_dev[dev]);
}


