// Library state shared by the device entry points (gemm_relu.cu) and the
// host-buffer entry point (host_entry.cu): per-device state, per-stream
// buffers, and the calls that run one GEMM on device buffers.  Host code
// only; every function that takes the state runs with g_mu held.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "gemm_relu.h"

namespace gr {
namespace rt {

constexpr int kMaxDevices = 64;
constexpr int kMaxDynSmem = 227 * 1024;  // sm_100-family opt-in limit per CTA
constexpr int kMaxHostChunks = 8;        // row blocks of the pipelined host-buffer entry point

struct StreamBuffers {
    void* stream = nullptr;
    float* ws = nullptr;  // stream-K partial tiles
    size_t ws_bytes = 0;
    uint32_t* counters = nullptr;  // split-K arrival counters + ready flags (zero between launches)
    size_t counter_bytes = 0;
    void* packed = nullptr;  // A copied to a 128-byte row pitch (pack_a plans)
    size_t packed_bytes = 0;
    uint32_t* pack_sync = nullptr;  // the two counters of that copy (zero between launches)
    size_t pack_sync_bytes = 0;
    void* hA = nullptr;  // staging for the host-buffer entry point
    void* hB = nullptr;
    void* hC = nullptr;
    size_t hA_bytes = 0, hB_bytes = 0, hC_bytes = 0;
    int32_t* h_err = nullptr;  // pinned copy of the error word (host-buffer entry point)
    // host-buffer entry point, pipelined: copy-in and copy-out streams and
    // the events that chain them to the compute stream (created on first use)
    bool pipe_ready = false;
    cudaStream_t cin = nullptr, cout = nullptr;
    cudaEvent_t ev_start = nullptr, ev_done = nullptr;
    cudaEvent_t ev_a[kMaxHostChunks] = {}, ev_c[kMaxHostChunks] = {};
};

struct DeviceState {
    bool inited = false;
    int status = GEMM_OK;
    int sm_count = 0;
    int max_pairs = 0;  // co-resident CTA pairs of the paired kernel
    int32_t* d_err = nullptr;
    bool attr_set[6] = {false, false, false, false, false, false};  // per kernel mode
    std::vector<StreamBuffers> streams;
};


extern std::mutex g_mu;
extern DeviceState g_dev[kMaxDevices];

// Argument checks of the C ABI (device_ptrs: the 16-byte alignment rule
// applies to A, B and C).
int check_args(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K, bool device_ptrs);
// The calling thread's current device, if the library can use it.
int current_device(int* dev);
// One-time per-device set-up (device check, encoder entry point, error word).
int init_device_locked(int dev);
// The buffers kept for (device, stream), created empty on first use.
StreamBuffers& buffers_for_locked(DeviceState& d, void* stream);
// Grow (never shrink) one device buffer; synchronizes `stream` first.
int grow(void** buf, size_t* have, size_t need, cudaStream_t stream, bool zero);
// Enqueue C = ReLU(A . B) on device buffers (plan, workspace, maps, launch).
int run_device(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int apply_relu, bool b_nk,
               bool bf16, cudaStream_t st, int dev);
// A launch gave up part-way: clear the error word and every counter.
int reset_after_error_locked(DeviceState& d);
// Release the side streams and events of the host-buffer pipeline.
void pipe_release(StreamBuffers& sb);

}  // namespace rt
}  // namespace gr
