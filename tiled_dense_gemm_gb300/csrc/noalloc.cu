// gemm_relu_noalloc: the small-M (swapped-operand) kernel with its split-K
// scratch in a fixed, file-scope device array instead of memory the library
// allocates.  Nothing on this path calls cudaMalloc, cudaFree or any other
// allocating routine.
//
// Why it exists: gemm_relu grows its split-K workspace with cudaMalloc the
// first time a shape needs it, and cudaMalloc / cudaFree may synchronize
// the device.  Some callers cannot allow that -- a latency-critical loop
// that must never stall on an allocation, or a process whose device memory
// is entirely pre-reserved by another allocator.  They call this entry
// point instead; it only ever touches the inputs, the output and the fixed
// array below.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "gemm_kernel.cuh"
#include "gemm_relu.h"

namespace gr {
namespace {

// Scratch layout (bytes):
//   [0, 16)                error word of the kernel (int32 at 0)
//   [256, kPartialOffset)  split-K arrival counters (one per split tile),
//                          then max_slots ready flags per split tile
//   [kPartialOffset, end)  fp32 partial tiles
constexpr size_t kScratchBytes = GEMM_RELU_NOALLOC_SCRATCH_BYTES;
constexpr size_t kCounterOffset = 256;
constexpr size_t kPartialOffset = 64 * 1024;
constexpr size_t kMaxCounters = (kPartialOffset - kCounterOffset) / sizeof(uint32_t);

// One copy per device, held for the life of the process.  In host code the
// name is only a handle for cudaGetSymbolAddress: the device address is
// looked up once per device and passed to the kernel as a pointer.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
constexpr int kMaxDynSmem = 227 * 1024;

struct NoAllocState {
    bool inited = false;
    int status = GEMM_OK;
    int sm_count = 0;
    uint8_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_na_mu;
NoAllocState g_na[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_na_encode = nullptr;

// Set-up on the first call for a device (the device is current): checks
// the device, finds the tensor-map encoder, resolves the scratch address
// and raises the kernel's shared-memory limit.  No allocation.
int setup_locked(int dev) {
    NoAllocState& s = g_na[dev];
    if (s.inited) return s.status;
    s.inited = true;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        major != 10 || minor != 3) {
        cudaGetLastError();
        return s.status = GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    if (cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return s.status = GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    if (!g_na_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return s.status = GEMM_ERR_UNSUPPORTED_DEVICE;
        }
        g_na_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return s.status = GEMM_ERR_CUDA;
    }
    s.scratch = static_cast<uint8_t*>(ptr);
    if (cudaFuncSetAttribute(gemm_relu_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxDynSmem) != cudaSuccess) {
        cudaGetLastError();
        return s.status = GEMM_ERR_LAUNCH;
    }
    return s.status = GEMM_OK;
}

int encode(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
           uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_na_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims,
                             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_INVALID_ARG;
}

}  // namespace
}  // namespace gr

using namespace gr;

extern "C" int gemm_relu_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N,
                                 int64_t K, int apply_relu, void* stream) {
    if (M < 0 || N < 0 || K < 0 || M > GEMM_RELU_MAX_DIM || N > GEMM_RELU_MAX_DIM ||
        K > GEMM_RELU_MAX_DIM)
        return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C || !A || !B) return GEMM_ERR_INVALID_ARG;
    if (K % 8 != 0 || N % 8 != 0) return GEMM_ERR_ALIGNMENT;
    if (((((uintptr_t)A) | ((uintptr_t)B) | ((uintptr_t)C)) & 15u) != 0) return GEMM_ERR_ALIGNMENT;
    // this variant covers the small-M kernel only, with K > 0
    if (M > 128 || K == 0) return GEMM_ERR_TOO_LARGE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_na_mu);
    int rc = setup_locked(dev);
    if (rc != GEMM_OK) return rc;
    NoAllocState& s = g_na[dev];

    gemm_relu_plan_t pl;
    rc = plan_problem(M, N, K, s.sm_count, -1, "swap", &pl);  // no clusters: plain launch
    if (rc != GEMM_OK) return rc;
    if (pl.path != 3 || pl.cluster != 1) return GEMM_ERR_TOO_LARGE;
    const size_t partial_bytes = (size_t)pl.workspace_bytes;
    if ((size_t)pl.counter_count * (1 + (size_t)pl.max_slots) > kMaxCounters ||
        partial_bytes > kScratchBytes - kPartialOffset)
        return GEMM_ERR_TOO_LARGE;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // The array keeps whatever the previous call left: the counters must
    // start at zero (partials are written before they are read).  The error
    // word is left as it is, for gemm_relu_noalloc_check_device_error.
    if (cudaMemsetAsync(s.scratch + kCounterOffset, 0, kPartialOffset - kCounterOffset, st) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }

    KParams kp;
    memset(&kp, 0, sizeof(kp));
    kp.plan = pl;
    kp.M = M;
    kp.N = N;
    kp.K = K;
    kp.apply_relu = apply_relu ? 1 : 0;
    kp.C = reinterpret_cast<uint16_t*>(C);
    kp.err = reinterpret_cast<int32_t*>(s.scratch);
    kp.counters = reinterpret_cast<uint32_t*>(s.scratch + kCounterOffset);
    kp.ws = reinterpret_cast<float*>(s.scratch + kPartialOffset);
    kp.timeout_ns = 2000000000ull + 2000ull * (uint64_t)pl.num_kb;
    {
        // the test hook of the bounded waits, as in gemm_relu
        const char* drop = getenv("GEMM_RELU_TEST_DROP_KB");
        if (drop && *drop) {
            const long kb = strtol(drop, nullptr, 10);
            if (kb < 0 || kb >= pl.num_kb) return GEMM_ERR_INVALID_ARG;
            kp.test_drop_kb = (int32_t)kb + 1;
            kp.timeout_ns = kTestTimeoutNs;
        }
    }
    kp.idesc = make_idesc_f16_f32(128u, (uint32_t)pl.mma_n, /*a_mn=*/true, /*b_mn=*/false);

    CUtensorMap ta, tb, tc;
    if ((rc = encode(&ta, A, (uint64_t)K, (uint64_t)M, kBlockK, (uint32_t)pl.tile_m)) != GEMM_OK) return rc;
    if ((rc = encode(&tb, B, (uint64_t)N, (uint64_t)K, 64u, (uint32_t)pl.block_k)) != GEMM_OK) return rc;
    if ((rc = encode(&tc, C, (uint64_t)N, (uint64_t)M, 64, 32)) != GEMM_OK) return rc;  // unused by this kernel

    gemm_relu_kernel<2><<<pl.grid, kThreads, pl.smem_bytes, st>>>(ta, tb, tb, tc, ta, kp);
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
    return GEMM_OK;
}

extern "C" int gemm_relu_noalloc_check_device_error(void* stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_na_mu);
    int rc = setup_locked(dev);
    if (rc != GEMM_OK) return rc;
    NoAllocState& s = g_na[dev];
    int32_t err = 0;
    if (cudaMemcpy(&err, s.scratch, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (err == 0) return GEMM_OK;
    // a launch gave up part-way: clear the word and the counters it may
    // have left set
    if (cudaMemsetAsync(s.scratch, 0, kPartialOffset, st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return GEMM_ERR_TIMEOUT;
}
