// C ABI of the GB300 gemm_relu library: argument checks, per-device state,
// tensor-map encoding, workspace management and kernel launch (the
// host-buffer entry point is in host_entry.cu).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <unordered_map>
#include <vector>

#include "gemm_kernel.cuh"
#include "gemm_relu.h"
#include "runtime.h"

namespace gr {

// C := +0 for K == 0 (the empty sum).
__global__ void zero_fill_kernel(uint4* c, int64_t n16) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride)
        c[i] = make_uint4(0u, 0u, 0u, 0u);
}

namespace rt {

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

struct PlanKey {
    int64_t M, N, K;
    bool operator==(const PlanKey& o) const { return M == o.M && N == o.N && K == o.K; }
};
struct PlanKeyHash {
    size_t operator()(const PlanKey& k) const {
        uint64_t h = (uint64_t)k.M * 0x9E3779B97F4A7C15ull;
        h ^= (uint64_t)k.N + 0x7F4A7C159E3779B9ull + (h << 6) + (h >> 2);
        h ^= (uint64_t)k.K + 0x94D049BB133111EBull + (h << 6) + (h >> 2);
        return (size_t)h;
    }
};

std::unordered_map<PlanKey, gemm_relu_plan_t, PlanKeyHash> g_plans[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int init_device_locked(int dev) {
    DeviceState& d = g_dev[dev];
    if (d.inited) return d.status;
    d.inited = true;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return d.status = GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    if (major != 10 || minor != 3) return d.status = GEMM_ERR_UNSUPPORTED_DEVICE;
    int optin = 0;
    cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (optin < kMaxDynSmem) return d.status = GEMM_ERR_UNSUPPORTED_DEVICE;
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return d.status = GEMM_ERR_UNSUPPORTED_DEVICE;
        }
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    {
        // how many CTA pairs of the paired kernel can be resident at once
        auto fn = gemm_relu_kernel<3>;
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem) ==
            cudaSuccess) {
            d.attr_set[3] = true;
            gemm_relu_plan_t probe;
            plan_problem(4096, 4096, 4096, d.sm_count, 0, "pair", &probe);
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(2 * (d.sm_count / 2), 1, 1);
            cfg.blockDim = dim3(kThreads, 1, 1);
            cfg.dynamicSmemBytes = (size_t)probe.smem_bytes;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) == cudaSuccess && n > 0) d.max_pairs = n;
        }
        cudaGetLastError();
        // no co-resident pairs reported: the paired kernel is not used
        if (d.max_pairs <= 0) d.max_pairs = -1;
    }
    if (cudaMalloc(&d.d_err, 16) != cudaSuccess) {
        cudaGetLastError();
        d.inited = false;
        return GEMM_ERR_OUT_OF_MEMORY;
    }
    if (cudaMemset(d.d_err, 0, 16) != cudaSuccess) {
        cudaGetLastError();
        return d.status = GEMM_ERR_CUDA;
    }
    return d.status = GEMM_OK;
}

int current_device(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    if (*dev < 0 || *dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    return GEMM_OK;
}

StreamBuffers& buffers_for_locked(DeviceState& d, void* stream) {
    for (auto& s : d.streams)
        if (s.stream == stream) return s;
    d.streams.emplace_back();
    d.streams.back().stream = stream;
    return d.streams.back();
}

// Grow (never shrink) one device buffer.  Synchronizes `stream` first so no
// launch still reads the old one.
int grow(void** buf, size_t* have, size_t need, cudaStream_t stream, bool zero) {
    if (*have >= need) return GEMM_OK;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (*buf) cudaFree(*buf);
    *buf = nullptr;
    *have = 0;
    size_t bytes = need + need / 4;  // headroom against repeated small growth
    if (cudaMalloc(buf, bytes) != cudaSuccess) {
        cudaGetLastError();
        *buf = nullptr;
        return GEMM_ERR_OUT_OF_MEMORY;
    }
    if (zero && cudaMemset(*buf, 0, bytes) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    *have = bytes;
    return GEMM_OK;
}

int encode_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer, bool bf16, uint64_t pitch_elems = 0) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {(pitch_elems ? pitch_elems : inner) * 2};  // bytes between rows
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                          const_cast<void*>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_INVALID_ARG;
}

// 3-D view of a row-major matrix whose rows hold `inner` elements (a
// multiple of 64): dimension 0 is 64 elements of a column block, 1 the rows
// (`outer`, `pitch_elems` apart), 2 the inner / 64 column blocks (128 bytes
// apart).  A box of `box_blocks` blocks lands block after block in shared
// memory, each one 128B-swizzled like a 2-D box of the same rows.  The
// column blocks never reach past a row's end, so every element read is
// inside the matrix; rows and blocks beyond it read as zero.
int encode_3d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer,
              uint32_t box_blocks, bool bf16, uint64_t pitch_elems) {
    if (inner % 64 != 0) return GEMM_ERR_INVALID_ARG;
    cuuint64_t dims[3] = {64, outer, inner / 64};
    cuuint64_t strides[2] = {(pitch_elems ? pitch_elems : inner) * 2, 128};
    cuuint32_t box[3] = {64, box_outer, box_blocks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                          const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_INVALID_ARG;
}

template <int kMode>
int launch_mode(DeviceState& d, const gemm_relu_plan_t& pl, const KParams& kp, const CUtensorMap& ta,
                const CUtensorMap& tb, const CUtensorMap& tb2, const CUtensorMap& tc, const CUtensorMap& ta2,
                cudaStream_t st) {
    auto fn = gemm_relu_kernel<kMode>;
    if (!d.attr_set[kMode]) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem) !=
            cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        d.attr_set[kMode] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3((unsigned)(pl.grid * pl.cluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)pl.smem_bytes;
    cfg.stream = st;
    // programmatic dependent launch: this kernel's set-up may overlap the
    // tail of the previous kernel on the stream (the kernel waits for that
    // kernel before touching global memory)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    unsigned n_attr = 1;
    // CTA pairs and cluster split-K: `cluster` CTAs per worker
    const unsigned cdim = (unsigned)pl.cluster;
    if (cdim > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cdim;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n_attr = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    if (cudaLaunchKernelEx(&cfg, fn, ta, tb, tb2, tc, ta2, kp) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
    return GEMM_OK;
}

int check_args(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
               bool device_ptrs) {
    if (M < 0 || N < 0 || K < 0 || M > GEMM_RELU_MAX_DIM || N > GEMM_RELU_MAX_DIM ||
        K > GEMM_RELU_MAX_DIM)
        return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
    if (K % 8 != 0 || N % 8 != 0) return GEMM_ERR_ALIGNMENT;
    if (device_ptrs) {
        if (((uintptr_t)C & 15u) != 0) return GEMM_ERR_ALIGNMENT;
        if (K > 0 && ((((uintptr_t)A) | ((uintptr_t)B)) & 15u) != 0) return GEMM_ERR_ALIGNMENT;
    }
    return GEMM_OK;
}

// The tensor maps of one call: A, B (and B's second, 2-D map), C, and A's
// copy at a 128-byte pitch (pack_a plans; else a copy of A's map).
struct Maps {
    CUtensorMap ta, tb, tb2, tc, ta2;
    int32_t a3d, b3d;
};

int encode_maps(const gemm_relu_plan_t& pl, const void* A, const void* B, void* C, int64_t M, int64_t N,
                int64_t K, bool b_nk, bool bf16, const char* force, const void* A2, uint64_t a2_pitch, Maps* m) {
    // the boxes of one stage's copies (3-D where the shapes allow)
    gemm_relu_boxes_t bx;
    int rc = plan_boxes(pl, M, N, K, b_nk, force, &bx);
    if (rc != GEMM_OK) return rc;
    if (bx.a_3d)
        rc = encode_3d(&m->ta, A, (uint64_t)K, (uint64_t)M, bx.a_box[1], bx.a_box[2], bf16, 0);
    else
        rc = encode_2d(&m->ta, A, (uint64_t)K, (uint64_t)M, bx.a_box[0], bx.a_box[1], bf16);
    if (rc != GEMM_OK) return rc;
    if (A2) {
        // (a pack_a plan has K % 64 != 0, so A's copies are 2-D)
        if (bx.a_3d) return GEMM_ERR_INVALID_ARG;
        rc = encode_2d(&m->ta2, A2, (uint64_t)K, (uint64_t)M, bx.a_box[0], bx.a_box[1], bf16, a2_pitch);
        if (rc != GEMM_OK) return rc;
    } else {
        m->ta2 = m->ta;
    }
    m->a3d = bx.a_3d;
    if (!b_nk) {
        // the second map: 64-column 2-D boxes (the partial chunk a 3-D view
        // of whole chunks leaves out)
        rc = encode_2d(&m->tb2, B, (uint64_t)N, (uint64_t)K, bx.b2_box[0], bx.b2_box[1], bf16);
        if (rc == GEMM_OK) {
            if (bx.b_3d)
                rc = encode_3d(&m->tb, B, (uint64_t)bx.b_view_inner, (uint64_t)K, bx.b_box[1], bx.b_box[2], bf16,
                               (uint64_t)N);
            else
                rc = encode_2d(&m->tb, B, (uint64_t)N, (uint64_t)K, bx.b_box[0], bx.b_box[1], bf16);
        }
    } else {
        rc = encode_2d(&m->tb2, B, (uint64_t)K, (uint64_t)N, bx.b2_box[0], bx.b2_box[1], bf16);
        if (rc == GEMM_OK) {
            if (bx.b_3d)
                rc = encode_3d(&m->tb, B, (uint64_t)K, (uint64_t)N, bx.b_box[1], bx.b_box[2], bf16, 0);
            else
                m->tb = m->tb2;
        }
    }
    if (rc != GEMM_OK) return rc;
    m->b3d = bx.b_3d;
    // C: 64-column x 32-row boxes, one per epilogue warp and chunk
    return encode_2d(&m->tc, C, (uint64_t)N, (uint64_t)M, 64, 32, bf16);
}

// Encoded tensor maps per (pointers, shape, B layout, element type): a map
// holds only an address, sizes, strides and box shapes, so it stays valid
// for any call with the same arguments, whatever the buffers hold.
struct MapKey {
    const void* A;
    const void* B;
    const void* C;
    const void* A2;  // A's copy at a 128-byte pitch, or null
    int64_t M, N, K;
    int32_t flags;
    bool operator==(const MapKey& o) const {
        return A == o.A && B == o.B && C == o.C && A2 == o.A2 && M == o.M && N == o.N && K == o.K &&
               flags == o.flags;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        uint64_t h = (uint64_t)(uintptr_t)k.A * 0x9E3779B97F4A7C15ull;
        h ^= (uint64_t)(uintptr_t)k.B + 0x7F4A7C159E3779B9ull + (h << 6) + (h >> 2);
        h ^= (uint64_t)(uintptr_t)k.C + 0x94D049BB133111EBull + (h << 6) + (h >> 2);
        h ^= (uint64_t)(uintptr_t)k.A2 + 0x2545F4914F6CDD1Dull + (h << 6) + (h >> 2);
        h ^= (uint64_t)k.M + 0xBF58476D1CE4E5B9ull + (h << 6) + (h >> 2);
        h ^= (uint64_t)k.N + 0x94D049BB133111EBull + (h << 6) + (h >> 2);
        h ^= (uint64_t)k.K + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
        h ^= (uint64_t)k.flags + (h << 6) + (h >> 2);
        return (size_t)h;
    }
};
constexpr size_t kMapCacheEntries = 1024;
std::unordered_map<MapKey, Maps, MapKeyHash> g_maps[kMaxDevices];

int run_device(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
               int apply_relu, bool b_nk, bool bf16, cudaStream_t st, int dev) {
    DeviceState& d = g_dev[dev];
    if (M == 0 || N == 0) return GEMM_OK;
    if (K == 0) {
        const int64_t n16 = M * N * 2 / 16;  // N % 8 == 0
        int blocks = (int)((n16 + 255) / 256);
        const int cap = d.sm_count * 8;
        if (blocks > cap) blocks = cap;
        zero_fill_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<uint4*>(C), n16);
        return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
    }
    gemm_relu_plan_t pl;
    const char* force = getenv("GEMM_RELU_FORCE_PATH");
    const bool forced = force && *force;
    if (forced) {
        // tuning / test override: plan every call, bypass the caches
        int rc = plan_problem(M, N, K, d.sm_count, d.max_pairs, force, &pl);
        if (rc != GEMM_OK) return rc;
    } else {
        auto& cache = g_plans[dev];
        PlanKey key{M, N, K};
        auto itp = cache.find(key);
        if (itp != cache.end()) {
            pl = itp->second;
        } else {
            int rc = plan_problem(M, N, K, d.sm_count, d.max_pairs, nullptr, &pl);
            if (rc != GEMM_OK) return rc;
            if (cache.size() > 4096) cache.clear();
            cache.emplace(key, pl);
        }
    }
    // the swapped kernel's exchange buffer holds one peer's partial
    if (pl.path == 3 && cluster_split(pl) && pl.cluster != 2) return GEMM_ERR_INVALID_ARG;
    KParams kp;
    memset(&kp, 0, sizeof(kp));
    kp.plan = pl;
    kp.M = M;
    kp.N = N;
    kp.K = K;
    kp.apply_relu = apply_relu ? 1 : 0;
    kp.b_kmajor = b_nk ? 1 : 0;
    kp.out_bf16 = bf16 ? 1 : 0;
    kp.C = reinterpret_cast<uint16_t*>(C);
    kp.err = d.d_err;
    // generous bound: 2 s plus 2 us per k-block of the longest wait
    kp.timeout_ns = 2000000000ull + 2000ull * (uint64_t)pl.num_kb;
    {
        // test hook of the bounded waits (see KParams::test_drop_kb)
        const char* drop = getenv("GEMM_RELU_TEST_DROP_KB");
        if (drop && *drop) {
            const long kb = strtol(drop, nullptr, 10);
            if (kb < 0 || kb >= pl.num_kb || pl.cluster != 1) return GEMM_ERR_INVALID_ARG;
            kp.test_drop_kb = (int32_t)kb + 1;
            kp.timeout_ns = kTestTimeoutNs;
        }
    }
    if (pl.sk_tiles > 0) {
        StreamBuffers& sb = buffers_for_locked(d, st);
        int rc = grow(reinterpret_cast<void**>(&sb.ws), &sb.ws_bytes, (size_t)pl.workspace_bytes, st, false);
        if (rc != GEMM_OK) return rc;
        // one arrival counter per split tile, then max_slots ready flags each
        rc = grow(reinterpret_cast<void**>(&sb.counters), &sb.counter_bytes,
                  (size_t)pl.counter_count * (1 + (size_t)pl.max_slots) * sizeof(uint32_t), st, true);
        if (rc != GEMM_OK) return rc;
        kp.ws = sb.ws;
        kp.counters = sb.counters;
    }
    // Neither A's nor B's row pitch a multiple of 128 bytes: the launch
    // also copies A to a 128-byte pitch (KParams::pack_sync) when the plan
    // says it pays
    void* A2 = nullptr;
    uint64_t a2_pitch = 0;  // elements
    if (pack_a_pays(pl, M, N, K, b_nk, forced ? force : nullptr)) {
        a2_pitch = ((uint64_t)K + 63) / 64 * 64;
        StreamBuffers& sb = buffers_for_locked(d, st);
        int rc = grow(&sb.packed, &sb.packed_bytes, (size_t)M * a2_pitch * 2, st, false);
        if (rc != GEMM_OK) return rc;
        rc = grow(reinterpret_cast<void**>(&sb.pack_sync), &sb.pack_sync_bytes, 2 * sizeof(uint32_t), st, true);
        if (rc != GEMM_OK) return rc;
        A2 = sb.packed;
        kp.pack_src = reinterpret_cast<const uint4*>(A);
        kp.pack_dst = reinterpret_cast<uint4*>(A2);
        kp.pack_rows = M;
        kp.pack_row_vecs = (int32_t)(K / 8);
        kp.pack_dst_pitch = (int64_t)(a2_pitch / 8);
        kp.pack_sync = sb.pack_sync;
    }
    Maps local;
    const Maps* m = &local;
    if (forced) {
        int rc = encode_maps(pl, A, B, C, M, N, K, b_nk, bf16, force, A2, a2_pitch, &local);
        if (rc != GEMM_OK) return rc;
    } else {
        auto& cache = g_maps[dev];
        const MapKey key{A, B, C, A2, M, N, K, (b_nk ? 1 : 0) | (bf16 ? 2 : 0)};
        auto it = cache.find(key);
        if (it == cache.end()) {
            int rc = encode_maps(pl, A, B, C, M, N, K, b_nk, bf16, nullptr, A2, a2_pitch, &local);
            if (rc != GEMM_OK) return rc;
            if (cache.size() >= kMapCacheEntries) cache.clear();
            it = cache.emplace(key, local).first;
        }
        m = &it->second;
    }
    kp.a3d = m->a3d;
    kp.b3d = m->b3d;
    if (pl.path == 3) {
        // M = 128 tile columns; B^T is MN-major when B is stored (K, N)
        kp.idesc = make_idesc_f16_f32(128u, (uint32_t)pl.mma_n, /*a_mn=*/!b_nk, /*b_mn=*/false, bf16);
        return launch_mode<2>(d, pl, kp, m->ta, m->tb, m->tb2, m->tc, m->ta2, st);
    }
    kp.idesc = make_idesc_f16_f32((uint32_t)pl.mma_m, (uint32_t)pl.mma_n, /*a_mn=*/false, /*b_mn=*/!b_nk, bf16);
    if (pl.path == 4) return launch_mode<3>(d, pl, kp, m->ta, m->tb, m->tb2, m->tc, m->ta2, st);
    if (pl.mma_n == 256) return launch_mode<0>(d, pl, kp, m->ta, m->tb, m->tb2, m->tc, m->ta2, st);
    if (pl.mma_n == 64) return launch_mode<5>(d, pl, kp, m->ta, m->tb, m->tb2, m->tc, m->ta2, st);
    return launch_mode<1>(d, pl, kp, m->ta, m->tb, m->tb2, m->tc, m->ta2, st);
}

// A launch gave up part-way (the error word is set): clear it and every
// counter, and report the timeout.  Caller holds g_mu.
int reset_after_error_locked(DeviceState& d) {
    cudaDeviceSynchronize();
    cudaMemset(d.d_err, 0, 16);
    for (auto& s : d.streams) {
        if (s.counters) cudaMemset(s.counters, 0, s.counter_bytes);
        if (s.pack_sync) cudaMemset(s.pack_sync, 0, s.pack_sync_bytes);
    }
    cudaDeviceSynchronize();
    cudaGetLastError();
    return GEMM_ERR_TIMEOUT;
}

}  // namespace rt
}  // namespace gr

using namespace gr;
using namespace gr::rt;

extern "C" int gemm_relu_ex(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                            int apply_relu, int b_layout, int dtype, void* stream) {
    if ((b_layout != GEMM_B_KN && b_layout != GEMM_B_NK) || (dtype != GEMM_DTYPE_F16 && dtype != GEMM_DTYPE_BF16))
        return GEMM_ERR_INVALID_ARG;
    int rc = check_args(A, B, C, M, N, K, true);
    if (rc != GEMM_OK) return rc;
    if (M == 0 || N == 0) return GEMM_OK;  // nothing to enqueue
    int dev;
    if ((rc = current_device(&dev)) != GEMM_OK) return rc;
    std::lock_guard<std::mutex> lock(g_mu);
    if ((rc = init_device_locked(dev)) != GEMM_OK) return rc;
    return run_device(A, B, C, M, N, K, apply_relu, b_layout == GEMM_B_NK, dtype == GEMM_DTYPE_BF16,
                      reinterpret_cast<cudaStream_t>(stream), dev);
}

extern "C" int gemm_relu(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                         int apply_relu, void* stream) {
    return gemm_relu_ex(A, B, C, M, N, K, apply_relu, GEMM_B_KN, GEMM_DTYPE_F16, stream);
}

extern "C" int gemm_relu_check_device_error(void* stream) {
    int dev;
    int rc = current_device(&dev);
    if (rc != GEMM_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.inited || !d.d_err) return d.inited ? d.status : GEMM_OK;
    int32_t err = 0;
    if (cudaMemcpy(&err, d.d_err, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (err == 0) return GEMM_OK;
    return reset_after_error_locked(d);
}

extern "C" const char* gemm_relu_status_string(int status) {
    switch (status) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
        case GEMM_ERR_ALIGNMENT: return "GEMM_ERR_ALIGNMENT";
        case GEMM_ERR_UNSUPPORTED_DEVICE: return "GEMM_ERR_UNSUPPORTED_DEVICE";
        case GEMM_ERR_OUT_OF_MEMORY: return "GEMM_ERR_OUT_OF_MEMORY";
        case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH";
        case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
        case GEMM_ERR_TOO_LARGE: return "GEMM_ERR_TOO_LARGE";
        default: return "GEMM_ERR_UNKNOWN";
    }
}

extern "C" void gemm_relu_shutdown(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int prev = -1;
    const bool have_dev = cudaGetDevice(&prev) == cudaSuccess;
    cudaGetLastError();
    for (int dev = 0; dev < kMaxDevices; ++dev) {
        DeviceState& d = g_dev[dev];
        if (!d.inited) continue;
        if (d.d_err || !d.streams.empty()) {
            cudaSetDevice(dev);
            cudaDeviceSynchronize();
            for (auto& s : d.streams) {
                cudaFree(s.ws);
                cudaFree(s.counters);
                cudaFree(s.packed);
                cudaFree(s.pack_sync);
                cudaFree(s.hA);
                cudaFree(s.hB);
                cudaFree(s.hC);
                if (s.h_err) cudaFreeHost(s.h_err);
                pipe_release(s);
            }
            cudaFree(d.d_err);
        }
        d = DeviceState();
        g_plans[dev].clear();
        g_maps[dev].clear();
    }
    if (have_dev) cudaSetDevice(prev);
    cudaGetLastError();
}
