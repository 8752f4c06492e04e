// Persistent, warp-specialised C = ReLU(A . B) kernel for sm_103a.
//
// Per CTA (224 threads, one CTA per SM; in the paired mode two CTAs on two
// SMs form a cluster and share each MMA, tcgen05 cta_group::2):
//   warps 0, 6  TMA producers: one thread each streams A's (warp 0) and B's
//               (warp 6) k-blocks into a ring of shared-memory stages
//               (128-byte swizzle), each stage guarded by a full/empty
//               mbarrier pair;
//   warp 1      allocates tensor memory; one thread issues tcgen05.mma
//               (fp16 or bf16 inputs -> fp32, 128 x N x 16 per instruction) into one
//               of two TMEM accumulators and commits stage releases;
//   warps 2-5   epilogue: TMEM -> registers (each warp owns a 32-lane
//               quarter of the accumulator), ReLU, round to fp16/bf16, store to
//               C; or, for a tile split along K, store an fp32 partial and
//               let the last CTA to finish sum the partials in slot order.
//               (Warp 2 also initialises the barriers at set-up, while the
//               producer warps build their state.)
// B is read as stored: (K, N) row-major (an MN-major MMA operand) or
// (N, K) row-major (K-major, C = ReLU(A . B^T)); the layout and the element
// type are runtime flags that change only descriptors, copy coordinates and
// the final rounding.
// The two accumulators let the epilogue of tile i overlap the mainloop of
// tile i+1.  Every wait is bounded: on timeout the CTA records an error
// word, tells its other roles to stop, lets in-flight copies and MMAs land,
// frees its tensor memory and returns.
//
// The schedule follows the tile/pipeline recipe of the TileLang GEMM+ReLU
// example ("Writing High-Performance Kernels in TileLang", GEMM section:
// shared-memory A/B tiles, a pipelined K loop, a tile-level MMA into a
// float accumulator, ReLU on the accumulator, copy out), rebuilt for
// Blackwell: TMA + mbarriers instead of cp.async, tcgen05 + TMEM instead of
// register fragments, and a persistent stream-K grid instead of one CTA per
// tile.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ptx.cuh"
#include "schedule.h"

namespace gr {

constexpr int kThreads = 224;
constexpr uint32_t kEpiThreads = 128;
constexpr uint32_t kEpiBarrier = 1;  // named barrier id for the epilogue warps
constexpr int kMaxStagesDev = 16;
constexpr uint64_t kTestTimeoutNs = 1000000;  // wait limit of a launch with the test hook set (1 ms)
constexpr uint32_t kOperandA = 128 * kBlockK * 2;  // bytes of one 128-row box of 64 k
constexpr uint32_t kSwizzleRow = 128;              // bytes per swizzled row
constexpr uint32_t kAtomBytes = 1024;              // 8 swizzled rows

enum : int32_t {
    kErrProducer = 0x11,
    kErrMmaStage = 0x21,
    kErrMmaAccum = 0x22,
    kErrEpilogue = 0x31,
    kErrFinal = 0x41,
    kErrConfig = 0x51,
};

struct __align__(8) Ctrl {
    uint64_t full[kMaxStagesDev];
    uint64_t empty[kMaxStagesDev];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t final_bar;
    uint64_t exch_bar;  // cluster split-K: the peers' partials are ready (rank 0)
    uint64_t peer_free;  // tiled cluster split-K: the peer's ring is idle (its MMAs are done)
    uint64_t fix_bar[4];  // split-K fixup of a CTA's final item: 64-column units of the partials landed
    uint32_t tmem_addr;
    int32_t abort_flag;
    int32_t last_flag;
    // where the stage-arming producer stopped (next stage, its phase parity,
    // whether the ring has wrapped) and how many fix_bar units the split-K
    // fixup armed: what an aborting CTA waits for before its shared memory
    // is released
    int32_t ring_s, ring_ph, ring_lap;
    int32_t fix_armed;
};
static_assert(sizeof(Ctrl) <= 1024, "control block exceeds its reserved 1 KiB");

struct KParams {
    gemm_relu_plan_t plan;
    int64_t M, N, K;
    int32_t apply_relu;
    int32_t b_kmajor;     // B stored (N, K) row-major (C = ReLU(A . B^T)) instead of (K, N)
    int32_t out_bf16;     // elements are bfloat16 (inputs and C) instead of binary16
    // 3-D tensor maps (64-element column blocks as a third dimension): one
    // copy fetches all 64-k blocks of a stage's A rows (a3d), or all
    // 64-column chunks / 64-k blocks of its B (b3d), instead of one copy each.
    // B stored (K, N) with N not a multiple of 64: the 3-D map covers the
    // whole chunks only, and a CTA whose columns reach the partial chunk
    // loads 64-column 2-D boxes through the second map of B instead.
    int32_t a3d, b3d;
    uint32_t idesc;
    uint64_t timeout_ns;
    // Test hook of the bounded waits, 0 in every normal call.  k + 1: the
    // producers of every CTA leave k-block k of the CTA's first work item
    // uncopied (its stage is still armed for the bytes), so the MMA warp's
    // wait for that stage runs out; the host pairs it with a short
    // timeout_ns and a plan without clusters.
    int32_t test_drop_kb;
    // A copied to a 128-byte row pitch inside the launch (plans with
    // pack_a, when neither operand's row pitch is a multiple of 128 bytes):
    // before its first tile, each CTA's epilogue warps copy their share of
    // A's rows to pack_dst and count the CTA on pack_sync[0]; the producer
    // of A's copies waits until every CTA has counted itself before the
    // first copy of its second work item, and from then on reads A through
    // the second map of A.  pack_sync[1] counts CTAs that have finished the
    // launch; the last one resets both words.  pack_sync null: no copy.
    const uint4* pack_src;
    uint4* pack_dst;
    int64_t pack_rows;
    int64_t pack_dst_pitch;  // 16-byte vectors
    int32_t pack_row_vecs;   // 16-byte vectors of a row of A
    uint32_t* pack_sync;
    uint16_t* C;          // 16-bit words of C (binary16 or bfloat16)
    float* ws;            // stream-K partial tiles: [sk_tile][slot][col][128 lanes]
    uint32_t* counters;   // stream-K arrivals, one per stream-K tile, zero between launches
    int32_t* err;         // first error code of the launch (0 = none)
};

// kMode 0: C tile 128 x 256; 1: C tile 128 x 128; 5: C tile 128 x 64;
// 2: swapped operands (C tile mpad x 128: B^T is the MMA A operand, A^T the
// MMA B operand); 3: CTA pair, C tile 256 x 256 (each CTA holds 128 rows of
// A and 128 columns of B, and accumulates its 128 rows x 256 columns).
template <int kMode>
struct ModeTraits {
    static_assert(kMode == 0 || kMode == 1 || kMode == 2 || kMode == 3 || kMode == 5, "unknown kernel mode");
    static constexpr bool kSwap = (kMode == 2);
    static constexpr bool kPair = (kMode == 3);
    static constexpr int kCG = kPair ? 2 : 1;
    static constexpr uint32_t kBN = (kMode == 5) ? 64 : (kMode == 1) ? 128 : 256;  // C columns per tile
    static constexpr uint32_t kTileM = kPair ? 256 : 128;      // C rows per tile (normal)
    static constexpr uint32_t kBCols = kPair ? kBN / 2 : kBN;  // B columns loaded per CTA
    static constexpr uint32_t kBChunks = kBCols / 64;          // their 64-wide chunks (B stored (K, N))
    // k-rows per ring stage (the plan's block_k): 128 (8 MMAs per stage, so
    // that the MMA warp's fixed per-stage work -- barrier wait, fence,
    // commit -- is paid once per 8 MMAs), except for the 256-column tiles:
    // their MMAs already outlast that work, and 64-row stages keep the ring
    // twice as deep (128 x 256: 128-row stages would leave only two)
    static constexpr uint32_t kBK = (kMode == 0 || kMode == 3) ? kBlockK : 2 * kBlockK;
    static constexpr uint32_t kSub = kBK / kBlockK;  // 64-k boxes per stage
};

// Bounded wait on an mbarrier phase.  Returns false if this CTA is aborting.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, Ctrl* ctrl,
                                           const KParams& p, int32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    volatile int32_t* abort_flag = &ctrl->abort_flag;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            *abort_flag = 1;
            atomicCAS(p.err, 0, site);
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag (used at teardown, when the
// point is to let outstanding work finish).
__device__ __forceinline__ bool wait_phase_for(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) return false;
    return true;
}

__device__ __forceinline__ float relu_if(float x, int32_t apply) {
    // x > 0 ? x : +0 also maps -0 and NaN to +0
    return apply ? (x > 0.0f ? x : 0.0f) : x;
}

// Two fp32 values rounded to nearest-even 16-bit floats, a in the low half.
__device__ __forceinline__ uint32_t pack2(float a, float b, int32_t bf16) {
    if (bf16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint16_t round16(float x, int32_t bf16) {
    if (bf16) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
    return __half_as_ushort(__float2half_rn(x));
}

// ------------------------------------------------------------------ roles
//
// The producer and MMA roles are single threads whose k-block loop is on
// the critical path of the tensor pipe: every instruction latency in it is
// exposed.  So the loop runs from registers only: the plan is copied once,
// ring stage / phase advance without division, barrier addresses are base +
// 8 * stage, and shared-memory descriptors are built once and advanced by
// adding to their start-address field (a 14-bit field of 16-byte units that
// cannot carry: shared addresses stay below 256 KiB).

// A TMA producer thread walks the work items and k-blocks, waits for a free
// ring stage, and issues the stage's copies (the kernel runs two: one for
// A's copies, which also arms each stage, one for B's).  issue() keeps its
// position between calls.
template <int kMode>
struct Producer {
    using T = ModeTraits<kMode>;
    const KParams& p;
    Ctrl* ctrl;
    const CUtensorMap* tmA;
    const CUtensorMap* tmB;
    // second map of B (K, N): 64-column 2-D boxes, for the columns a 3-D
    // map of whole chunks leaves out
    const CUtensorMap* tmB2;
    const CUtensorMap* tmA2;  // A at its 128-byte pitch (see KParams::pack_sync)
    gemm_relu_plan_t pl;
    uint32_t stages, stride, a_bytes, rank, S, full0, empty0, tx_bytes;
    WorkIter wi;
    WorkItem w;
    bool have_item;
    bool armed;  // the current stage's expected bytes are armed already (prime: stage 0 of the fresh ring)
    int32_t kb, a_row, b_col;
    uint32_t s, ph;
    // an operand that only one row (column) of tiles reads is streamed
    // through L2 exactly once: its lines go first
    bool once_a, once_b;
    uint64_t pol_first;
    uint32_t a_sub_bytes;  // swapped: bytes of one 64-k box of A's padded rows
    bool b_nk;             // B stored (N, K): its boxes are (64 k) x (rows of N)
    bool a3d, b3d;         // one 3-D copy per operand and stage (see KParams)
    bool b_edge;           // B (K, N), b3d: this item's columns reach past the 3-D map's whole chunks
    int32_t part;          // copies this thread issues: 0 all, 1 A's (and arms each stage), 2 B's
    int32_t items;         // work items begun
    int32_t issued;        // stages armed and issued by run()
    int32_t drop_kb;       // test hook: k-block of the first item not copied (-1: none)

    __device__ __forceinline__ Producer(const KParams& p_, Ctrl* ctrl_, uint32_t stages_, uint32_t stride_,
                                        uint32_t a_bytes_, const CUtensorMap* tmA_, const CUtensorMap* tmB_,
                                        const CUtensorMap* tmB2_, const CUtensorMap* tmA2_, int32_t worker,
                                        uint32_t rank_, int32_t part_ = 0)
        : p(p_), ctrl(ctrl_), tmA(tmA_), tmB(tmB_), tmB2(tmB2_), tmA2(tmA2_), pl(p_.plan), stages(stages_),
          stride(stride_),
          a_bytes(a_bytes_), rank(rank_), have_item(false), armed(false), kb(0), a_row(0), b_col(0), s(0), ph(0) {
        S = (uint32_t)pl.num_stages;
        full0 = smem_u32(&ctrl->full[0]);
        empty0 = smem_u32(&ctrl->empty[0]);
        // a pair's copies all complete on the leader's barrier, which
        // expects the bytes of both CTAs
        tx_bytes = (T::kPair ? 2u : 1u) * (uint32_t)pl.stage_bytes;
        a_sub_bytes = (uint32_t)pl.tile_m * kSwizzleRow;
        b_nk = p_.b_kmajor != 0;
        once_a = pl.tiles_n == 1;
        once_b = pl.tiles_m == 1;
        a3d = p_.a3d != 0;
        b3d = p_.b3d != 0;
        b_edge = false;
        part = part_;
        items = 0;
        issued = 0;
        drop_kb = p_.test_drop_kb - 1;
        pol_first = l2_policy_evict_first();
        wi.init(pl, worker, (int32_t)rank);
    }

    // Issue up to `budget` k-blocks of copies (all remaining if < 0).
    // Returns false if the CTA is aborting.
    __device__ __forceinline__ bool issue(int32_t budget) { return run<false>(budget); }

    // L2 prefetches of the boxes of the next `budget` k-blocks, with no
    // barrier and no copy: safe before the previous kernel of the stream
    // has finished (a prefetch returns nothing; lines written meanwhile are
    // current in L2).  Call it on a copy: it advances the position.
    __device__ __forceinline__ void prefetch(int32_t budget) { run<true>(budget); }

    template <bool kPre>
    __device__ __forceinline__ void ld_pair(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t x, int32_t y) {
        if constexpr (kPre)
            tma_prefetch_2d(m, x, y);
        else
            tma_load_2d_pair(dst, m, bar, x, y);
    }

    template <bool kPre>
    __device__ __forceinline__ void ld(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t x, int32_t y,
                                       bool hinted) {
        if constexpr (kPre)
            tma_prefetch_2d(m, x, y);
        else
            tma_load_2d_maybe_hint(dst, m, bar, x, y, hinted, pol_first);
    }

    // 3-D copies at column block 0: (row or k, block)
    template <bool kPre>
    __device__ __forceinline__ void ld3(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t y, int32_t z,
                                        bool hinted) {
        if constexpr (kPre)
            tma_prefetch_3d(m, 0, y, z);
        else
            tma_load_3d_maybe_hint(dst, m, bar, 0, y, z, hinted, pol_first);
    }

    template <bool kPre>
    __device__ __forceinline__ void ld3_pair(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t y, int32_t z) {
        if constexpr (kPre)
            tma_prefetch_3d(m, 0, y, z);
        else
            tma_load_3d_pair(dst, m, bar, 0, y, z);
    }

    // Move to the next work item; false when there is none.
    __device__ __forceinline__ bool next_item() {
        if (!wi.next(pl, w)) return false;
        have_item = true;
        ++items;
        kb = w.kb0;
        // first row of A and first column of B this CTA loads
        if constexpr (T::kPair) {
            a_row = w.tm * (int32_t)T::kTileM + 128 * (int32_t)rank;
            b_col = w.tn * (int32_t)T::kBN + (int32_t)T::kBCols * (int32_t)rank;
        } else if constexpr (!T::kSwap) {
            a_row = w.tm * 128;
            b_col = w.tn * (int32_t)T::kBN;
        } else {
            a_row = w.tm * pl.tile_m;
            b_col = w.tn * pl.tile_n;
        }
        {
            constexpr int32_t kChunks = T::kSwap ? 2 : (int32_t)T::kBChunks;
            b_edge = b_col / 64 + kChunks > (int32_t)(p.N / 64);
        }
        return true;
    }

    // The first work item, for a call ahead of the set-up barrier (parameters
    // and arithmetic only).
    __device__ __forceinline__ void first_item() {
        if (!have_item) next_item();
    }

    // Everything before the first copy, for a call ahead of the dependency
    // wait so that it overlaps the previous kernel: the first work item
    // (parameters and arithmetic) and the first stage's expected-bytes
    // arrival (shared memory; the ring is fresh, so stage 0 needs no empty
    // wait).
    __device__ __forceinline__ void prime() {
        if (!have_item && !next_item()) return;
        if (s == 0 && ph == 0 && !armed) {
            arm();
            armed = true;
        }
    }

    // Expect the stage's bytes on its full barrier (a pair: the leader's,
    // which counts both CTAs' copies).
    __device__ __forceinline__ void arm() {
        if (part != 2 && (!T::kPair || rank == 0)) mbar_arrive_expect_tx(full0 + 8u * s, tx_bytes);
    }

    // The stage's copies from A's tensor map (its rows; the MMA B operand
    // when swapped) ...
    template <bool kPre>
    __device__ __forceinline__ void copies_a(uint32_t full, uint32_t a_dst, uint32_t b_dst, int32_t k0) {
        if constexpr (T::kPair) {
            const uint32_t full_leader = mapa_shared(full, 0);
            if (a3d) {
                ld3_pair<kPre>(a_dst, tmA, full_leader, a_row, k0 / kBlockK);
            } else {
#pragma unroll
                for (uint32_t i = 0; i < T::kSub; ++i)
                    ld_pair<kPre>(a_dst + i * kOperandA, tmA, full_leader, k0 + (int32_t)(i * kBlockK), a_row);
            }
        } else if constexpr (!T::kSwap) {
            if (a3d) {
                ld3<kPre>(a_dst, tmA, full, a_row, k0 / kBlockK, once_a);
            } else {
#pragma unroll
                for (uint32_t i = 0; i < T::kSub; ++i)
                    ld<kPre>(a_dst + i * kOperandA, tmA, full, k0 + (int32_t)(i * kBlockK), a_row, once_a);
            }
        } else {
            // MMA B operand: the (padded) rows of A, one box per 64 k
            if (a3d) {
                ld3<kPre>(b_dst, tmA, full, a_row, k0 / kBlockK, once_a);
            } else {
#pragma unroll
                for (uint32_t i = 0; i < T::kBK / kBlockK; ++i)
                    ld<kPre>(b_dst + i * a_sub_bytes, tmA, full, k0 + (int32_t)(i * kBlockK), a_row, once_a);
            }
        }
    }

    // ... and from B's (the MMA A operand when swapped).
    template <bool kPre>
    __device__ __forceinline__ void copies_b(uint32_t full, uint32_t a_dst, uint32_t b_dst, int32_t k0) {
        constexpr uint32_t kBChunk = T::kBK * kSwizzleRow;  // one 64-column chunk of B (K, N)
        if constexpr (T::kPair) {
            const uint32_t full_leader = mapa_shared(full, 0);
            if (b_nk) {
                // this CTA's kBCols rows of B, one K-major box per 64 k
                if (b3d) {
                    ld3_pair<kPre>(b_dst, tmB, full_leader, b_col, k0 / kBlockK);
                } else {
#pragma unroll
                    for (uint32_t i = 0; i < T::kSub; ++i)
                        ld_pair<kPre>(b_dst + i * T::kBCols * kSwizzleRow, tmB, full_leader,
                                      k0 + (int32_t)(i * kBlockK), b_col);
                }
            } else if (b3d && !b_edge) {
                // all of this CTA's 64-column chunks in one copy
                ld3_pair<kPre>(b_dst, tmB, full_leader, k0, b_col / 64);
            } else {
                // one 2-D box per chunk (b3d: the columns reach the partial
                // last chunk, through the second map)
                const CUtensorMap* m2 = b3d ? tmB2 : tmB;
#pragma unroll
                for (uint32_t j = 0; j < T::kBChunks; ++j)
                    ld_pair<kPre>(b_dst + j * kBChunk, m2, full_leader, b_col + 64 * (int32_t)j, k0);
            }
        } else if constexpr (!T::kSwap) {
            if (b_nk && b3d) {
                ld3<kPre>(b_dst, tmB, full, b_col, k0 / kBlockK, once_b);
            } else if (b_nk) {
                // the tile's kBN rows of B, K-major like A, one box per 64 k
#pragma unroll
                for (uint32_t i = 0; i < T::kSub; ++i)
                    ld<kPre>(b_dst + i * T::kBN * kSwizzleRow, tmB, full, k0 + (int32_t)(i * kBlockK), b_col,
                             once_b);
            } else if (b3d && !b_edge) {
                // all of the tile's 64-column chunks in one copy
                ld3<kPre>(b_dst, tmB, full, k0, b_col / 64, once_b);
            } else {
                // (b3d: the partial last chunk, through the 2-D second map)
                const CUtensorMap* m2 = b3d ? tmB2 : tmB;
#pragma unroll
                for (uint32_t j = 0; j < T::kBN / 64; ++j)
                    ld<kPre>(b_dst + j * kBChunk, m2, full, b_col + 64 * (int32_t)j, k0, once_b);
            }
        } else {
            // MMA A operand: the tile's 128 columns of B, one 64-wide chunk of
            // kBK k-rows per TMA box
            if (b3d && (b_nk || !b_edge)) {
                // one copy: the tile's B rows (B stored (N, K)) for every
                // 64 k, or both 64-column chunks (B (K, N))
                if (b_nk)
                    ld3<kPre>(a_dst, tmB, full, b_col, k0 / kBlockK, once_b);
                else
                    ld3<kPre>(a_dst, tmB, full, k0, b_col / 64, once_b);
            } else if (b3d) {
                // the partial last chunk: 2-D boxes through the second map
                ld<kPre>(a_dst, tmB2, full, b_col, k0, once_b);
                ld<kPre>(a_dst + kBChunk, tmB2, full, b_col + 64, k0, once_b);
            } else if (b_nk) {
                // B stored (N, K): the tile's B rows, one K-major box per 64 k
#pragma unroll
                for (uint32_t i = 0; i < T::kBK / kBlockK; ++i)
                    ld<kPre>(a_dst + i * 128u * kSwizzleRow, tmB, full, k0 + (int32_t)(i * kBlockK), b_col, once_b);
            } else {
                ld<kPre>(a_dst, tmB, full, b_col, k0, once_b);
                ld<kPre>(a_dst + kBChunk, tmB, full, b_col + 64, k0, once_b);
            }
        }
    }

    // Bounded wait until every CTA has copied its share of A to the
    // 128-byte pitch; then A's copies switch to that copy.
    __device__ __forceinline__ bool wait_packed() {
        volatile uint32_t* arrived = p.pack_sync;
        if (*arrived < gridDim.x) {
            volatile int32_t* abort_flag = &ctrl->abort_flag;
            const uint64_t t0 = globaltimer_ns();
            while (*arrived < gridDim.x) {
                if (*abort_flag) return false;
                if (globaltimer_ns() - t0 > p.timeout_ns) {
                    *abort_flag = 1;
                    atomicCAS(p.err, 0, kErrProducer);
                    return false;
                }
            }
        }
        __threadfence();
        fence_proxy_async_global();  // the other CTAs' stores, before this thread's TMA reads
        tmA = tmA2;
        return true;
    }

    template <bool kPre>
    __device__ __forceinline__ bool run(int32_t budget) {
        while (budget != 0) {
            if (!have_item || kb == w.kb1) {
                if (!next_item()) return true;
                if constexpr (!kPre && !T::kSwap) {
                    if (items == 2 && part != 2 && p.pack_sync && !wait_packed()) return false;
                }
            }
            if constexpr (!kPre) {
                if (!armed) {
                    if (!wait_phase(empty0 + 8u * s, ph ^ 1u, ctrl, p, kErrProducer)) return false;
                    arm();
                }
                armed = false;
            }
            const uint32_t full = full0 + 8u * s;
            const uint32_t a_dst = stages + s * stride;
            const uint32_t b_dst = a_dst + a_bytes;
            const int32_t k0 = kb * (int32_t)T::kBK;
            if (kPre || kb != drop_kb || items != 1) {
                if (part != 2) copies_a<kPre>(full, a_dst, b_dst, k0);
                if (part != 1) copies_b<kPre>(full, a_dst, b_dst, k0);
            }
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
            ++kb;
            if constexpr (!kPre) ++issued;
            if (budget > 0) --budget;
        }
        return true;
    }

    // Record where the stage-arming thread stopped (for the drain of an
    // aborting CTA; a pair's stages are armed in its leader only).
    __device__ __forceinline__ void save_ring() {
        if (part != 2 && (!T::kPair || rank == 0)) {
            ctrl->ring_s = (int32_t)s;
            ctrl->ring_ph = (int32_t)ph;
            ctrl->ring_lap = issued >= (int32_t)S ? 1 : 0;
        }
    }
};

template <int kMode>
__device__ __forceinline__ void mma_role(const KParams& p, Ctrl* ctrl, uint32_t stages,
                                         uint32_t stride, uint32_t a_bytes, uint32_t tmem_base,
                                         int32_t worker, uint32_t rank) {
    using T = ModeTraits<kMode>;
    const gemm_relu_plan_t pl = p.plan;
    const uint32_t S = (uint32_t)pl.num_stages;
    const uint32_t idesc = p.idesc;
    const uint32_t cols_per_buf = (uint32_t)pl.tmem_cols / 2;
    const uint32_t full0 = smem_u32(&ctrl->full[0]);
    const uint32_t empty0 = smem_u32(&ctrl->empty[0]);
    const uint32_t tfull0 = smem_u32(&ctrl->tmem_full[0]);
    const uint32_t tempty0 = smem_u32(&ctrl->tmem_empty[0]);
    // Descriptors of stage 0 and, per MMA of a stage, the offset (16-byte
    // units) of each operand's k16 slice:
    //   K-major operand (A; B stored (N, K); when swapped A^T, and B^T of a
    //     B stored (N, K)): +32 bytes inside the swizzled row, and one box
    //     of rows further per 64 k;
    //   MN-major operand (B stored (K, N); B^T of it when swapped): +16
    //     k-rows (2 atoms); its 64-wide chunks are LBO apart.
    constexpr uint32_t kK = T::kBK / 16;  // MMAs per stage
    constexpr uint32_t kMNStep = (2 * kAtomBytes) >> 4;
    const bool b_nk = p.b_kmajor != 0;
    uint64_t a_desc0, b_desc0;
    uint32_t a_off[kK], b_off[kK];
    if constexpr (T::kSwap) {
        const uint32_t a_box16 = (128u * kSwizzleRow) >> 4;  // one 64-k box of the tile's B rows
        const uint32_t b_box16 = ((uint32_t)pl.tile_m * kSwizzleRow) >> 4;  // one 64-k box of A's rows
        a_desc0 = b_nk ? make_sw128_desc(stages, 16, kAtomBytes)
                       : make_sw128_desc(stages, T::kBK * kSwizzleRow, kAtomBytes);
        b_desc0 = make_sw128_desc(stages + a_bytes, 16, kAtomBytes);
#pragma unroll
        for (uint32_t k = 0; k < kK; ++k) {
            a_off[k] = b_nk ? (k / 4) * a_box16 + (k % 4) * 2u : k * kMNStep;
            b_off[k] = (k / 4) * b_box16 + (k % 4) * 2u;
        }
    } else {
        // A: one 128-row K-major box per 64 k; B (N, K): one box of its rows
        // per 64 k; B (K, N): 64-column chunks of kBK k-rows
        constexpr uint32_t kARows16 = kOperandA >> 4;
        constexpr uint32_t kBRows16 = ((T::kPair ? T::kBCols : T::kBN) * kSwizzleRow) >> 4;
        a_desc0 = make_sw128_desc(stages, 16, kAtomBytes);
        b_desc0 = b_nk ? make_sw128_desc(stages + a_bytes, 16, kAtomBytes)
                       : make_sw128_desc(stages + a_bytes, T::kBK * kSwizzleRow, kAtomBytes);
#pragma unroll
        for (uint32_t k = 0; k < kK; ++k) {
            a_off[k] = (k / 4) * kARows16 + (k % 4) * 2u;
            b_off[k] = b_nk ? (k / 4) * kBRows16 + (k % 4) * 2u : k * kMNStep;
        }
    }
    const uint32_t stride16 = stride >> 4;
    WorkIter wi;
    wi.init(pl, worker, (int32_t)rank);
    WorkItem w;
    uint32_t s = 0, ph = 0, local = 0;
    // The set-up above reads only parameters, so it overlaps the previous
    // kernel (pinned here so that it is not sunk past the wait); the loop
    // reads only shared and tensor memory, but its timeout path writes the
    // error word, so it starts after the wait.
    asm volatile("" : "+l"(a_desc0), "+l"(b_desc0)::"memory");
    grid_dependency_wait();
    while (wi.next(pl, w)) {
        const uint32_t buf = local & 1u;
        const uint32_t bph = (local >> 1) & 1u;
        if (!wait_phase(tempty0 + 8u * buf, bph ^ 1u, ctrl, p, kErrMmaAccum)) return;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * cols_per_buf;
        for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
            if (!wait_phase(full0 + 8u * s, ph, ctrl, p, kErrMmaStage)) return;
            tc_fence_after();
            const uint64_t a_desc = a_desc0 + (uint64_t)(s * stride16);
            const uint64_t b_desc = b_desc0 + (uint64_t)(s * stride16);
            const uint32_t acc = (kb > w.kb0) ? 1u : 0u;
#pragma unroll
            for (uint32_t k = 0; k < kK; ++k)
                mma_f16_ss<T::kCG>(d_tmem, a_desc + a_off[k], b_desc + b_off[k], idesc, k > 0 ? 1u : acc);
            // stage free (in both CTAs of a pair) once these MMAs are done
            mma_commit<T::kCG>(empty0 + 8u * s, 0x3);
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
        mma_commit<T::kCG>(tfull0 + 8u * buf, 0x3);  // accumulator ready
        ++local;
    }
}

// ------------------------------------------------------------------ epilogue
//
// The epilogue works on chunks of kChunk accumulator columns of its TMEM
// lane (= one output row for the tiled paths, one output column for the
// swapped path):
//   tiled / pair: 64 columns.  ReLU + round to fp16, written by each warp
//     into its own 128B-swizzled 32-row x 128-byte staging buffer (two per
//     warp, alternating), then stored by one TMA bulk copy per warp; the
//     copy clips rows >= M and columns >= N.
//   swapped: 16 columns (16 rows of C).  Stored directly: a warp writes 32
//     consecutive elements of one C row per instruction.

template <int kMode>
struct EpiTraits {
    static constexpr int kChunk = ModeTraits<kMode>::kSwap ? 16 : 64;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 q) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(q.x), "r"(q.y), "r"(q.z),
                 "r"(q.w)
                 : "memory");
}

// Tiled / pair paths: one 64-column chunk of this warp's 32 rows -> C.
// `lane` is the row within the warp's slab; `sbuf` alternates buffers.
__device__ __forceinline__ void sink_tma(const CUtensorMap* tmC, uint32_t stage_buf, uint32_t lane,
                                         const float* v, int32_t apply_relu, int32_t bf16, int64_t col,
                                         int64_t row0, int64_t M, int64_t N) {
    // the copy issued two chunks ago from this buffer must have read it
    if (lane == 0) bulk_wait_group_read<1>();
    __syncwarp();
    const uint32_t row_addr = stage_buf + lane * 128u;
#pragma unroll
    for (uint32_t u = 0; u < 8; ++u) {
        uint4 q;
        q.x = pack2(relu_if(v[8 * u + 0], apply_relu), relu_if(v[8 * u + 1], apply_relu), bf16);
        q.y = pack2(relu_if(v[8 * u + 2], apply_relu), relu_if(v[8 * u + 3], apply_relu), bf16);
        q.z = pack2(relu_if(v[8 * u + 4], apply_relu), relu_if(v[8 * u + 5], apply_relu), bf16);
        q.w = pack2(relu_if(v[8 * u + 6], apply_relu), relu_if(v[8 * u + 7], apply_relu), bf16);
        st_shared_v4(row_addr + ((u ^ (lane & 7u)) << 4), q);  // 128-byte swizzle
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (col < N && row0 < M) tma_store_2d(tmC, stage_buf, (int32_t)col, (int32_t)row0);
        bulk_commit_group();
    }
}

// Swapped path: 16 accumulator columns (= C rows m0 .. m0+15) of C column n.
__device__ __forceinline__ void sink_direct_swap(uint16_t* C, const float* v, int32_t apply_relu,
                                                 int32_t bf16, int64_t n, int64_t m0, int64_t M, int64_t N) {
    if (n >= N) return;
#pragma unroll
    for (int j = 0; j < 16; ++j)
        if (m0 + j < M) C[(m0 + j) * N + n] = round16(relu_if(v[j], apply_relu), bf16);
}

template <int kMode>
__device__ __forceinline__ void tmem_load_chunk(uint32_t taddr, float* v) {
    if constexpr (EpiTraits<kMode>::kChunk == 64) {
        tmem_load_64cols(taddr, *reinterpret_cast<float(*)[64]>(v));
    } else {
        tmem_load_16cols(taddr, *reinterpret_cast<float(*)[16]>(v));
    }
}

template <int kMode>
__device__ __forceinline__ void epilogue_role(const KParams& p, Ctrl* ctrl, uint32_t tmem_base,
                                              int32_t worker, uint32_t rank, const CUtensorMap* tmC,
                                              uint32_t stages, uint32_t staging) {
    using T = ModeTraits<kMode>;
    constexpr int kChunk = EpiTraits<kMode>::kChunk;
    constexpr int kQ = kChunk / 4;  // float4 groups per chunk
    const gemm_relu_plan_t pl = p.plan;
    const int64_t M = p.M, N = p.N;
    const int32_t apply_relu = p.apply_relu;
    uint16_t* const C = p.C;
    const int32_t out_bf16 = p.out_bf16;
    float* const ws = p.ws;
    const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t quarter = warp & 3u;  // TMEM lanes a warp may access: 32 * (warp % 4) ...
    const uint32_t lane_row = quarter * 32 + lane;  // TMEM lane = accumulator row
    // swapped: the C column (within the tile) of this lane (the M = 128 MMA
    // puts accumulator row r in lane r)
    const int32_t swap_col = (int32_t)lane_row;
    const uint32_t half = T::kPair ? rank : 0u;      // which 128 rows of a pair tile
    const uint32_t cols_per_buf = (uint32_t)pl.tmem_cols / 2;
    const uint32_t ncols = (uint32_t)pl.mma_n;
    const bool shared_reduction = concurrent_split(pl);
    const int64_t tile_elems = (int64_t)128 * ncols;
    const uint32_t my_staging = staging + quarter * 8192u;  // two 4 KiB buffers per warp
    uint32_t sbuf = 0;
    volatile int32_t* last_flag = &ctrl->last_flag;
    WorkIter wi;
    wi.init(pl, worker, (int32_t)rank);
    WorkItem w;
    uint32_t local = 0;
    float v[kChunk];

    if constexpr (!T::kSwap) {
        if (p.pack_sync) {
            // this CTA's share of the copy of A to a 128-byte pitch: rows
            // blockIdx.x * 4 + quarter, then every 4 * gridDim.x rows; one
            // warp per row at a time, eight 16-byte loads in flight per lane
            const int64_t nw = (int64_t)gridDim.x * 4;
            for (int64_t r = (int64_t)blockIdx.x * 4 + quarter; r < p.pack_rows; r += nw) {
                const uint4* src = p.pack_src + r * p.pack_row_vecs;
                uint4* dst = p.pack_dst + r * p.pack_dst_pitch;
                for (int32_t c0 = 0; c0 < p.pack_row_vecs; c0 += 8 * 32) {
                    uint4 q[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int32_t c = c0 + u * 32 + (int32_t)lane;
                        if (c < p.pack_row_vecs) q[u] = __ldcs(src + c);
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int32_t c = c0 + u * 32 + (int32_t)lane;
                        if (c < p.pack_row_vecs) dst[c] = q[u];
                    }
                }
            }
            fence_proxy_async_global();  // before other CTAs' TMA reads of these rows
            __threadfence();
            named_bar_sync(kEpiBarrier, kEpiThreads);
            if (threadIdx.x == 64) atomicAdd(p.pack_sync, 1u);
        }
    }

    // where chunk c of this thread's lane goes
    auto sink = [&](const WorkItem& it, uint32_t c) {
        if constexpr (T::kSwap) {
            if (swap_col < pl.tile_n)
                sink_direct_swap(C, v, apply_relu, out_bf16, (int64_t)it.tn * pl.tile_n + swap_col,
                                 (int64_t)it.tm * pl.tile_m + c, M, N);
        } else {
            const int64_t row0 = (int64_t)it.tm * T::kTileM + 128 * half + 32 * quarter;
            const int64_t col = (int64_t)it.tn * T::kBN + c;
            sink_tma(tmC, my_staging + sbuf * 4096u, lane, v, apply_relu, out_bf16, col, row0, M, N);
            sbuf ^= 1u;
        }
    };

    while (wi.next(pl, w)) {
        const uint32_t buf = local & 1u;
        const uint32_t bph = (local >> 1) & 1u;
        bool ok = wait_phase(smem_u32(&ctrl->tmem_full[buf]), bph, ctrl, p, kErrEpilogue);
        ok = named_bar_and(kEpiBarrier, kEpiThreads, ok);  // all epilogue warps agree
        if (!ok) break;
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((quarter * 32u) << 16) + buf * cols_per_buf;
        // accumulator buffer back to the MMA warp
        auto release_tmem = [&]() {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (T::kPair)
                    mbar_arrive_cluster(mapa_shared(smem_u32(&ctrl->tmem_empty[buf]), 0));
                else
                    mbar_arrive(smem_u32(&ctrl->tmem_empty[buf]));
            }
        };
        if (w.nslots == 1) {
            for (uint32_t c = 0; c < ncols; c += kChunk) {
                __syncwarp();  // tcgen05.ld is warp-collective
                tmem_load_chunk<kMode>(taddr + c, v);
                sink(w, c);
            }
            release_tmem();
            ++local;
            continue;
        }
        // A tile split along K (one share per slot).  Each CTA first takes
        // an arrival ticket.  All but the last write their fp32 partial and
        // then raise their slot's ready flag; the last waits for the other
        // slots' flags and sums the slots in slot order, its own share read
        // straight from tensor memory, so its partial is never written.
        // Partials are per CTA (one per pair half), as float4 groups of 4
        // columns interleaved by lane:
        //   element (col, lane) at ((col / 4) * 128 + lane) * 4 + col % 4
        // so a warp writes / reads 512 contiguous bytes per instruction.
        if (cluster_split(pl)) {
            // Cluster split-K.  Each CTA holds one K range of this tile (its
            // only item, so its ring is idle); rank 0 adds the other ranks'
            // fp32 accumulators to its own in rank order.  Partials are
            // lane-interleaved float4 groups as for global partials.
            //   swapped (small partials): rank r > 0 pushes its partial
            //     into slot r - 1 of rank 0's exchange buffer (behind the
            //     ring; the plan reserves one slot, cluster = 2) with
            //     asynchronous remote stores whose bytes complete rank 0's
            //     exchange barrier; rank 0 reads them locally.
            //   tiled, >= 128 columns: a symmetric exchange (below);
            //   tiled, narrower: rank r > 0 leaves its partial in its own
            //     ring and arrives on rank 0's barrier; rank 0 reads it over
            //     DSMEM.
            // The cluster barrier at teardown keeps the ranks alive until
            // rank 0 is done.
            const uint32_t exch = smem_u32(&ctrl->exch_bar);
            const uint32_t slot_bytes = ncols * 128u * 4u;
            // bounded wait, with cluster acquire, on a one-shot barrier
            auto wait_cluster = [&](uint32_t bar) {
                const uint64_t t0 = globaltimer_ns();
                volatile int32_t* abort_flag = &ctrl->abort_flag;
                while (!mbar_try_wait_acq_cluster(bar, 0)) {
                    if (*abort_flag || globaltimer_ns() - t0 > p.timeout_ns) {
                        *abort_flag = 1;
                        atomicCAS(p.err, 0, kErrEpilogue);
                        return false;
                    }
                }
                return true;
            };
            if (!T::kSwap && pl.cluster == 2 && ncols >= 128) {
                // Tiled, two ranks: a symmetric exchange.  Rank r owns the
                // columns [r * h, (r + 1) * h) of the tile (h = ncols / 2).
                // Once both rings are idle (each rank's MMAs are done), each
                // rank pushes the other's columns of its fp32 accumulator
                // into the other's ring (asynchronous remote stores whose
                // bytes complete the receiver's exchange barrier), then sums
                // its own columns -- rank 0's K range first -- and stores them.
                const uint32_t h = ncols / 2;
                const uint32_t peer = rank ^ 1u;
                if (threadIdx.x == 64) mbar_arrive_cluster(mapa_shared(smem_u32(&ctrl->peer_free), peer));
                bool ready = named_bar_and(kEpiBarrier, kEpiThreads, wait_cluster(smem_u32(&ctrl->peer_free)));
                if (!ready) {
                    release_tmem();
                    break;
                }
                const uint32_t xbuf = mapa_shared(stages, peer);
                const uint32_t xbar = mapa_shared(exch, peer);
                for (uint32_t c = 0; c < h; c += kChunk) {
                    __syncwarp();
                    tmem_load_chunk<kMode>(taddr + peer * h + c, v);
#pragma unroll
                    for (int j = 0; j < kQ; ++j)
                        st_async_v4_cluster(xbuf + (((c / 4 + j) * 128u + lane_row) << 4),
                                            make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                                       __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3])),
                                            xbar);
                }
                ready = named_bar_and(kEpiBarrier, kEpiThreads, wait_cluster(exch));
                if (!ready) {
                    release_tmem();
                    break;
                }
                for (uint32_t c = 0; c < h; c += kChunk) {
                    __syncwarp();
                    tmem_load_chunk<kMode>(taddr + rank * h + c, v);
                    float4 x[kQ];
#pragma unroll
                    for (int j = 0; j < kQ; ++j) x[j] = ld_shared_f4(stages + (((c / 4 + j) * 128u + lane_row) << 4));
                    // (rank 0's share + rank 1's: fp32 addition of two terms
                    // does not depend on the operand order)
#pragma unroll
                    for (int j = 0; j < kQ; ++j) {
                        v[4 * j] += x[j].x;
                        v[4 * j + 1] += x[j].y;
                        v[4 * j + 2] += x[j].z;
                        v[4 * j + 3] += x[j].w;
                    }
                    sink(w, rank * h + c);
                }
                release_tmem();
                ++local;
                continue;
            }
            if (T::kSwap && rank != 0) {
                const uint32_t xbuf = mapa_shared(staging + (rank - 1u) * slot_bytes, 0);
                const uint32_t xbar = mapa_shared(exch, 0);
                for (uint32_t c = 0; c < ncols; c += kChunk) {
                    __syncwarp();
                    tmem_load_chunk<kMode>(taddr + c, v);
#pragma unroll
                    for (int j = 0; j < kQ; ++j)
                        st_async_v4_cluster(xbuf + (((c / 4 + j) * 128u + lane_row) << 4),
                                            make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                                       __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3])),
                                            xbar);
                }
                release_tmem();
                ++local;
                continue;
            }
            if (rank != 0) {
                for (uint32_t c = 0; c < ncols; c += kChunk) {
                    __syncwarp();
                    tmem_load_chunk<kMode>(taddr + c, v);
#pragma unroll
                    for (int j = 0; j < kQ; ++j)
                        st_shared_v4(stages + (((c / 4 + j) * 128u + lane_row) << 4),
                                     make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                                __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3])));
                }
                release_tmem();
                fence_acq_rel_cluster();
                named_bar_sync(kEpiBarrier, kEpiThreads);
                if (threadIdx.x == 64) mbar_arrive_cluster(mapa_shared(exch, 0));
                ++local;
                continue;
            }
            bool ready = named_bar_and(kEpiBarrier, kEpiThreads, wait_cluster(exch));
            if (!ready) {
                release_tmem();
                break;
            }
            for (uint32_t c = 0; c < ncols; c += kChunk) {
                __syncwarp();
                tmem_load_chunk<kMode>(taddr + c, v);  // rank 0's share
                for (uint32_t r = 1; r < (uint32_t)pl.cluster; ++r) {
                    float4 x[kQ];
#pragma unroll
                    for (int j = 0; j < kQ; ++j) {
                        const uint32_t off = ((c / 4 + j) * 128u + lane_row) << 4;
                        if constexpr (T::kSwap)
                            x[j] = ld_shared_f4(staging + (r - 1u) * slot_bytes + off);
                        else
                            x[j] = ld_shared_cluster_f4(mapa_shared(stages + off, r));
                    }
#pragma unroll
                    for (int j = 0; j < kQ; ++j) {
                        v[4 * j] += x[j].x;
                        v[4 * j + 1] += x[j].y;
                        v[4 * j + 2] += x[j].z;
                        v[4 * j + 3] += x[j].w;
                    }
                }
                sink(w, c);
            }
            release_tmem();
            ++local;
            continue;
        }
        const int64_t split_id = T::kPair ? (int64_t)w.sk_index * 2 + rank : (int64_t)w.sk_index;
        uint32_t* const counter = p.counters + split_id;
        uint32_t* const flags = p.counters + pl.counter_count + split_id * pl.max_slots;
        if (shared_reduction) {
            // Every slot of this tile runs at the same time (at most one split
            // item per worker), so the reduction is shared: slot s owns
            // columns [s * own, (s + 1) * own).  Each slot publishes the
            // columns the others own, waits (bounded) until all others have
            // published, then sums and stores its own columns.  The last
            // slot to finish reading resets the counter and flags.
            const float4* const tbase = reinterpret_cast<const float4*>(ws + split_id * pl.max_slots * tile_elems);
            const int64_t sq = tile_elems / 4;
            const uint32_t own = ncols / (uint32_t)w.nslots;
            const uint32_t own0 = (uint32_t)w.slot * own;
            float4* const mine = const_cast<float4*>(tbase) + w.slot * sq;
            for (uint32_t c = 0; c < ncols; c += kChunk) {
                if (c >= own0 && c < own0 + own) continue;
                __syncwarp();
                tmem_load_chunk<kMode>(taddr + c, v);
#pragma unroll
                for (int j = 0; j < kQ; ++j)
                    __stcg(mine + (int64_t)(c / 4 + j) * 128 + lane_row,
                           make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
            }
            named_bar_sync(kEpiBarrier, kEpiThreads);
            if (threadIdx.x == 64) {
                __threadfence();  // the partial is visible before the flag
                atomicExch(flags + w.slot, 1u);
            }
            bool ready = true;
            if (threadIdx.x == 64) {
                volatile uint32_t* vf = flags;
                volatile int32_t* abort_flag = &ctrl->abort_flag;
                const uint64_t t0 = globaltimer_ns();
                for (int32_t sl = 0; sl < w.nslots && ready; ++sl) {
                    if (sl == w.slot) continue;
                    while (vf[sl] == 0u) {
                        if (*abort_flag || globaltimer_ns() - t0 > p.timeout_ns) {
                            *abort_flag = 1;
                            atomicCAS(p.err, 0, kErrEpilogue);
                            ready = false;
                            break;
                        }
                    }
                }
                __threadfence();
            }
            ready = named_bar_and(kEpiBarrier, kEpiThreads, ready);
            if (!ready) {
                release_tmem();
                break;
            }
            for (uint32_t c = own0; c < own0 + own; c += kChunk) {
                __syncwarp();
                tmem_load_chunk<kMode>(taddr + c, v);  // own share
                float4 acc[kQ];
#pragma unroll
                for (int j = 0; j < kQ; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                const float4* src = tbase + (int64_t)(c / 4) * 128 + lane_row;
                for (int32_t sl = 0; sl < w.nslots; ++sl) {
                    float4 x[kQ];
                    if (sl == w.slot) {
#pragma unroll
                        for (int j = 0; j < kQ; ++j) x[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < kQ; ++j) x[j] = __ldcg(src + sl * sq + j * 128);
                    }
#pragma unroll
                    for (int j = 0; j < kQ; ++j) {
                        acc[j].x += x[j].x;
                        acc[j].y += x[j].y;
                        acc[j].z += x[j].z;
                        acc[j].w += x[j].w;
                    }
                }
#pragma unroll
                for (int j = 0; j < kQ; ++j) {
                    v[4 * j] = acc[j].x;
                    v[4 * j + 1] = acc[j].y;
                    v[4 * j + 2] = acc[j].z;
                    v[4 * j + 3] = acc[j].w;
                }
                sink(w, c);
            }
            release_tmem();
            named_bar_sync(kEpiBarrier, kEpiThreads);  // this slot has read every partial it needs
            if (threadIdx.x == 64) {
                if (atomicAdd(counter, 1u) == (uint32_t)(w.nslots - 1)) {
                    // every slot is done reading: reset for the next launch
                    for (int32_t sl = 0; sl < w.nslots; ++sl) flags[sl] = 0u;
                    __threadfence();
                    *counter = 0u;
                }
            }
            ++local;
            continue;
        }
        named_bar_sync(kEpiBarrier, kEpiThreads);  // last_flag of the previous item is consumed
        if (threadIdx.x == 64) {
            const uint32_t prev = atomicAdd(counter, 1u);
            *last_flag = (prev == (uint32_t)(w.nslots - 1)) ? 1 : 0;
        }
        named_bar_sync(kEpiBarrier, kEpiThreads);
        const bool last = *last_flag != 0;
        const float4* const base = reinterpret_cast<const float4*>(ws + split_id * pl.max_slots * tile_elems);
        const int64_t slot_q = tile_elems / 4;
        if (!last) {
            float4* part = const_cast<float4*>(base) + w.slot * slot_q;
            for (uint32_t c = 0; c < ncols; c += kChunk) {
                __syncwarp();
                tmem_load_chunk<kMode>(taddr + c, v);
#pragma unroll
                for (int j = 0; j < kQ; ++j)
                    __stcg(part + (int64_t)(c / 4 + j) * 128 + lane_row,
                           make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
            }
            release_tmem();
            __threadfence();  // the partial is visible before the flag
            named_bar_sync(kEpiBarrier, kEpiThreads);
            if (threadIdx.x == 64) atomicExch(flags + w.slot, 1u);
            ++local;
            continue;
        }
        // last arriver: every other slot has taken its ticket; wait (bounded)
        // until each has published its partial
        bool ready = true;
        if (threadIdx.x == 64) {
            volatile uint32_t* vf = flags;
            volatile int32_t* abort_flag = &ctrl->abort_flag;
            const uint64_t t0 = globaltimer_ns();
            for (int32_t sl = 0; sl < w.nslots && ready; ++sl) {
                if (sl == w.slot) continue;
                while (vf[sl] == 0u) {
                    if (*abort_flag || globaltimer_ns() - t0 > p.timeout_ns) {
                        *abort_flag = 1;
                        atomicCAS(p.err, 0, kErrEpilogue);
                        ready = false;
                        break;
                    }
                }
            }
        }
        ready = named_bar_and(kEpiBarrier, kEpiThreads, ready);
        if (!ready) {
            release_tmem();
            break;
        }
        __threadfence();
        // When this is the CTA's final item its ring is idle: fetch the
        // other slots' partials into it with bulk copies (one per 64-column
        // unit and slot, all in flight at once) instead of latency-bound
        // loads from every thread.  The ring must hold them all.
        const uint32_t part_bytes = ncols * 512u;  // one slot: 128 lanes x ncols fp32
        bool fast;
        {
            WorkIter peek = wi;
            WorkItem nx;
            fast = !peek.next(pl, nx) && (uint32_t)(w.nslots - 1) * part_bytes <= staging - stages;
        }
        if (fast && threadIdx.x == 64) {
            fence_proxy_async_global();
            ctrl->fix_armed = (int32_t)((ncols + 63u) / 64u);
            for (uint32_t u = 0; u * 64u < ncols; ++u) {
                const uint32_t ub = (ncols - u * 64u < 64u ? ncols - u * 64u : 64u) * 512u;
                mbar_arrive_expect_tx(smem_u32(&ctrl->fix_bar[u]), (uint32_t)(w.nslots - 1) * ub);
                uint32_t q = 0;
                for (int32_t sl = 0; sl < w.nslots; ++sl) {
                    if (sl == w.slot) continue;
                    bulk_load(stages + q * part_bytes + u * 64u * 512u,
                              reinterpret_cast<const char*>(base + sl * slot_q) + u * 64u * 512u, ub,
                              smem_u32(&ctrl->fix_bar[u]));
                    ++q;
                }
            }
        }
        for (uint32_t c = 0; c < ncols; c += kChunk) {
            if (fast && c % 64u == 0) {
                bool ok = wait_phase(smem_u32(&ctrl->fix_bar[c / 64u]), 0, ctrl, p, kErrEpilogue);
                if (!named_bar_and(kEpiBarrier, kEpiThreads, ok)) break;
            }
            __syncwarp();
            tmem_load_chunk<kMode>(taddr + c, v);  // own share
            float4 acc[kQ];
#pragma unroll
            for (int j = 0; j < kQ; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            const float4* src = base + (int64_t)(c / 4) * 128 + lane_row;
            uint32_t q = 0;
            for (int32_t sl = 0; sl < w.nslots; ++sl) {
                float4 x[kQ];
                if (sl == w.slot) {
#pragma unroll
                    for (int j = 0; j < kQ; ++j) x[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                } else if (fast) {
                    const uint32_t srow = stages + q * part_bytes + (((c / 4) * 128u + lane_row) << 4);
#pragma unroll
                    for (int j = 0; j < kQ; ++j) x[j] = ld_shared_f4(srow + ((uint32_t)j * 128u << 4));
                    ++q;
                } else {
#pragma unroll
                    for (int j = 0; j < kQ; ++j) x[j] = __ldcg(src + sl * slot_q + j * 128);
                }
#pragma unroll
                for (int j = 0; j < kQ; ++j) {
                    acc[j].x += x[j].x;
                    acc[j].y += x[j].y;
                    acc[j].z += x[j].z;
                    acc[j].w += x[j].w;
                }
            }
#pragma unroll
            for (int j = 0; j < kQ; ++j) {
                v[4 * j] = acc[j].x;
                v[4 * j + 1] = acc[j].y;
                v[4 * j + 2] = acc[j].z;
                v[4 * j + 3] = acc[j].w;
            }
            sink(w, c);
        }
        release_tmem();
        named_bar_sync(kEpiBarrier, kEpiThreads);
        if (threadIdx.x == 64) {
            // every slot of this tile has arrived and published: reset the
            // counter and flags for the next launch
            for (int32_t sl = 0; sl < w.nslots; ++sl) flags[sl] = 0u;
            *counter = 0u;
        }
        ++local;
    }
    // every TMA store of C issued by this warp has completed
    if (!T::kSwap && lane == 0) bulk_wait_group_all();
    __syncwarp();
}

// ------------------------------------------------------------------ kernel

// Bounded wait (100 us in all) for the copies an aborting CTA issued: the
// full barrier of every ring stage armed in the current lap (parity
// ring_ph) and, once the ring has wrapped, in the previous one (the other
// parity), and the fixup's bulk-copy barriers.
__device__ __forceinline__ void drain_copies(Ctrl* ctrl, uint32_t S) {
    const uint64_t t0 = globaltimer_ns();
    const uint64_t limit = 100000ull;
    const uint32_t ring_s = (uint32_t)ctrl->ring_s, ring_ph = (uint32_t)ctrl->ring_ph;
    const bool lap = ctrl->ring_lap != 0;
    for (uint32_t i = 0; i < S; ++i) {
        if (i >= ring_s && !lap) continue;  // never armed
        const uint32_t parity = i < ring_s ? ring_ph : ring_ph ^ 1u;
        while (!mbar_try_wait(smem_u32(&ctrl->full[i]), parity))
            if (globaltimer_ns() - t0 > limit) return;
    }
    for (int32_t u = 0; u < ctrl->fix_armed; ++u)
        while (!mbar_try_wait(smem_u32(&ctrl->fix_bar[u]), 0))
            if (globaltimer_ns() - t0 > limit) return;
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_relu_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmC,
                     const __grid_constant__ CUtensorMap tmA2,
                     const __grid_constant__ KParams p) {
    using T = ModeTraits<kMode>;
    extern __shared__ __align__(1024) uint8_t smem[];
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem);
    const uint32_t base = smem_u32(smem);
    const uint32_t stages = (base + (uint32_t)sizeof(Ctrl) + 1023u) & ~1023u;
    const gemm_relu_plan_t& pl = p.plan;
    // MMA A operand per stage: 128 rows of 64 k; swapped, the tile's two
    // 64-wide chunks of B columns (kBK k-rows each)
    const uint32_t a_bytes = T::kSwap ? 2u * T::kBK * kSwizzleRow : T::kSub * kOperandA;
    const uint32_t b_bytes = (T::kPair ? T::kBChunks * T::kBK * kSwizzleRow
                                       : ((uint32_t)pl.mma_n * T::kBK * 2 + 1023u) & ~1023u);
    const uint32_t stride = a_bytes + b_bytes;
    const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // CTA pairs (one MMA for two CTAs) and cluster split-K run in clusters
    const bool clustered = T::kPair || cluster_split(pl);
    const uint32_t rank = clustered ? cluster_ctarank() : 0u;
    const int32_t worker = clustered ? (int32_t)(blockIdx.x / (uint32_t)pl.cluster) : (int32_t)blockIdx.x;
    // The plan must be one this kernel shape was built for (the host never
    // builds another): swapped tiles 128 columns wide, tiled and paired
    // tiles of the kernel's width.  Every CTA decides alike, before any
    // barrier.
    if ((T::kSwap && pl.tile_n != 128) || (!T::kSwap && (uint32_t)pl.mma_n != T::kBN)) {
        if (threadIdx.x == 0) atomicCAS(p.err, 0, kErrConfig);
        return;
    }

    // Set-up: warp 2 (an epilogue warp, idle until the first accumulator)
    // initialises the barriers, warp 1 allocates tensor memory, and the
    // producer warps meanwhile build their state (below).
    if (warp == 2 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if constexpr (!T::kSwap) tma_prefetch_desc(&tmC);
        for (int s = 0; s < pl.num_stages; ++s) {
            mbar_init(smem_u32(&ctrl->full[s]), 1);
            mbar_init(smem_u32(&ctrl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&ctrl->tmem_full[b]), 1);
            // a pair's leader also counts the peer's epilogue warps
            mbar_init(smem_u32(&ctrl->tmem_empty[b]), (T::kPair ? 2u : 1u) * (kEpiThreads / 32));
        }
        mbar_init(smem_u32(&ctrl->final_bar), 1);
        for (int u = 0; u < 4; ++u) mbar_init(smem_u32(&ctrl->fix_bar[u]), 1);
        // cluster split-K: swapped, the peers push their partials into this
        // CTA's buffer (one local arrival, completed by their bytes); tiled,
        // each peer arrives once its partial sits in its own ring
        // (tiled, cluster of 2 and >= 128 columns: the symmetric exchange --
        // one local arrival, completed by the peer's pushed bytes)
        const bool sym_exch = !T::kSwap && cluster_split(pl) && pl.cluster == 2 && pl.mma_n >= 128;
        mbar_init(smem_u32(&ctrl->exch_bar),
                  (!T::kSwap && pl.cluster > 1 && !sym_exch) ? (uint32_t)pl.cluster - 1u : 1u);
        mbar_init(smem_u32(&ctrl->peer_free), 1);
        ctrl->abort_flag = 0;
        ctrl->last_flag = 0;
        ctrl->ring_s = 0;
        ctrl->ring_ph = 0;
        ctrl->ring_lap = 0;
        ctrl->fix_armed = 0;
        fence_mbar_init();

        if (T::kSwap && cluster_split(pl) && rank == 0)
            mbar_arrive_expect_tx(smem_u32(&ctrl->exch_bar),
                                  ((uint32_t)pl.cluster - 1u) * (uint32_t)pl.mma_n * 128u * 4u);
        if (sym_exch) mbar_arrive_expect_tx(smem_u32(&ctrl->exch_bar), (uint32_t)pl.mma_n / 2u * 128u * 4u);
    }
    if (warp == 1) {
        tmem_alloc<T::kCG>(smem_u32(&ctrl->tmem_addr), (uint32_t)pl.tmem_cols);
        tmem_relinquish<T::kCG>();
    }
    // The set-up barrier.  Each warp reaches it once, from its own branch
    // below (a warp-uniform barrier instruction in each).  Everything before
    // it touches only this CTA's (or cluster's) on-chip state, so it may
    // overlap the previous kernel of the stream; nothing after it may read
    // or write global memory before that kernel has completed.  The next
    // kernel may start launching once it is passed: it waits the same way.
    auto setup_barrier = [&]() {
        tc_fence_before();
        if (clustered)
            cluster_sync();  // the peers' barriers are initialised before any remote arrive
        else
            cta_barrier_sync();
        tc_fence_after();
        grid_launch_dependents();
    };
    if (warp == 0 || warp == 6) {
        // Two producer threads, one per operand: a single thread issues one
        // TMA copy per ~250-450 cycles, so two in parallel stream faster.
        // Warp 0 issues A's copies and arms each stage, warp 6 B's.  The
        // whole warp builds the producer's state -- parameters and the first
        // work item, no shared or global memory: ~1500 cycles of integer
        // work -- during the set-up, before the barrier; lane 0 then arms
        // the first stage, waits for the previous kernel and copies.
        Producer<kMode> prod(p, ctrl, stages, stride, a_bytes, &tmA, &tmB, &tmB2, &tmA2, worker, rank,
                             warp == 0 ? 1 : 2);
        prod.first_item();
        setup_barrier();
        if (lane == 0) {
            prod.prime();
            grid_dependency_wait();
            prod.issue(-1);
            prod.save_ring();
        }
        __syncwarp();
    } else {
        setup_barrier();
        if (T::kSwap && warp == 2 && lane == 0) {
            // Small M: warm L2 with the boxes of this CTA's first two rings
            // of k-blocks (B streams from DRAM) while the previous kernel
            // finishes; an idle epilogue warp issues the prefetches (see
            // Producer::prefetch).  (The tiled kernels measured faster
            // without: their prefetches hold up the first copies in the TMA
            // unit.)
            Producer<kMode> pre(p, ctrl, stages, stride, a_bytes, &tmA, &tmB, &tmB2, &tmA2, worker, rank);
            pre.prefetch(2 * pl.num_stages);
        }
        // (the MMA thread waits inside its role, after its set-up)
        if (warp != 1) grid_dependency_wait();
    }

    const uint32_t tmem_base = ctrl->tmem_addr;
    if (warp == 1) {
        if (lane == 0 && (!T::kPair || rank == 0)) {  // one thread (of a pair's leader) issues the MMAs
            mma_role<kMode>(p, ctrl, stages, stride, a_bytes, tmem_base, worker, rank);
            // no MMA may still be running when tensor memory is released
            mma_commit<T::kCG>(smem_u32(&ctrl->final_bar), 0x1);
            if (!wait_phase_for(smem_u32(&ctrl->final_bar), 0, p.timeout_ns)) atomicCAS(p.err, 0, kErrFinal);
        }
        __syncwarp();
    } else if (warp >= 2 && warp <= 5) {
        // C staging for the TMA stores sits after the ring (tiled paths)
        const uint32_t staging = stages + (uint32_t)pl.num_stages * stride;
        epilogue_role<kMode>(p, ctrl, tmem_base, worker, rank, &tmC, stages, staging);
    }

    // Every role has returned, so the abort flag is final.  An aborting CTA
    // waits (bounded) until the copies it issued into its ring stages and
    // fixup buffers have landed -- each armed stage's full barrier completes
    // its phase when its bytes arrive -- before its shared memory is
    // released; a stage armed for bytes that were never issued ends the
    // wait at the limit.
    __syncthreads();
    if (threadIdx.x == 0 && *(volatile int32_t*)&ctrl->abort_flag) drain_copies(ctrl, (uint32_t)pl.num_stages);
    tc_fence_before();
    if (clustered)
        cluster_sync_relaxed();  // a peer's shared memory may be read (MMA, DSMEM) until here
    else
        __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<T::kCG>(tmem_base, (uint32_t)pl.tmem_cols);
    }
    if (p.pack_sync && threadIdx.x == 0) {
        // every role of this CTA is done (its producer is past its wait for
        // the copy of A): the last CTA to get here resets both words for
        // the next launch
        if (atomicAdd(p.pack_sync + 1, 1u) == gridDim.x - 1) {
            p.pack_sync[0] = 0u;
            p.pack_sync[1] = 0u;
        }
    }
}

}  // namespace gr
