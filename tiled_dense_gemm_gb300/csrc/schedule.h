// Work decomposition shared by the host planner and the persistent kernel.
//
// The output C is cut into tiles (tile_m x tile_n).  Each tile is a
// reduction over num_kb k-blocks of 64.  A persistent grid of `grid` CTAs
// walks:
//   1. data-parallel tiles [0, dp_tiles): CTA c takes tiles c, c+grid, ...,
//      each over its whole K range;
//   2. stream-K tiles [dp_tiles, num_tiles): their (tile, k-block) units are
//      laid end to end and cut into `grid` contiguous runs of q or q+1 units
//      (the first r CTAs take q+1).  A run may start or end inside a tile;
//      the CTAs sharing a tile each own one "slot" of it, numbered in K
//      order, and the last one to finish adds the slots' fp32 partial tiles
//      in slot order (so the result does not depend on which CTA is last);
//      or, with `splits` > 1, split tiles cut into `splits` equal K ranges,
//      one item each.  When every worker has at most one such item and the
//      columns divide into whole epilogue chunks per slot, the slots of a
//      tile share its reduction (concurrent_split): the split tiles are
//      then tiles [0, sk_tiles), the whole ones [sk_tiles, num_tiles), and
//      each worker runs its split item first.
// This generalises the split-KV decode idea of the TileLang MLA example
// ("Writing High-Performance Kernels in TileLang", MLA section: spread a
// long reduction over idle SMs and combine the pieces) to the K dimension
// of a GEMM.
#pragma once

#include <stdint.h>

#include "gemm_relu.h"

#if defined(__CUDACC__)
#define GR_HD __host__ __device__ __forceinline__
#else
#define GR_HD inline
#endif

namespace gr {

constexpr int kBlockK = 64;  // k-block: 64 fp16 = one 128-byte swizzle row

// Rasterisation: tiles are numbered so that a group of `group_m` tile rows
// is walked column by column; CTAs running at the same time then share A
// row-panels and B column-panels in L2.
GR_HD void tile_coords(const gemm_relu_plan_t& p, int32_t t, int32_t& tm, int32_t& tn) {
    const int32_t per_group = p.group_m * p.tiles_n;
    const int32_t g = t / per_group;
    const int32_t first_m = g * p.group_m;
    const int32_t rows = (p.tiles_m - first_m) < p.group_m ? (p.tiles_m - first_m) : p.group_m;
    const int32_t r = t - g * per_group;
    tm = first_m + r % rows;
    tn = r / rows;
}

// First stream-K unit of CTA c (c may equal grid: one past the end).
GR_HD int64_t sk_begin(const gemm_relu_plan_t& p, int32_t c) {
    return (int64_t)c * p.sk_q + (c < p.sk_r ? c : p.sk_r);
}

// CTA that owns stream-K unit x.
GR_HD int32_t sk_owner(const gemm_relu_plan_t& p, int64_t x) {
    const int64_t big = (int64_t)p.sk_r * (p.sk_q + 1);
    if (x < big) return (int32_t)(x / (p.sk_q + 1));
    return (int32_t)(p.sk_r + (x - big) / p.sk_q);
}

// Split tiles whose slots all run at once (at most one split item per
// worker) and whose columns divide into whole epilogue chunks per slot:
// their slots share the reduction (each sums and stores 1/splits of the
// columns) instead of leaving it all to the last arriver.
GR_HD bool concurrent_split(const gemm_relu_plan_t& p) {
    const int32_t chunk = (p.path == 3) ? 16 : 64;  // epilogue chunk (columns)
    return p.splits > 1 && (int64_t)p.sk_tiles * p.splits <= p.grid && p.mma_n % (p.splits * chunk) == 0;
}

struct WorkItem {
    int32_t tile;      // linear tile id
    int32_t tm, tn;    // tile row / column
    int32_t kb0, kb1;  // k-blocks [kb0, kb1)
    int32_t slot;      // share index within a split tile (0 when whole)
    int32_t nslots;    // CTAs sharing this tile (1 when whole)
    int32_t sk_index;  // stream-K tile index (tile - dp_tiles), -1 when data-parallel
};

// Cluster split-K: a one-CTA kernel shape (path 2 or 3) launched in
// clusters of `cluster` CTAs, each cluster one worker; CTA rank r of the
// cluster computes K range r of every tile of the worker, and the CTAs
// combine their accumulators through distributed shared memory.
GR_HD bool cluster_split(const gemm_relu_plan_t& p) {
    return (p.path == 2 || p.path == 3) && p.cluster > 1;
}

// Integer division is a software routine on the GPU (a 64-bit one several
// hundred cycles of dependent instructions), and these run before a CTA's
// first copy: every quotient that fits in 32 bits is taken in 32 bits
// (split items: u < sk_tiles * splits; k-block bounds: slot * num_kb with
// slot <= 16 and num_kb < 2^25).
struct WorkIter {
    int32_t cta;
    int32_t rank;  // CTA rank in the cluster (cluster split-K); 0 otherwise
    int32_t dp_i, dp_n;
    int64_t u, u1;  // stream-K units, or split items when p.splits > 1
    bool cs;        // concurrent_split(p), taken once

    GR_HD void init(const gemm_relu_plan_t& p, int32_t c, int32_t r = 0) {
        cta = c;
        cs = concurrent_split(p);
        rank = cluster_split(p) ? r : 0;
        dp_i = 0;
        dp_n = (c < p.dp_tiles) ? (p.dp_tiles - 1 - c) / p.grid + 1 : 0;
        if (p.sk_tiles > 0 && p.splits > 1) {
            u = c;
            u1 = (int64_t)p.sk_tiles * p.splits;
        } else if (p.sk_tiles > 0) {
            u = sk_begin(p, c);
            u1 = sk_begin(p, c + 1);
        } else {
            u = u1 = 0;
        }
    }

    GR_HD bool next_dp(const gemm_relu_plan_t& p, WorkItem& w) {
        if (dp_i >= dp_n) return false;
        // (with the split items first, the split tiles also come first in
        // the raster order, so that the first round's tiles are neighbours)
        w.tile = (cs ? p.sk_tiles : 0) + cta + dp_i * p.grid;
        w.sk_index = -1;
        if (cluster_split(p)) {
            w.kb0 = rank * p.num_kb / p.cluster;
            w.kb1 = (rank + 1) * p.num_kb / p.cluster;
            w.slot = rank;
            w.nslots = p.cluster;
        } else {
            w.kb0 = 0;
            w.kb1 = p.num_kb;
            w.slot = 0;
            w.nslots = 1;
        }
        ++dp_i;
        tile_coords(p, w.tile, w.tm, w.tn);
        return true;
    }

    GR_HD bool next_split(const gemm_relu_plan_t& p, WorkItem& w) {
        if (u >= u1) return false;
        // split item: tile fastest, so workers running together read the
        // same K range of neighbouring tiles
        const int32_t sp = (int32_t)u / p.sk_tiles;
        const int32_t t = (int32_t)u - sp * p.sk_tiles;
        w.sk_index = t;
        w.tile = cs ? t : p.dp_tiles + t;
        w.kb0 = sp * p.num_kb / p.splits;
        w.kb1 = (sp + 1) * p.num_kb / p.splits;
        w.slot = sp;
        w.nslots = p.splits;
        u += p.grid;
        tile_coords(p, w.tile, w.tm, w.tn);
        return true;
    }

    // Items in the order a worker runs them: data-parallel tiles, then its
    // split or stream-K share -- except when the slots of each split tile
    // share its reduction (concurrent_split): then the split item comes
    // first, so that all slots of a tile run together at the start and the
    // reduction overlaps the worker's next tile (double-buffered TMEM)
    // instead of adding to the end of the launch.
    GR_HD bool next(const gemm_relu_plan_t& p, WorkItem& w) {
        if (cs) {
            if (next_split(p, w)) return true;
            return next_dp(p, w);
        }
        if (next_dp(p, w)) return true;
        if (p.splits > 1) return next_split(p, w);
        if (u < u1) {
            const int64_t t = u / p.num_kb;
            const int32_t kb0 = (int32_t)(u - t * p.num_kb);
            const int64_t left = u1 - u;
            const int32_t kb1 = (int64_t)(p.num_kb - kb0) < left ? p.num_kb : kb0 + (int32_t)left;
            const int32_t first = sk_owner(p, t * p.num_kb);
            const int32_t last = sk_owner(p, (t + 1) * p.num_kb - 1);
            w.sk_index = (int32_t)t;
            w.tile = p.dp_tiles + (int32_t)t;
            w.kb0 = kb0;
            w.kb1 = kb1;
            w.slot = cta - first;
            w.nslots = last - first + 1;
            u += kb1 - kb0;
            tile_coords(p, w.tile, w.tm, w.tn);
            return true;
        }
        return false;
    }
};

// Planner with the runtime's limits: at most `max_pairs` co-resident CTA
// pairs (<= 0: num_sms / 2).  `force` is the GEMM_RELU_FORCE_PATH value or
// nullptr.  Defined in plan.cpp.
int plan_problem(int64_t M, int64_t N, int64_t K, int num_sms, int max_pairs, const char* force,
                 gemm_relu_plan_t* plan);

// Whether A is first copied to a row pitch that is a multiple of 128 bytes
// (the plan's pack_a, decided for B stored (K, N), refined here for B
// stored (N, K)); `force` ":pk" / ":npk" forces it on (when K % 64 != 0) or
// off.  Defined in plan.cpp.
bool pack_a_pays(const gemm_relu_plan_t& plan, int64_t M, int64_t N, int64_t K, bool b_nk, const char* force);

// The TMA boxes of one ring stage's copies under `plan` (3-D where the
// shapes allow, unless `force` holds ":no3d").  Defined in plan.cpp.
int plan_boxes(const gemm_relu_plan_t& plan, int64_t M, int64_t N, int64_t K, bool b_nk, const char* force,
               gemm_relu_boxes_t* boxes);

}  // namespace gr
