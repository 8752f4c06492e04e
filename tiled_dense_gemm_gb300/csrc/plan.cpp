// Host planner: picks tile shape, operand roles and the data-parallel /
// stream-K split for one problem size, by a small cost model evaluated
// over the exact work lists the kernel will walk.  Pure host code.
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "gemm_relu.h"
#include "schedule.h"

namespace gr {

// Shared-memory layout constants (must match the kernel).
constexpr int32_t kCtrlBytes = 1024;        // barriers + flags
constexpr int32_t kAlignSlack = 1024;       // dynamic smem rounded up to 1 KiB
constexpr int32_t kSmemLimit = 227 * 1024;  // opt-in shared memory per CTA
constexpr int32_t kStagingBytes = 32 * 1024;  // C staging for TMA stores (tiled paths)
constexpr int32_t kMaxStages = 16;
constexpr int32_t kSwizzleRowBytes = 128;   // one swizzled shared-memory row

// Cost model in microseconds, calibrated against GB300 measurements
// (sm clock ~1.9-2.1 GHz): per-k-block mainloop time of each kernel shape,
// the exposed part of a finished tile's store, and the split-K costs (fp32
// partial write by a non-last CTA, and the last CTA's reduction per slot).
struct Costs {
    double kb;               // one k-block through the mainloop
    double fill;             // launch to first data: set-up and the first TMA round trip
    double tile_store;       // storing one finished tile (TMEM -> C)
    double partial;          // writing one fp32 partial tile
    double reduce_per_slot;  // the last CTA's work per slot of a split tile
    double exchange;         // cluster split-K: reading the peer's fp32 tile over DSMEM
};

static Costs costs_for(int32_t path, int32_t mma_n, int32_t stage_bytes) {
    Costs c;
    c.fill = 3.0;
    // measured: ~1 us of handshake + the peer's 128 x mma_n fp32 tile at
    // ~32 B/clk over DSMEM, plus the cluster teardown
    c.exchange = 1.0 + 128.0 * mma_n * 4.0 / 32000.0;
    if (path == 4) {  // CTA pair, 256 x 256 (each CTA 128 x 256)
        c.kb = 0.29;
        c.tile_store = 2.5;
        c.partial = 3.0;           // measured: ~3 us to publish a 128 KiB partial
        c.reduce_per_slot = 3.0;
    } else if (path == 2 && mma_n >= 256) {
        c.kb = 0.37;
        c.tile_store = 2.5;
        c.partial = 6.0;
        c.reduce_per_slot = 4.0;
    } else if (path == 2 && mma_n <= 64) {  // 128 x 64
        c.kb = 0.20;
        c.tile_store = 0.7;
        c.partial = 1.5;
        c.reduce_per_slot = 1.0;
    } else if (path == 2) {
        c.kb = 0.30;
        c.tile_store = 1.3;
        c.partial = 3.0;
        c.reduce_per_slot = 2.0;
    }
    // the figures above are per 64 k-rows; stages of 128 k-rows cost twice
    if (path == 2 && mma_n < 256) c.kb *= 2.0;
    if (path == 3) {
        // swapped operands, streaming B: ~0.4 us per 18 KiB stage per SM
        c.kb = 0.40 * stage_bytes / 18432.0;
        c.tile_store = 0.5;
        c.partial = 1.0;
        c.reduce_per_slot = 1.5;
    }
    return c;
}

// Makespan estimate of a filled-in plan: the slowest CTA's mainloop time
// plus its exposed epilogue work.  A finished tile's store mostly overlaps
// the next tile's mainloop (double-buffered accumulator), so only a quarter
// of it is counted, except for the CTA's last tile.  For a split tile the
// slot-0 owner reaches its share last (it is the end of its run), so it is
// charged the fixup.
static double estimate(const gemm_relu_plan_t& p, const Costs& c) {
    double worst = 0.0;
    for (int32_t cta = 0; cta < p.grid; ++cta) {
        WorkIter wi;
        wi.init(p, cta);
        const int32_t dp_n = wi.dp_n;
        const bool shared = concurrent_split(p);
        double t = c.fill + (double)dp_n * ((double)p.num_kb * c.kb + 0.25 * c.tile_store);
        wi.dp_i = dp_n;  // data-parallel items are costed above
        bool any = dp_n > 0;
        WorkItem w;
        while (wi.next(p, w)) {
            any = true;
            t += (double)(w.kb1 - w.kb0) * c.kb;
            if (w.nslots == 1)
                t += 0.25 * c.tile_store;
            else if (shared)  // publish, read and store (S-1)/S, (S-1)/S and 1/S of the tile; the
                              // split item runs first, so this overlaps the worker's next tile
                              // when that tile's mainloop is long enough (measured: K = 2048
                              // gains, K = 1024 loses)
                t += (dp_n > 0 && (double)p.num_kb * c.kb >= 8.0 ? 0.25 : 1.0) *
                     ((c.partial + c.reduce_per_slot) * (w.nslots - 1) / w.nslots + c.tile_store / w.nslots);
            else
                t += c.partial + (w.slot == 0 ? w.nslots * c.reduce_per_slot + c.tile_store : 0.0);
        }
        if (!any) continue;
        t += 0.75 * c.tile_store;
        if (t > worst) worst = t;
    }
    return worst;
}

static int32_t compute_max_slots(const gemm_relu_plan_t& p) {
    int32_t best = 1;
    for (int32_t t = 0; t < p.sk_tiles; ++t) {
        const int32_t first = sk_owner(p, (int64_t)t * p.num_kb);
        const int32_t last = sk_owner(p, (int64_t)(t + 1) * p.num_kb - 1);
        if (last - first + 1 > best) best = last - first + 1;
    }
    return best;
}

static void finish_split(gemm_relu_plan_t& p, int32_t grid, int32_t dp, int32_t sk,
                         int32_t splits = 1) {
    p.grid = grid;
    p.dp_tiles = dp;
    p.sk_tiles = sk;
    p.splits = (sk > 0 && splits > 1) ? splits : 1;
    if (sk > 0 && p.splits > 1) {
        p.sk_q = p.sk_r = 0;
        p.max_slots = p.splits;
    } else if (sk > 0) {
        const int64_t units = (int64_t)sk * p.num_kb;
        p.sk_q = (int32_t)(units / grid);
        p.sk_r = (int32_t)(units % grid);
        p.max_slots = compute_max_slots(p);
    } else {
        p.sk_q = p.sk_r = 0;
        p.max_slots = 1;
    }
    // one fp32 partial of 128 rows x mma_n columns per (tile, CTA of the worker, slot)
    p.workspace_bytes = (int64_t)sk * p.cluster * p.max_slots * 128 * p.mma_n * 4;
    p.counter_count = (int64_t)sk * p.cluster;
}

// Fill the shape-dependent fields for one kernel shape: path 2 with
// mma_n = 64, 128 or 256; path 3 (mma_n = M padded to 16, tiles of 128
// columns); path 4 (CTA pairs, mma_n = 256).
static void shape_plan(gemm_relu_plan_t& p, int64_t M, int64_t N, int64_t K, int32_t path, int32_t mma_n) {
    p.path = path;
    p.mma_n = mma_n;
    p.cluster = (path == 4) ? 2 : 1;
    p.mma_m = (path == 4) ? 256 : 128;
    if (path == 2) {
        p.tile_m = 128;
        p.tile_n = mma_n;
    } else if (path == 4) {
        p.tile_m = 256;
        p.tile_n = mma_n;
    } else {
        p.tile_m = mma_n;  // padded M
        p.tile_n = 128;
    }
    p.tiles_m = (int32_t)((M + p.tile_m - 1) / p.tile_m);
    p.tiles_n = (int32_t)((N + p.tile_n - 1) / p.tile_n);
    p.num_tiles = p.tiles_m * p.tiles_n;
    // k-rows per stage: 128, except 256-column tiles (tensor-bound already;
    // 64-row stages keep their ring deeper)
    p.block_k = (mma_n == 256 && path != 3) ? kBlockK : 2 * kBlockK;
    p.num_kb = (int32_t)((K + p.block_k - 1) / p.block_k);
    p.group_m = p.tiles_m < 8 ? p.tiles_m : 8;
    // per CTA: columns of the MMA B operand it loads (half of the tile for
    // a pair; the padded rows of A when swapped)
    const int32_t b_cols = (path == 4) ? mma_n / 2 : mma_n;
    const int32_t b_bytes = b_cols * p.block_k * 2;
    // MMA A operand per stage: 128 rows, or for the swapped kernel the
    // tile's two 64-wide chunks of B columns
    const int32_t a_region = 128 * p.block_k * 2;
    // bytes the TMA copies of one stage deliver
    p.stage_bytes = a_region + b_bytes;
    // B region (1 KiB aligned: the swizzle atoms)
    const int32_t b_region = ((b_bytes + 1023) / 1024) * 1024;
    const int32_t stride = a_region + b_region;
    // tiled paths: C staging for the TMA stores; swapped: the buffer a
    // cluster split-K peer pushes its fp32 partial into (128 x mma_n)
    const int32_t staging = (path == 3) ? 128 * mma_n * 4 : kStagingBytes;
    const int32_t budget = kSmemLimit - kCtrlBytes - kAlignSlack - staging;
    int32_t stages = budget / stride;
    if (stages > kMaxStages) stages = kMaxStages;
    p.num_stages = stages;
    p.smem_bytes = kCtrlBytes + kAlignSlack + stages * stride + staging;
    int32_t cols = 2 * mma_n;
    int32_t alloc = 32;
    while (alloc < cols) alloc *= 2;
    p.tmem_cols = alloc;
}

// Choose the best split for the current shape over at most `workers`
// persistent workers; returns its estimated cost.
static double choose_split(gemm_relu_plan_t& p, int32_t workers, bool dp_only, int32_t force_splits,
                           bool operands_fit_l2, int32_t pairs = 0) {
    // a single tile row reads each B column block once whatever the order
    operands_fit_l2 = operands_fit_l2 || p.tiles_m == 1;
    const Costs c = costs_for(p.path, p.mma_n, p.stage_bytes);
    const int32_t T = p.num_tiles;
    gemm_relu_plan_t best = p;
    double best_cost = -1.0;
    auto consider = [&](int32_t grid, int32_t dp, int32_t sk) {
        if (grid < 1) return;
        if (sk > 0 && (int64_t)sk * p.num_kb < grid) grid = (int32_t)((int64_t)sk * p.num_kb);
        gemm_relu_plan_t q = p;
        finish_split(q, grid, dp, sk);
        double cost = estimate(q, c);
        // small preference for fewer partial tiles at equal cost
        cost += 1e-3 * (double)q.sk_tiles;
        if (best_cost < 0.0 || cost < best_cost) {
            best_cost = cost;
            best = q;
        }
    };
    if (force_splits > 1) {
        // every tile cut into force_splits K ranges (at most one per k-block)
        const int32_t sp = force_splits < p.num_kb ? force_splits : p.num_kb;
        const int64_t items = (int64_t)T * sp;
        gemm_relu_plan_t q = p;
        finish_split(q, (int32_t)(items < workers ? items : workers), 0, T, sp);
        p = q;
        return estimate(q, c);
    }
    // plain data-parallel
    consider(T < workers ? T : workers, T, 0);
    // cluster split-K: each tile by a cluster of 2 CTAs, one K half each,
    // combined through distributed shared memory; one wave of clusters
    if (!dp_only && pairs > 0 && p.path != 4 && T <= pairs && p.num_kb >= 8) {
        gemm_relu_plan_t q = p;
        finish_split(q, T, T, 0);
        q.cluster = 2;
        q.max_slots = 2;
        double cost = c.fill + (double)((p.num_kb + 1) / 2) * c.kb + c.tile_store + c.exchange;
        if (best_cost < 0.0 || cost < best_cost) {
            best_cost = cost;
            best = q;
        }
    }
    if (!dp_only) {
        if (T >= workers) {
            const int32_t full = T / workers;
            if (T % workers != 0) consider(workers, (full - 1) * workers, T - (full - 1) * workers);
            // full waves data-parallel, the leftover tiles cut into S equal
            // K ranges spread over the workers (a short split-K tail wave)
            if (T % workers != 0)
                for (int32_t sp = 2; sp <= 4 && sp <= p.num_kb; ++sp) {
                    gemm_relu_plan_t q = p;
                    finish_split(q, workers, full * workers, T % workers, sp);
                    // (+0.5 us: the fixup's cost varies; take the split tail
                    // only for a clear gain)
                    const double cost = estimate(q, c) + 0.5 + 1e-3 * (double)q.sk_tiles;
                    if (best_cost < 0.0 || cost < best_cost) {
                        best_cost = cost;
                        best = q;
                    }
                }
        } else if (p.num_kb > 1 && operands_fit_l2) {
            // fewer tiles than workers: split every tile along K over more
            // workers.  Only when A and B stay in L2: the workers sharing a
            // B column block then reach its rows at different times, and
            // without L2 each would fetch it from DRAM again.
            for (int32_t g = T + 1; g <= workers; ++g) consider(g, 0, T);
        }
    }
    p = best;
    return best_cost;
}

static bool starts_with(const char* s, const char* prefix) {
    while (*prefix)
        if (*s++ != *prefix++) return false;
    return true;
}

static bool contains(const char* s, const char* what) {
    for (; *s; ++s)
        if (starts_with(s, what)) return true;
    return false;
}

int plan_problem(int64_t M, int64_t N, int64_t K, int num_sms, int max_pairs, const char* force,
                 gemm_relu_plan_t* plan) {
    if (!plan || M < 0 || N < 0 || K < 0 || M > GEMM_RELU_MAX_DIM || N > GEMM_RELU_MAX_DIM ||
        K > GEMM_RELU_MAX_DIM || num_sms < 1)
        return GEMM_ERR_INVALID_ARG;
    memset(plan, 0, sizeof(*plan));
    if (M == 0 || N == 0) {
        plan->path = 0;
        return GEMM_OK;
    }
    if (K == 0) {
        plan->path = 1;
        return GEMM_OK;
    }
    // tile and k-block counts must fit 32-bit work indices
    const int64_t kb = (K + kBlockK - 1) / kBlockK;
    const int64_t tiles_small = ((M + 127) / 128) * ((N + 127) / 128);
    if (tiles_small > (int64_t)1 << 30 || kb > (int64_t)1 << 30) return GEMM_ERR_INVALID_ARG;

    const char* f = force ? force : "";
    const bool dp_only = contains(f, ":dp");
    const bool force_csk = contains(f, ":c2");
    const bool force_sk = contains(f, ":sk");
    int32_t force_tail = 0;  // ":tS": full waves data-parallel, leftover tiles split S ways
    for (const char* q = f; *q; ++q)
        if (q[0] == ':' && q[1] == 't' && q[2] >= '0' && q[2] <= '9') force_tail = q[2] - '0';
    int32_t force_splits = 0;
    for (const char* q = f; *q; ++q)
        if (q[0] == ':' && q[1] == 's' && q[2] >= '0' && q[2] <= '9') {
            force_splits = 0;
            for (const char* d = q + 2; *d >= '0' && *d <= '9'; ++d) force_splits = force_splits * 10 + (*d - '0');
        }
    // co-resident 2-CTA clusters (CTA pairs, cluster split-K); < 0: none
    int32_t pairs = (max_pairs > 0 && max_pairs < num_sms / 2) ? max_pairs : num_sms / 2;
    if (max_pairs < 0) pairs = 0;

    // A + B small enough to stay resident in the 126 MiB L2 next to C
    const bool operands_fit_l2 = 2.0 * ((double)M * K + (double)K * N) <= 48.0 * 1024 * 1024;
    // small M: the swapped-operand kernel (MMA N = padded M) for M <= 32;
    // for 32 < M <= 64 only where it splits K without stream-K (below);
    // else, and above, the 128 x 128 tiled kernel measured faster
    bool want_swap = M <= 64, want_t256 = M > 128, want_t128 = M > 32, want_pair = M > 128 && pairs > 0;
    bool want_t64 = want_t128;
    const bool swap_only = M <= 32 || starts_with(f, "swap");
    if (starts_with(f, "swap") && M <= 128) {
        want_t256 = want_t128 = want_pair = want_t64 = false;
        want_swap = true;
    } else if (starts_with(f, "tiled256")) {
        want_swap = want_t128 = want_pair = want_t64 = false;
        want_t256 = true;
    } else if (starts_with(f, "tiled64")) {
        want_swap = want_t256 = want_t128 = want_pair = false;
        want_t64 = true;
    } else if (starts_with(f, "tiled128")) {
        want_swap = want_t256 = want_pair = want_t64 = false;
        want_t128 = true;
    } else if (starts_with(f, "pair") && pairs > 0) {
        want_swap = want_t256 = want_t128 = want_t64 = false;
        want_pair = true;
    }

    double best_cost = -1.0;
    auto take = [&](int32_t path, int32_t mma_n, int32_t workers) {
        gemm_relu_plan_t q;
        memset(&q, 0, sizeof(q));
        shape_plan(q, M, N, K, path, mma_n);
        double cost = choose_split(q, workers, dp_only, force_splits, operands_fit_l2, pairs);
        if (force_tail > 1 && q.num_tiles >= workers && q.num_tiles % workers != 0) {
            q.cluster = (path == 4) ? 2 : 1;
            const int32_t sp = force_tail < q.num_kb ? force_tail : q.num_kb;
            finish_split(q, workers, (q.num_tiles / workers) * workers, q.num_tiles % workers, sp);
            cost = 0.0;
        }
        if (force_sk) {
            // every tile stream-K over all workers
            const int64_t units = (int64_t)q.num_tiles * q.num_kb;
            q.cluster = (path == 4) ? 2 : 1;  // no cluster split-K
            finish_split(q, (int32_t)(units < workers ? units : workers), 0, q.num_tiles);
            cost = 0.0;
        }
        if (force_csk && pairs > 0 && path != 4 && q.num_tiles <= pairs && q.num_kb >= 2) {
            finish_split(q, q.num_tiles, q.num_tiles, 0);
            q.cluster = 2;
            q.max_slots = 2;
            cost = 0.0;
        }
        if (best_cost < 0.0 || cost < best_cost) {
            best_cost = cost;
            *plan = q;
        }
    };
    if (want_swap) {
        // small M: C^T = B^T A^T, so N runs along the 128-wide MMA M side
        // and M (padded to 16) is the MMA N side.
        const int32_t mpad = (int32_t)((M + 15) / 16) * 16;
        // Streaming B: cut each 128-column tile into S equal K ranges with
        // S = SMs / tiles (tile-fastest item order, so CTAs running together
        // sweep whole rows of B), when that keeps >= 3/4 of the SMs busy;
        // otherwise let the cost model pick data-parallel or stream-K.
        gemm_relu_plan_t q;
        memset(&q, 0, sizeof(q));
        shape_plan(q, M, N, K, 3, mpad);
        // (S <= 4: the last CTA of a tile reads the other S - 1 partials)
        const int32_t sp = q.num_tiles > 0 ? num_sms / q.num_tiles : 0;
        if (force_splits <= 1 && !dp_only && !starts_with(f, "swap") && sp >= 2 && pairs > 0 &&
            q.num_tiles <= pairs && q.num_kb >= 8 && 4 * q.num_tiles * 2 >= 3 * num_sms) {
            // two K halves per tile in one 2-CTA cluster: no global partials
            finish_split(q, q.num_tiles, q.num_tiles, 0);
            q.cluster = 2;
            q.max_slots = 2;
            *plan = q;
            return GEMM_OK;
        }
        // (32 < M <= 64: only with >= 32 k-blocks; shorter K measured
        // faster on the tiled kernel)
        if (force_splits <= 1 && !dp_only && !starts_with(f, "swap") && sp >= 2 && sp <= 4 &&
            sp <= q.num_kb && 4 * q.num_tiles * sp >= 3 * num_sms && (M <= 32 || q.num_kb >= 32)) {
            finish_split(q, q.num_tiles * sp, 0, q.num_tiles, sp);
            q.grid = q.num_tiles * sp;
            *plan = q;
            return GEMM_OK;
        }
        if (swap_only) take(3, mpad, num_sms);
    }
    if (want_pair) take(4, 256, pairs);
    if (want_t256) take(2, 256, num_sms);
    if (want_t128) take(2, 128, num_sms);
    if (want_t64) take(2, 64, num_sms);
    plan->pack_a = pack_a_pays(*plan, M, N, K, false, f) ? 1 : 0;
    return GEMM_OK;
}

// A row pitch that is not a multiple of 128 bytes makes every 128-byte TMA
// box row straddle two L2 lines.  One such operand costs the tiled kernels
// little; both together cost much more (3000 x 5000 x 2056: 56.5 us against
// 48.0 with only A's pitch misaligned and 47.8 with only B's).  So when
// both pitches are misaligned and A is reused by several tile columns,
// A is copied to a 128-byte pitch first (a copy of 2 MK bytes each way).
bool pack_a_pays(const gemm_relu_plan_t& pl, int64_t M, int64_t N, int64_t K, bool b_nk, const char* force) {
    if (pl.path != 2 && pl.path != 4) return false;
    if (K % 64 == 0) return false;  // A's pitch is aligned already
    if (force && strstr(force, ":npk")) return false;
    if (force && strstr(force, ":pk")) return true;
    const bool b_misaligned = b_nk ? true : (N % 64 != 0);
    return b_misaligned && pl.path == 4 && pl.tiles_n >= 4 && 2.0 * (double)M * (double)K >= 4.0 * 1024 * 1024;
}

}  // namespace gr

namespace gr {

int plan_boxes(const gemm_relu_plan_t& pl, int64_t M, int64_t N, int64_t K, bool b_nk, const char* force,
               gemm_relu_boxes_t* o) {
    (void)M;
    if (!o || pl.path < 2) return GEMM_ERR_INVALID_ARG;
    memset(o, 0, sizeof(*o));
    const bool swap = pl.path == 3;
    const bool pair = pl.path == 4;
    const uint32_t sub = (uint32_t)pl.block_k / kBlockK;  // 64-k blocks per stage
    const uint32_t bk = (uint32_t)pl.block_k;
    // One copy per operand and stage where the shapes allow (the TMA unit
    // pays a fixed cost per copy, so fewer, larger boxes stream faster).
    const bool allow3d = !(force && strstr(force, ":no3d"));
    // A: 64 k by 128 rows (the padded rows of A when swapped) per 64-k
    // block; one 3-D copy of a stage's two blocks when K is a multiple of 64
    o->a_box[0] = kBlockK;
    o->a_box[1] = swap ? (uint32_t)pl.tile_m : 128u;
    o->a_box[2] = 1;
    if (allow3d && sub == 2 && K % kBlockK == 0) {
        o->a_3d = 1;
        o->a_box[2] = sub;
    }
    if (!b_nk) {
        // B (K, N): 64-column boxes of a stage's k-rows, the second map's
        // boxes the same
        o->b_box[0] = 64u;
        o->b_box[1] = bk;
        o->b_box[2] = 1;
        o->b2_box[0] = 64u;
        o->b2_box[1] = bk;
        // all of a CTA's whole chunks in one 3-D copy (two or more); with N
        // not a multiple of 64 the view covers the whole chunks, and a CTA
        // reaching the partial one uses the second (2-D) map
        const uint32_t cols = swap ? 128u : (pair ? (uint32_t)pl.mma_n / 2 : (uint32_t)pl.mma_n);
        if (allow3d && N >= 64 && cols % 64 == 0 && cols >= 128) {
            o->b_3d = 1;
            o->b_box[2] = cols / 64;
            o->b_view_inner = (N / 64) * 64;
        }
    } else {
        // B (N, K): 64 k by the rows of N one CTA loads per stage
        const uint32_t rows = swap ? 128u : (pair ? (uint32_t)pl.mma_n / 2 : (uint32_t)pl.mma_n);
        o->b_box[0] = kBlockK;
        o->b_box[1] = rows;
        o->b_box[2] = 1;
        o->b2_box[0] = kBlockK;
        o->b2_box[1] = rows;
        if (allow3d && sub == 2 && K % kBlockK == 0) {
            o->b_3d = 1;
            o->b_box[2] = sub;
        }
    }
    return GEMM_OK;
}

}  // namespace gr

extern "C" int gemm_relu_plan_boxes(const gemm_relu_plan_t* plan, int64_t M, int64_t N, int64_t K, int b_layout,
                                    gemm_relu_boxes_t* boxes) {
    if (!plan || (b_layout != GEMM_B_KN && b_layout != GEMM_B_NK)) return GEMM_ERR_INVALID_ARG;
    return gr::plan_boxes(*plan, M, N, K, b_layout == GEMM_B_NK, getenv("GEMM_RELU_FORCE_PATH"), boxes);
}

extern "C" int gemm_relu_plan(int64_t M, int64_t N, int64_t K, int num_sms,
                              gemm_relu_plan_t* plan) {
    return gr::plan_problem(M, N, K, num_sms, 0, getenv("GEMM_RELU_FORCE_PATH"), plan);
}

extern "C" int gemm_relu_plan_work_item(const gemm_relu_plan_t* plan, int cta, int idx,
                                        int32_t* tile, int32_t* tile_m_idx, int32_t* tile_n_idx,
                                        int32_t* kb_begin, int32_t* kb_end, int32_t* slot,
                                        int32_t* nslots) {
    using namespace gr;
    // `cta` is the worker index, except for cluster split-K plans, where it
    // is the CTA index (worker * cluster + rank)
    if (!plan) return -1;
    const bool csk = cluster_split(*plan);
    const int32_t ctas = csk ? plan->grid * plan->cluster : plan->grid;
    if (cta < 0 || idx < 0 || plan->path < 2 || cta >= ctas) return -1;
    WorkIter wi;
    if (csk)
        wi.init(*plan, cta / plan->cluster, cta % plan->cluster);
    else
        wi.init(*plan, cta);
    WorkItem w = {};
    for (int i = 0; i <= idx; ++i)
        if (!wi.next(*plan, w)) return 0;
    if (tile) *tile = w.tile;
    if (tile_m_idx) *tile_m_idx = w.tm;
    if (tile_n_idx) *tile_n_idx = w.tn;
    if (kb_begin) *kb_begin = w.kb0;
    if (kb_end) *kb_end = w.kb1;
    if (slot) *slot = w.slot;
    if (nslots) *nslots = w.nslots;
    return 1;
}
