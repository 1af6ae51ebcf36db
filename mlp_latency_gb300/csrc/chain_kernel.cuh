// chain_kernel.cuh -- the persistent, warp-specialised tcgen05 kernel that runs a GEMM chain
// with the CTA-pipelining protocol of "CTA-Pipelining: A Latency-Oriented Spatial Scaling
// Method for Multi-GPU Systems" (arXiv 2607.07862).
//
// The kernel runs as clusters of `cs` CTAs (cs = 1, 2, 4 or 8), one CTA per SM.  A cluster
// takes one work item at a time: cs/S tiles of a stage, each tile shared by S CTAs that split
// its reduction dimension (split-K, S = 1 .. cs).  Rank r works on tile r / S, k-slice r % S.
//
// Warp roles (256 threads per CTA):
//   warp 0      TMA producer: for a consumer item, first polls the item's work-queue slot
//               (the injected prologue of section III-A, Fig. 1) to learn its tile; then
//               streams A (activations, K-major) and B (weights) tiles of its k-slice into an
//               NS-deep shared-memory ring.
//   warp 1      MMA issuer: one thread issues tcgen05.mma into a double-buffered TMEM
//               accumulator; warp 1 also owns the TMEM allocation.
//   warp 2      scheduler (rank 0 of each cluster only): takes a ticket per cluster item and
//               broadcasts it (stage, tile or queue slot, k-slice) to every CTA of the cluster
//               through distributed shared memory (the scheduler warp's CGA broadcast of
//               section III-C, Fig. 2b).
//   warp 3      pulls the protocol's counters, queues and dependency tables into L2 at launch;
//               in a Lamport run it then validates every consumer A tile before the MMAs
//               (role_validate).
//   warps 4-7   epilogue: TMEM -> registers -> (split-K reduction) -> (GeLU / residual) ->
//               bf16 -> global, then the injected epilogue: fence, scoreboard releases and
//               queue pushes (section III-A; fence placement per the memory-consistency
//               discussion of section V).
// The scheduler and epilogue warps would otherwise wait at pipeline barriers, so the protocol
// work overlaps the next tile's mainloop: the hiding of section III-C, Fig. 2b.
#pragma once
#include <type_traits>

#include <cuda_bf16.h>

#include "protocol.h"
#include "ptx.cuh"

namespace mlpc {

constexpr int kMaxStages = 4;
constexpr int kMaxCluster = 8;
constexpr int kBM = 128;          // rows of the largest tile (= TMEM lanes); a launch uses bm = 64 or 128
constexpr int kBK = 64;           // 64 bf16 = 128 bytes = one 128B-swizzle row
constexpr int kThreads = 256;
constexpr int kEpiWarps = 4;      // epilogue warps; each releases its own rows of a tile
constexpr int kSchedDepth = 4;
constexpr int kMaxPipe = 16;
constexpr int kTicketLead = 4;    // k-blocks before the end of a slice at which the next ticket is taken
constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KB: the A tile of a 128-row tile

// Device status codes (match mlp_status).
constexpr uint32_t kStatusTimeout = 5;
constexpr uint32_t kStatusBadTile = 7;

struct StageParams {
    int32_t M, K, N;
    int32_t BN;             // tile width (32, 64, 128, 256)
    int32_t tiles_m, tiles_n;
    int32_t k_blocks;
    int32_t b_swz;          // bytes of one B swizzle row: 128 (BN >= 64) or 64 (BN = 32)
    __nv_bfloat16 *out;     // M x N row-major
    const __nv_bfloat16 *residual;  // M x N (the chain input) or null
    int32_t gelu;
    int32_t b_kmajor;       // 1: weights stored N x K, B tile is K-major (one box of BN rows)
    int32_t b_3d;           // weights K x N with N a multiple of the box width: the map is a 3-D
                            // view (box column, k, box) and one copy loads every box of a B tile
    int32_t split;          // CTAs sharing one tile (divides the cluster size): S k-slices, each on
                            // one CTA, or on a CTA pair (then 2 S, rank 2 q + h: slice q, half h)
    int32_t kb_per_split;   // k blocks of each slice (the last one may get fewer)
    int32_t tiles_per_item; // cluster size / S
    int32_t items;          // cluster items of this stage
    float *partials;        // split-K through global memory: one 128 x BN fp32 buffer per CTA
    int32_t dsmem_reduce;   // split-K through the owners' shared memory (BN * 512 <= recv_bytes)
    int32_t gated;          // SwiGLU: B tiles of gate (mapB) and up (mapU) weights, accumulators
                            // side by side in TMEM, output SiLU(gate) * up; unsplit
    int32_t xsplit;         // split-K slices on separate clusters (pipelined CTA pairs, a one-wave stage
                            // after a one-group boundary): a cluster item is one slice of one tile,
                            // siblings exchange partial sums through their own buffers and count on
                            // xcount (per tile and pair half) instead of the cluster's barriers
    uint32_t *xcount;       // xsplit: releases of the slices' partials, accumulating over runs
    int32_t kpf;            // 64-deep k blocks per ring fill: 0 or 1, or 2 (one CTA per tile, plain
                            // stage, even k blocks per slice): mapA is then a 3-D view (column, row,
                            // k block) and mapB a 3-D (K-major) or 4-D (column in box, k, box,
                            // k block) one, so each operand of a fill is still one copy
};

// Stage boundary s -> s+1.  The scoreboard holds one counter per group of consumer tiles with
// identical producer sets (a row panel for GEMM chains); see dep_groups.h.
struct BoundaryParams {
    const int32_t *pg_off;     // producer tile -> groups it feeds (CSR)
    const int32_t *pg_tgt;
    const int32_t *grp_off;    // group -> member consumer tiles (CSR)
    const int32_t *grp_mem;
    const int32_t *grp_init;   // releases each group waits for per run: producer tiles x split x kEpiWarps
    const int32_t *cgrp;       // consumer tile -> its group
    uint32_t *count;           // one counter per group: releases so far, over all runs of the handle
    unsigned long long *queue; // one slot per consumer tile
    uint32_t *tail;            // queue slots reserved so far, over all runs of the handle
    uint32_t slots_per_run;    // consumer tiles: the tail's increments in one run
    // K-granular mode: per producer tile, the releases seen so far (ready_quota per run,
    // accumulated over the handle's runs and compared against the run's epoch).
    uint32_t *ready;
    uint32_t ready_quota;      // releases of one producer tile in one run: split x kEpiWarps
    // Queue-free boundary: one scoreboard group for the whole boundary (a single row panel, or one
    // raster group of all panels), or no more consumer items than co-resident clusters (every
    // consumer item gets a cluster of its own, so no CTA could run a ready tile in place of one it
    // waits for).  The queue would carry no order that matters: consumer slot q takes member q of
    // the groups in group order (grp_mem as stored) and acquires its group's counter directly, and
    // releases push nothing.  Queue protocol only (the Lamport mode keeps its queue entries).
    int32_t queue_free;
};

struct EventRec {
    int32_t stage, tile, smid, cta;
    uint64_t t_start, t_end;
    uint32_t seq_start, seq_end;
    uint64_t t_acc;   // accumulator complete (split tiles: the split-0 slice)
};

struct ChainParams {
    CUtensorMap mapA[kMaxStages];
    CUtensorMap mapB[kMaxStages];
    CUtensorMap mapU;                    // up-projection weights of a gated first stage
    StageParams st[kMaxStages];
    BoundaryParams bd[kMaxStages - 1];
    int32_t num_stages;
    int32_t pipelined;
    int32_t kwait;                       // pipelined with per-k-block producer waits, no work-queue
    int32_t lamport;                     // pipelined, fence-free: consumers validate what they load
    int32_t force_reload;                // Lamport test hook: reload every consumer A tile once
    int32_t pdl_wait;                    // programmatic dependent of the previous stage's launch:
                                         // the TMA warp waits for it before its first load
    int32_t pdl_trigger;                 // a later stage is launched as this launch's dependent
    int32_t pair;                        // 2: CTA pairs (chain_kernel<2>), each tile 2 bm rows
    int32_t first_stage;                 // non-pipelined launches run this single stage
    int32_t m_tile_begin, m_tile_end;    // ... over these row tiles
    int32_t stage_base[kMaxStages + 1];  // pipelined: first ticket (cluster item) of each stage
    int32_t tile_base[kMaxStages + 1];   // first event-log record of each stage
    int32_t cs;                          // cluster size
    int32_t bm;                          // rows per tile: 128, or 64 (tcgen05 M = 64)
    uint32_t a_bytes;                    // bytes of one A tile in a ring slot: bm x 64 bf16
    int32_t raster_group;
    int32_t num_pipe;                    // shared-memory ring depth
    uint32_t stage_bytes;                // bytes of one ring slot (A + B)
    uint32_t tmem_cols;
    int32_t acc_stride;                  // TMEM columns between the two accumulator buffers
    int32_t acc_split;                   // 1, or 2: k16 steps alternate between two sub-accumulators
    int32_t sub_stride;                  // TMEM columns between the sub-accumulators of a buffer
    int32_t partial_floats;              // floats per CTA partial buffer (128 x max tile width)
    uint32_t recv_bytes;                 // split-K receive buffer in shared memory (0: none)
    int32_t drop_tile;                   // fault injection (-1: off)
    uint64_t timeout_ns;
    uint32_t *ticket;                    // tickets taken so far, over all runs of the handle
    uint32_t tickets_per_run;            // cluster items of all stages: the ticket's increments in one run
    unsigned long long *launches;        // CTAs started so far: run e's CTAs read e x ctas ..
    uint32_t *status;
    uint32_t *seq;
    EventRec *events;                    // null: no event log; else one record per tile of every
                                         // stage (tile_base), then one per CTA of the launch
    const uint8_t *meta;                 // protocol state (counters, queues, dependency tables) ...
    uint32_t meta_bytes;                 // ... prefetched into L2 at launch (0: none)
};

struct __align__(8) Ctrl {
    uint64_t full[kMaxPipe], empty[kMaxPipe];
    uint64_t tfull[2], tempty[2];
    uint64_t sfull[kSchedDepth], sempty[kSchedDepth];
    uint64_t drain;
    uint64_t want_next;   // TMA -> scheduler: take the next ticket now
    uint64_t valid[kMaxPipe];   // Lamport: the slot's A tile holds no sentinel (warp 3 -> MMA)
    uint64_t reload[kMaxPipe];  // Lamport: completion of a reloaded A tile
    uint64_t epoch_bar;   // the run's epoch is in `epoch` (warp 3, once per launch)
    uint64_t red_bar;     // split-K: every sibling's partial is written
    uint64_t done_bar;    // split-K: every sibling has read its parts of my partial
    int32_t item_stage[kSchedDepth], item_tile[kSchedDepth], item_split[kSchedDepth];
    uint32_t tmem_base;
    volatile int32_t abort_flag;
    int32_t skip;
    uint32_t epoch;
};

constexpr uint32_t kEpiStageBytes = 32 * 64;   // per epilogue warp: 32 rows x 32 bf16 columns
constexpr uint32_t kRecvBytes = 64 * 1024;     // split-K receive buffer: S parts of a 128 x 128/S slice

// Shared memory: [ring: num_pipe x stage_bytes][4 x epilogue staging][split-K receive buffer]
// [Ctrl], the ring 1024-byte aligned.
__host__ __device__ inline uint32_t staging_offset(int num_pipe, uint32_t stage_bytes)
{
    return static_cast<uint32_t>(num_pipe) * stage_bytes;
}

__host__ __device__ inline uint32_t recv_offset(int num_pipe, uint32_t stage_bytes)
{
    return staging_offset(num_pipe, stage_bytes) + 4 * kEpiStageBytes;
}

__host__ __device__ inline uint32_t ctrl_offset(int num_pipe, uint32_t stage_bytes, uint32_t recv_bytes)
{
    return recv_offset(num_pipe, stage_bytes) + recv_bytes;
}

__host__ inline size_t chain_smem_bytes(int num_pipe, uint32_t stage_bytes, uint32_t recv_bytes)
{
    return 1024 + ctrl_offset(num_pipe, stage_bytes, recv_bytes) + sizeof(Ctrl);
}

// ------------------------------------------------------------------------ bounded waits --
// Every wait has a deadline.  On expiry the waiter records kStatusTimeout (first error wins)
// and raises the CTA's abort flag so the other roles stop too.  Returns false on abort.
// Drain waits (after an abort, for this CTA's own copies and MMAs in flight) ignore the abort
// flag and use a short fixed limit.  Waits on phases completed by other CTAs of the cluster
// acquire at cluster scope.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, Ctrl *c, const ChainParams &p,
                                         bool honor_abort = true, bool cluster_scope = false)
{
    auto probe = [&]() { return cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (probe())
        return true;
    const uint64_t t0 = globaltimer_ns();
    const uint64_t limit = honor_abort ? 2 * p.timeout_ns + 1000000000ull : 200000000ull;
    while (true) {
        if (probe())
            return true;
        if (honor_abort && c->abort_flag)
            return false;
        if (globaltimer_ns() - t0 > limit) {
            atomicCAS(p.status, 0u, kStatusTimeout);
            c->abort_flag = 1;
            return false;
        }
    }
}

// Warp-collective wait: lane 0 waits, the result is broadcast so the warp stays converged.
__device__ __forceinline__ bool warp_wait_bar(uint64_t *bar, uint32_t parity, Ctrl *c, const ChainParams &p,
                                              bool cluster_scope = false)
{
    uint32_t ok = 0;
    if ((threadIdx.x & 31) == 0)
        ok = wait_bar(bar, parity, c, p, true, cluster_scope) ? 1u : 0u;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
}

// As warp_wait_bar, and then every lane acquires the completed phase itself (a try_wait that
// succeeds at once), so every lane may read what the arriving thread published.
__device__ __forceinline__ bool warp_wait_bar_all(uint64_t *bar, uint32_t parity, Ctrl *c, const ChainParams &p)
{
    if (!warp_wait_bar(bar, parity, c, p))
        return false;
    mbar_try_wait(bar, parity);
    return true;
}

__device__ __forceinline__ float gelu_tanh_f32(float x)
{
    const float k0 = 0.7978845608028654f;             // sqrt(2 / pi)
    const float k01 = 0.7978845608028654f * 0.044715f;
    // the epilogue's critical path on one-wave stages: one MUFU tanh instead of a tanhf call,
    // and the polynomial as x (k0 + k0 k1 x^2), then h + h t with h = x / 2: six instructions
    const float t = tanh_approx(x * fmaf(k01, x * x, k0));
    const float h = 0.5f * x;
    return fmaf(h, t, h);
}

// Arrive on the same mbarrier in CTA `rank` of this cluster, `count` times, without release
// semantics (the caller fences once before a batch of these).
__device__ __forceinline__ void arrive_rank_relaxed(uint64_t *bar, uint32_t rank, uint32_t count)
{
    mbar_arrive_relaxed_cluster(map_to_rank(bar, rank), count);
}

// Arrive on the same mbarrier in CTA `rank` of this cluster, `count` times.
__device__ __forceinline__ void arrive_rank(uint64_t *bar, uint32_t rank, uint32_t count)
{
    const uint32_t a = map_to_rank(bar, rank);
    if (count == 1)
        mbar_arrive_cluster(a);
    else
        asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(a), "r"(count)
                     : "memory");
}

// ------------------------------------------------------------------------------ scheduler --
// The tiles of one cluster item: pipelined ticket t, or the `item`-th static item of a
// non-pipelined launch.  Returns the stage (-1: no work left) and fills tiles[0 .. ntiles).
__device__ __forceinline__ int32_t item_tiles(const ChainParams &p, int32_t t, int32_t &ntiles,
                                              int32_t (&tiles)[kMaxCluster], int32_t &slice)
{
    ntiles = 0;
    slice = -1;
    if (p.pipelined) {
        if (t >= p.stage_base[p.num_stages])
            return -1;
        const int32_t s = stage_of_ticket(p.stage_base, t);
        const StageParams &sp = p.st[s];
        const int32_t ntile_stage = sp.tiles_m * sp.tiles_n;
        if (sp.xsplit) {   // one k-slice of one tile (or work-queue slot); its siblings are the neighbouring tickets
            const int32_t slices = sp.split / p.pair;
            const int32_t local = t - p.stage_base[s];
            const int32_t first = local / slices;
            slice = local % slices;
            ntiles = 1;
            tiles[0] = s == 0 ? raster_tile(first, sp.tiles_m, sp.tiles_n, p.raster_group) : first;
            return s;
        }
        const int32_t first = (t - p.stage_base[s]) * sp.tiles_per_item;
        ntiles = min(sp.tiles_per_item, ntile_stage - first);
        // Stage 0 tiles (and every stage's in the K-granular mode) follow the raster order; a
        // consumer item of the queue protocol carries work-queue slots (first + j), which the
        // CTAs that run it poll themselves (resolve_queue_slot), so the broadcast is off the
        // path from a queue push to the first load.
        for (int32_t j = 0; j < ntiles; ++j)
            tiles[j] = (s == 0 || p.kwait) ? raster_tile(first + j, sp.tiles_m, sp.tiles_n, p.raster_group) : first + j;
        return s;
    }
    const StageParams &sp = p.st[p.first_stage];
    const int32_t n_local = (p.m_tile_end - p.m_tile_begin) * sp.tiles_n;
    const int32_t first = t * sp.tiles_per_item;
    if (first >= n_local)
        return -1;
    ntiles = min(sp.tiles_per_item, n_local - first);
    for (int32_t j = 0; j < ntiles; ++j)
        tiles[j] = p.m_tile_begin * sp.tiles_n + first + j;
    return p.first_stage;
}

// The tile and split index of cluster rank r in an item (see StageParams::split, ::xsplit).
__device__ __forceinline__ void item_member(const ChainParams &p, int32_t stage, int32_t ntiles,
                                            const int32_t (&tiles)[kMaxCluster], int32_t slice, int32_t S, int32_t r,
                                            int32_t &tile, int32_t &split)
{
    if (slice >= 0) {
        tile = tiles[0];
        split = slice * p.pair + r;
        return;
    }
    const int32_t j = r / S;
    tile = (stage >= 0 && j < ntiles) ? tiles[j] : -1;
    split = r % S;
}

// Rank 0 of each cluster: obtain the cluster's next items and broadcast them.  Item 0 is
// ticket (or static item) = the cluster's id, which every CTA writes into its own ring slot 0 at
// launch; from item 1 on, pipelined tickets come from a device-wide counter offset by the
// number of clusters.
__device__ __forceinline__ void role_scheduler(const ChainParams &p, Ctrl *c)
{
    const int32_t cs = p.cs;
    const int32_t nclusters = static_cast<int32_t>(num_clusters_x());
    if (c->item_stage[0] < 0)
        return;   // not even a first item for this cluster
    if (p.pipelined && !wait_bar(&c->epoch_bar, 0, c, p))   // tickets are read relative to the epoch
        return;
    for (int32_t it = 1;; ++it) {
        const int32_t slot = it % kSchedDepth;
        const uint32_t ph = (it / kSchedDepth) & 1;
        if (!wait_bar(&c->sempty[slot], ph ^ 1, c, p, true, true))
            return;
        // Take tickets just in time: a ticket taken early would sit in this cluster while
        // others idle, so wait until the TMA warp is about to finish its current slice.
        if (!wait_bar(&c->want_next, (it - 1) & 1, c, p))
            return;
        const int32_t t = p.pipelined ? nclusters + static_cast<int32_t>(run_relative(
                                                        atom_add_relaxed_gpu(p.ticket, 1u), c->epoch, p.tickets_per_run))
                                      : static_cast<int32_t>(cluster_id_x()) + it * nclusters;
        int32_t ntiles = 0, slice = -1;
        int32_t tiles[kMaxCluster];
        const int32_t stage = item_tiles(p, t, ntiles, tiles, slice);
        // Broadcast: rank r gets tile r / S of the item (or none) and k-slice r % S (a slice item
        // of a cross-cluster split: the tile, and CTA r of the slice's pair).  All items are
        // written first and released by one fence: a release arrive per rank would cost a round
        // trip each and start the last rank's slice that much later than the first's.
        const int32_t S = stage >= 0 ? p.st[stage].split : 1;
        for (int32_t r = 0; r < cs; ++r) {
            int32_t tile, split;
            item_member(p, stage, ntiles, tiles, slice, S, r, tile, split);
            st_cluster_s32(map_to_rank(&c->item_stage[slot], r), stage);
            st_cluster_s32(map_to_rank(&c->item_tile[slot], r), tile);
            st_cluster_s32(map_to_rank(&c->item_split[slot], r), split);
        }
        fence_acq_rel_cluster();
        for (int32_t r = 0; r < cs; ++r)
            arrive_rank_relaxed(&c->sfull[slot], r, 1);
        if (stage < 0)
            return;
    }
}

// The item of ring slot `slot`: stage, tile (in a pipelined run's consumer stages: the
// work-queue slot that names the tile) and k-slice.
struct Item {
    int32_t stage, tile, split;
};

// The queue entry names the tile; the synchronisation with the producers is an acquire of the
// tile's group counter, which every producer warp incremented with a release (fence + relaxed
// add): reading the run's final count makes all of their stores visible.  The pusher therefore
// stores the entries without a fence of its own.  False after an error (status recorded, abort
// raised).
__device__ __forceinline__ bool acquire_group(const ChainParams &p, Ctrl *c, int32_t s, int32_t tile)
{
    const BoundaryParams &bd = p.bd[s - 1];
    const int32_t g = bd.cgrp[tile];
    const uint32_t want = run_target(bd.grp_init[g], c->epoch);
    const uint64_t t0 = globaltimer_ns();
    while (!count_reached(ld_acquire_gpu_u32(bd.count + g), want)) {
        if (c->abort_flag)
            return false;
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            atomicCAS(p.status, 0u, kStatusTimeout);
            c->abort_flag = 1;
            return false;
        }
    }
    return true;
}

// Consumer prologue (the injected prologue of section III-A, Fig. 1): poll work-queue slot
// `qslot` of the boundary before stage s until this run's entry lands, with back-off and a
// deadline.  Returns the consumer tile it names, or -1 after an error (status recorded, this
// CTA's abort flag raised).  The caller orders its later TMA reads with a proxy fence.
__device__ __forceinline__ int32_t resolve_queue_slot(const ChainParams &p, Ctrl *c, int32_t s, int32_t qslot,
                                                      bool acquire)
{
    // Relaxed polls: the entry only names the tile (the acquire is on the group counter below).
    // A queue-free boundary names the members in group order: slot q is grp_mem[q].
    const bool queue_free = p.bd[s - 1].queue_free != 0;
    const unsigned long long *q = p.bd[s - 1].queue + qslot;
    uint64_t v = queue_free ? queue_entry(c->epoch, p.bd[s - 1].grp_mem[qslot]) : ld_relaxed_gpu_u64(q);
    if (!queue_entry_ready(v, c->epoch)) {
        const uint64_t t0 = globaltimer_ns();
        uint32_t backoff = 32;
        while (true) {
            __nanosleep(backoff);
            backoff = backoff < 64 ? backoff * 2 : 64;
            v = ld_relaxed_gpu_u64(q);
            if (queue_entry_ready(v, c->epoch))
                break;
            if (c->abort_flag)
                return -1;
            if (ld_relaxed_gpu_u32(p.status) != 0) {
                c->abort_flag = 1;
                return -1;
            }
            if (globaltimer_ns() - t0 > p.timeout_ns) {
                atomicCAS(p.status, 0u, kStatusTimeout);
                c->abort_flag = 1;
                return -1;
            }
        }
    }
    const int32_t tile = queue_entry_tile(v);
    if (tile < 0 || tile >= p.st[s].tiles_m * p.st[s].tiles_n) {
        atomicCAS(p.status, 0u, kStatusBadTile);
        c->abort_flag = 1;
        return -1;
    }
    if (acquire && !acquire_group(p, c, s, tile))
        return -1;
    return tile;
}

__device__ __forceinline__ Item read_item(Ctrl *c, int32_t slot)
{
    return Item{c->item_stage[slot], c->item_tile[slot], c->item_split[slot]};
}

// Hand ring slot `slot` back to the scheduler (a release: the item's reads come first).
__device__ __forceinline__ void free_item_slot(Ctrl *c, int32_t slot)
{
    arrive_rank(&c->sempty[slot], 0, 1);
}

__device__ __forceinline__ Item take_item(Ctrl *c, int32_t slot)
{
    const Item it = read_item(c, slot);
    free_item_slot(c, slot);
    return it;
}

// K-granular consumer wait: block until every epilogue warp of every split-K slice of producer
// tile `ptile` (the stage before s) has released its rows in this run.  Relaxed polls with
// back-off and a deadline; the caller fences once after the last wait of a k-block.  Returns
// false after an error (status recorded, abort raised).
__device__ __forceinline__ bool wait_producer(const ChainParams &p, Ctrl *c, int32_t s, int32_t ptile)
{
    const BoundaryParams &bd = p.bd[s - 1];
    const uint32_t want = run_target(static_cast<int32_t>(bd.ready_quota), c->epoch);
    const uint32_t *r = bd.ready + ptile;
    if (count_reached(ld_relaxed_gpu_u32(r), want))
        return true;
    const uint64_t t0 = globaltimer_ns();
    uint32_t backoff = 32;
    while (true) {
        __nanosleep(backoff);
        backoff = backoff < 64 ? backoff * 2 : 64;
        if (count_reached(ld_relaxed_gpu_u32(r), want))
            return true;
        if (c->abort_flag)
            return false;
        if (ld_relaxed_gpu_u32(p.status) != 0) {
            c->abort_flag = 1;
            return false;
        }
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            atomicCAS(p.status, 0u, kStatusTimeout);
            c->abort_flag = 1;
            return false;
        }
    }
}

// Producer column tiles hi+1, hi+2, ... (up to `last`) of the row panel at `pbase` that have
// already released in this run, taken in batches of relaxed loads issued together; returns the
// last column tile of the unbroken ready run starting at hi.
__device__ __forceinline__ int32_t scan_ready(const ChainParams &p, const Ctrl *c, int32_t s, int32_t pbase,
                                              int32_t hi, int32_t last)
{
    const BoundaryParams &bd = p.bd[s - 1];
    const uint32_t want = run_target(static_cast<int32_t>(bd.ready_quota), c->epoch);
    while (hi < last) {
        uint32_t v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            v[j] = hi + 1 + j <= last ? ld_relaxed_gpu_u32(bd.ready + pbase + hi + 1 + j) : 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (hi + 1 + j > last || !count_reached(v[j], want))
                return hi + j;
        }
        hi += 8;
    }
    return hi;
}

// The k-slice of a tile's CTA `split` (see StageParams::split).
template <int kPair>
__device__ __forceinline__ int32_t kslice_of(int32_t split)
{
    return kPair == 2 ? split >> 1 : split;
}

__device__ __forceinline__ void slice_range(int32_t k_blocks, int32_t kb_per_split, int32_t split, int32_t &kb0,
                                            int32_t &kb1)
{
    kb0 = split * kb_per_split;
    kb1 = min(k_blocks, kb0 + kb_per_split);
}

// ---------------------------------------------------------------------------- TMA producer --
// With a CTA pair (kPair = 2) each CTA loads its own 128 rows of the 256-row A tile and its half
// of the B tile's columns into its own ring, and both CTAs' copies complete on the leader's full
// barrier.  The leader arms each fill (expect_tx of both CTAs' bytes) before it lets the peer fill
// the same slot (a relaxed arrive on the peer's empty barrier), so the peer only ever copies into
// phases the leader waits for; the leader's own empty barrier is released by its MMA commit.
template <int kPair>
__device__ __forceinline__ void role_tma(const ChainParams &p, Ctrl *c, uint8_t *ring, bool leader)
{
    constexpr bool kPairMode = kPair == 2;
    // Kernel parameters live in constant memory behind a generic pointer; every asm statement
    // with a memory clobber would force them to be re-read, so the loop works from registers.
    const int32_t num_pipe = p.num_pipe;
    const uint32_t stage_bytes = p.stage_bytes;
    const uint64_t pol_act = policy_evict_last();    // activations are re-read by many tiles
    const uint64_t pol_w = policy_evict_first();     // each weight tile is read by one row panel
    const bool pipelined = p.pipelined != 0;
    const bool kwait = pipelined && p.kwait != 0;
    EventRec *const events = pipelined ? p.events : nullptr;
    const int32_t bm = p.bm;
    const uint32_t a_bytes = p.a_bytes;
    const uint32_t rank = cluster_ctarank();
    const uint32_t half = kPairMode ? (rank & 1u) : 0u;   // 0: the pair's leader
    // shared::cluster addresses of the leader's full barriers and of the peer's empty barriers
    const uint32_t full_lead0 = kPairMode ? map_to_rank(&c->full[0], rank & ~1u) : 0u;
    const uint32_t empty_peer0 = kPairMode ? map_to_rank(&c->empty[0], rank | 1u) : 0u;
    int32_t ps = 0;
    uint32_t pph = 0;
    // Programmatic dependent launch: the previous GEMM's output (this launch's A) is complete and
    // visible after this.  (Sending the first ring-full of weight copies before the wait measured
    // slower: they compete with the previous GEMM's last loads; so did prefetching its weights
    // into L2 with bulk tensor prefetches, which occupy the TMA engine like copies.)
    if (p.pdl_wait)
        griddep_wait();
    // Ring slots are filled in order 0, 1, ..., num_pipe - 1, 0, ...: the count of copies issued
    // says how often each slot was filled (a per-slot array would live in local memory, and its
    // read-modify-write sits on the per-k-block issue path).
    uint32_t issued = 0;
    bool have_epoch = false;   // the run's epoch is needed from the first consumer item on
    for (int32_t it = 0;; ++it) {
        const int32_t slot = it % kSchedDepth;
        if (!wait_bar(&c->sfull[slot], (it / kSchedDepth) & 1, c, p, true, true))
            break;
        // The slot goes back to the scheduler only after this item's loads are issued: the
        // release round trip then stays off the path to the first load.
        const Item item = read_item(c, slot);
        if (item.stage < 0 || item.tile < 0) {
            free_item_slot(c, slot);
            if (item.stage < 0)
                break;
            continue;
        }
        const int32_t s = item.stage;
        int32_t tile = item.tile;
        const bool kwait_s = kwait && s > 0;
        if (pipelined && s > 0 && !have_epoch) {   // queue entries and ready counts carry the epoch
            if (!wait_bar(&c->epoch_bar, 0, c, p)) {
                free_item_slot(c, slot);
                break;
            }
            have_epoch = true;
        }
        // At a queue-free boundary the slot names its tile without a wait (the acquire follows).
        const bool queue_free = pipelined && s > 0 && !kwait && !p.lamport && p.bd[s - 1].queue_free != 0;
        if (pipelined && s > 0 && !kwait) {
            tile = resolve_queue_slot(p, c, s, item.tile, !p.lamport && !queue_free);   // Lamport: validated instead
            if (tile < 0) {
                free_item_slot(c, slot);
                break;
            }
        }
        auto log_start = [&]() {   // (a consumer's start is taken after its acquire)
            if (events && item.split == 0) {
                EventRec *e = events + p.tile_base[s] + tile;
                e->stage = s;
                e->tile = tile;
                e->smid = static_cast<int32_t>(smid());
                e->cta = static_cast<int32_t>(blockIdx.x);
                e->seq_start = atom_add_relaxed_gpu(p.seq, 1u);
                e->t_start = globaltimer_ns();
            }
        };
        const StageParams &spr = p.st[s];
        const int32_t tiles_n = spr.tiles_n, BN = spr.BN, b_swz = spr.b_swz, b_kmajor = spr.b_kmajor;
        const bool b_3d = spr.b_3d != 0;
        const int32_t k_blocks = spr.k_blocks, kbps = spr.kb_per_split;
        const CUtensorMap *mapA = &p.mapA[s];
        const CUtensorMap *mapB = &p.mapB[s];
        const bool gated = spr.gated != 0;
        // a pair's tile is 2 bm rows: this CTA's rows and its half of the tile's columns (of a gated
        // tile, whose MMA is twice as wide, the leader's half is the gate tile and the peer's the up
        // tile, both at the tile's columns)
        const bool gated_pair = kPairMode && gated;
        const int32_t bn_cta = gated_pair ? BN : BN / kPair;
        const int32_t m0 = (tile / tiles_n) * (kPair * bm) + static_cast<int32_t>(half) * bm;
        const int32_t n0 = (tile % tiles_n) * BN + (gated_pair ? 0 : static_cast<int32_t>(half) * bn_cta);
        const int32_t box_cols = b_swz / 2;
        const uint32_t box_bytes = kBK * b_swz;
        const int32_t nbox = (bn_cta + box_cols - 1) / box_cols;   // a ragged last box is loaded whole
        const uint32_t b_tile_bytes = b_kmajor ? static_cast<uint32_t>(kBK * bn_cta * 2) : static_cast<uint32_t>(nbox) * box_bytes;
        const uint32_t bytes = a_bytes + (gated && !kPairMode ? 2u : 1u) * b_tile_bytes;
        int32_t kb0, kb1;
        slice_range(k_blocks, kbps, kslice_of<kPair>(item.split), kb0, kb1);   // a pair's halves run the same slice
        const int32_t lead_kb = kb1 - kb0 > kTicketLead ? kb1 - kTicketLead : kb0;
        // K-granular mode: the A tile of k block kb reads columns [kb*64, kb*64+64) of the
        // previous stage's output, written by producer tiles kb*64/pBN .. (kb*64+63)/pBN of the
        // same row panel; ready_hi is the last producer column tile known released.
        const int32_t pBN = kwait_s ? p.st[s - 1].BN : 1;
        const int32_t ptn = kwait_s ? p.st[s - 1].tiles_n : 1;
        const int32_t pbase = kwait_s ? (tile / tiles_n) * ptn : 0;
        int32_t ready_hi = -1;
        const int32_t slice_last = kwait_s ? min(((kb1 - 1) * kBK + kBK - 1) / pBN, ptn - 1) : 0;
        // Weights before the acquire (queue-free boundary, one-block fills; one CTA per tile with
        // the B tile in one copy, or a CTA pair): the first ring-full of weight copies goes out
        // while the producers finish, the activation copies of those fills after the acquire.
        const bool early = queue_free && spr.kpf != 2 && (kPairMode || b_kmajor || b_3d || nbox == 1);
        if (queue_free && !early && !acquire_group(p, c, s, tile)) {
            free_item_slot(c, slot);
            break;
        }
        if (!early) {
            if (s > 0 && !kwait_s)   // TMA (async proxy) reads of a producer's output come after the acquire
                fence_proxy_async_global();
            log_start();
        }
        bool ok = true;
        if constexpr (kPairMode) {
            // Pair stages have no K-granular waits or Lamport: the B tile's half is one copy (N x K
            // weights, or a 3-D view of K x N ones), or one per box (ragged N); of a gated stage,
            // the gate tile (leader) or the up tile (peer).
            const CUtensorMap *mapBh = gated_pair && half ? &p.mapU : mapB;
            const int32_t bx = b_kmajor ? 0 : (b_3d ? 0 : n0);
            const int32_t by = b_kmajor ? n0 : (b_3d ? n0 / box_cols : 0);
            const int32_t b_form = b_kmajor ? 0 : (b_3d ? 1 : 2);
            const uint32_t pair_bytes = 2u * bytes;
            // Wait for the slot of k block kb (the leader for its MMA's release of the slot's
            // previous fill, the peer for the leader's go-ahead for this fill), arm it (leader) and
            // send this CTA's half of the B tile.
            auto arm_fill_b = [&](int32_t kb) {
                if (leader && kb == lead_kb)
                    mbar_arrive(&c->want_next);
                if (!wait_bar(&c->empty[ps], half ? pph : pph ^ 1, c, p, true, half != 0))
                    return false;
                uint8_t *a = ring + static_cast<size_t>(ps) * stage_bytes;
                const uint32_t fb = full_lead0 + static_cast<uint32_t>(ps) * 8u;
                if (!half) {
                    mbar_arrive_expect_tx(&c->full[ps], pair_bytes);
                    mbar_arrive_relaxed_cluster(empty_peer0 + static_cast<uint32_t>(ps) * 8u, 1u);
                }
                const int32_t k = kb * kBK;
                if (b_form == 0)
                    tma_load_2d_pair(a + a_bytes, mapBh, fb, k, by, pol_w);
                else if (b_form == 1)
                    tma_load_3d_pair(a + a_bytes, mapBh, fb, 0, k, by, pol_w);
                else   // a ragged N keeps the 2-D map: one copy per 64-column box of the half
                    for (int32_t j = 0; j < nbox; ++j)
                        tma_load_2d_pair(a + a_bytes + j * box_bytes, mapBh, fb, bx + j * box_cols, k, pol_w);
                return true;
            };
            int32_t kb_first = kb0;
            if (early) {   // as in the one-CTA loop below: weights, the acquire, then activations
                const int32_t n_early = min(num_pipe, kb1 - kb0);
                const int32_t ps0 = ps;
                int32_t armed = 0;
                for (; armed < n_early; ++armed) {
                    if (!arm_fill_b(kb0 + armed)) {
                        ok = false;
                        break;
                    }
                    if (++ps == num_pipe) {
                        ps = 0;
                        pph ^= 1;
                    }
                }
                if (ok && !acquire_group(p, c, s, tile))
                    ok = false;
                fence_proxy_async_global();
                if (ok)
                    log_start();
                for (int32_t i = 0; i < armed; ++i) {
                    const int32_t sl = ps0 + i < num_pipe ? ps0 + i : ps0 + i - num_pipe;
                    tma_load_2d_pair(ring + static_cast<size_t>(sl) * stage_bytes, mapA,
                                     full_lead0 + static_cast<uint32_t>(sl) * 8u, (kb0 + i) * kBK, m0, pol_act);
                    ++issued;
                }
                kb_first = kb0 + armed;
            }
            for (int32_t kb = kb_first; kb < kb1 && ok; ++kb) {
                if (!arm_fill_b(kb)) {
                    ok = false;
                    break;
                }
                tma_load_2d_pair(ring + static_cast<size_t>(ps) * stage_bytes, mapA,
                                 full_lead0 + static_cast<uint32_t>(ps) * 8u, kb * kBK, m0, pol_act);
                ++issued;
                if (++ps == num_pipe) {
                    ps = 0;
                    pph ^= 1;
                }
            }
        } else if (spr.kpf == 2) {
            // Two k blocks per fill (never K-granular or gated): the slot holds the A tiles of k
            // blocks kb and kb + 1, then their B tiles, each laid out as in a one-block fill; one
            // copy per operand, one barrier phase, twice the bytes, half the ring slots.  (Slices
            // hold an even number of blocks, so lead_kb - kb0 is even and kb meets it.)
            const int32_t by = b_kmajor ? n0 : n0 / box_cols;
            const uint32_t fill_bytes = 2u * bytes;
            for (int32_t kb = kb0; kb < kb1; kb += 2) {
                if (leader && kb == lead_kb)
                    mbar_arrive(&c->want_next);
                if (!wait_bar(&c->empty[ps], pph ^ 1, c, p)) {
                    ok = false;
                    break;
                }
                uint8_t *a = ring + static_cast<size_t>(ps) * stage_bytes;
                mbar_arrive_expect_tx(&c->full[ps], fill_bytes);
                if (b_kmajor)
                    tma_load_3d(a + 2u * a_bytes, mapB, &c->full[ps], 0, by, kb, pol_w);
                else
                    tma_load_4d(a + 2u * a_bytes, mapB, &c->full[ps], 0, 0, by, kb, pol_w);
                tma_load_3d(a, mapA, &c->full[ps], 0, m0, kb, pol_act);
                ++issued;
                if (++ps == num_pipe) {
                    ps = 0;
                    pph ^= 1;
                }
            }
        } else if (!kwait_s && (b_kmajor || b_3d || nbox == 1)) {
            // The common case: two copies per k block (three for a gated stage: gate and up
            // weights), the B tile in one copy whatever its layout, no per-k-block mode
            // branches; see role_mma for why that matters.
            const int32_t bx = b_kmajor ? 0 : (b_3d ? 0 : n0);   // B coordinates, k excluded
            const int32_t by = b_kmajor ? n0 : (b_3d ? n0 / box_cols : 0);
            const int32_t b_form = b_kmajor ? 0 : (b_3d ? 1 : 2);
            const CUtensorMap *mapU = &p.mapU;
            int32_t kb_first = kb0;
            if (early) {
                // Arm the first ring-full of fills with their weight copies, acquire the producers'
                // output, then send the activation copies of the armed fills (also after a failed
                // wait: every armed fill's transaction count must complete, so that the drain
                // below accounts for its copies).
                const int32_t n_early = min(num_pipe, kb1 - kb0);
                const int32_t ps0 = ps;
                int32_t armed = 0;
                for (; armed < n_early; ++armed) {
                    const int32_t kb = kb0 + armed;
                    if (leader && kb == lead_kb)
                        mbar_arrive(&c->want_next);
                    if (!wait_bar(&c->empty[ps], pph ^ 1, c, p)) {
                        ok = false;
                        break;
                    }
                    uint8_t *a = ring + static_cast<size_t>(ps) * stage_bytes;
                    mbar_arrive_expect_tx(&c->full[ps], bytes);
                    for (int32_t u = 0; u < (gated ? 2 : 1); ++u) {
                        const CUtensorMap *mb = u ? mapU : mapB;
                        uint8_t *bt = a + a_bytes + u * b_tile_bytes;
                        if (b_form == 0)
                            tma_load_2d(bt, mb, &c->full[ps], kb * kBK, by, pol_w);
                        else if (b_form == 1)
                            tma_load_3d(bt, mb, &c->full[ps], 0, kb * kBK, by, pol_w);
                        else
                            tma_load_2d(bt, mb, &c->full[ps], bx, kb * kBK, pol_w);
                    }
                    if (++ps == num_pipe) {
                        ps = 0;
                        pph ^= 1;
                    }
                }
                if (ok && !acquire_group(p, c, s, tile))
                    ok = false;
                fence_proxy_async_global();
                if (ok)
                    log_start();
                for (int32_t i = 0; i < armed; ++i) {
                    const int32_t sl = ps0 + i < num_pipe ? ps0 + i : ps0 + i - num_pipe;
                    tma_load_2d(ring + static_cast<size_t>(sl) * stage_bytes, mapA, &c->full[sl], (kb0 + i) * kBK, m0,
                                pol_act);
                    ++issued;
                }
                kb_first = kb0 + armed;
            }
            // One loop per stage kind, so the plain loop carries no test for the gated copy.
            auto k_loop = [&](auto gated_kind) {
                constexpr bool kGated = decltype(gated_kind)::value;
                for (int32_t kb = kb_first; kb < kb1; ++kb) {
                    if (leader && kb == lead_kb)
                        mbar_arrive(&c->want_next);
                    if (!wait_bar(&c->empty[ps], pph ^ 1, c, p)) {
                        ok = false;
                        break;
                    }
                    uint8_t *a = ring + static_cast<size_t>(ps) * stage_bytes;
                    mbar_arrive_expect_tx(&c->full[ps], bytes);
                    const int32_t k = kb * kBK;
#pragma unroll
                    for (int32_t u = 0; u < (kGated ? 2 : 1); ++u) {   // gate (or plain) weights, then up
                        const CUtensorMap *mb = u ? mapU : mapB;
                        uint8_t *bt = a + a_bytes + u * b_tile_bytes;
                        if (b_form == 0)
                            tma_load_2d(bt, mb, &c->full[ps], k, by, pol_w);
                        else if (b_form == 1)
                            tma_load_3d(bt, mb, &c->full[ps], 0, k, by, pol_w);
                        else
                            tma_load_2d(bt, mb, &c->full[ps], bx, k, pol_w);
                    }
                    tma_load_2d(a, mapA, &c->full[ps], k, m0, pol_act);
                    ++issued;
                    if (++ps == num_pipe) {
                        ps = 0;
                        pph ^= 1;
                    }
                }
            };
            if (ok) {
                if (gated)
                    k_loop(std::true_type{});
                else
                    k_loop(std::false_type{});
            }
        } else
        for (int32_t kb = kb0; kb < kb1; ++kb) {
            if (leader && kb == lead_kb)
                mbar_arrive(&c->want_next);
            if (!wait_bar(&c->empty[ps], pph ^ 1, c, p)) {
                ok = false;
                break;
            }
            uint8_t *a = ring + static_cast<size_t>(ps) * stage_bytes;
            uint8_t *b = a + a_bytes;
            mbar_arrive_expect_tx(&c->full[ps], bytes);
            // Weights first: they depend on nothing, so in the K-granular mode they are in
            // flight while this k block's producers finish.
            for (int32_t u = 0; u < (gated ? 2 : 1); ++u) {   // gate (or plain) weights, then up
                const CUtensorMap *mb = u ? &p.mapU : mapB;
                uint8_t *bt = b + u * b_tile_bytes;
                if (b_kmajor) {
                    tma_load_2d(bt, mb, &c->full[ps], kb * kBK, n0, pol_w);
                } else if (b_3d) {   // every box of the tile in one copy: (box column, k, box)
                    tma_load_3d(bt, mb, &c->full[ps], 0, kb * kBK, n0 / box_cols, pol_w);
                } else {
                    for (int32_t j = 0; j < nbox; ++j)
                        tma_load_2d(bt + j * box_bytes, mb, &c->full[ps], n0 + j * box_cols, kb * kBK, pol_w);
                }
            }
            if (kwait_s) {
                const int32_t hi = min((kb * kBK + kBK - 1) / pBN, ptn - 1);
                if (hi > ready_hi) {
                    for (int32_t n1 = max(ready_hi + 1, (kb * kBK) / pBN); n1 <= hi && ok; ++n1)
                        ok = wait_producer(p, c, s, pbase + n1);
                    // The acquire fence below is the expensive part (it waits for this SM's
                    // copies in flight), so first take in, without waiting, every later producer
                    // of this slice that is already done: one fence then covers them all.
                    ready_hi = ok ? scan_ready(p, c, s, pbase, hi, slice_last) : hi;
                    fence_acq_rel_gpu();          // acquire the producers' releases ...
                    fence_proxy_async_global();   // ... and order the TMA reads after them
                }
            }
            // (after a failed wait the load still goes out, so that the slot's transaction
            // count completes and the drain below accounts for every copy in flight)
            tma_load_2d(a, mapA, &c->full[ps], kb * kBK, m0, pol_act);
            ++issued;
            if (++ps == num_pipe) {
                ps = 0;
                pph ^= 1;
            }
            if (!ok)
                break;
        }
        free_item_slot(c, slot);
        if (!ok)
            break;
    }
    if (c->abort_flag && !half) {
        // Let every copy this thread issued land before the CTA's shared memory goes away.  A
        // pair's leader waits for both CTAs' copies: the peer fills only phases the leader armed,
        // and keeps its shared memory until the kernel's final cluster barrier.
        const uint32_t np = static_cast<uint32_t>(num_pipe);
        for (uint32_t i = 0; i < np; ++i) {
            const uint32_t fills = issued / np + (i < issued % np ? 1u : 0u);
            if (fills > 0)
                wait_bar(&c->full[i], (fills - 1) & 1, c, p, false);
        }
    }
}

// ------------------------------------------------------------------------------ MMA issuer --
// With a CTA pair the leader issues every MMA (M = 2 bm rows, its TMEM holding the first bm rows
// and the peer's the rest), releases its own ring slots (the TMA role forwards them to the peer)
// and signals both CTAs' accumulator barriers; the peer's MMA thread only walks the item ring.
template <int kPair>
__device__ __forceinline__ void role_mma(const ChainParams &p, Ctrl *c, uint8_t *ring, uint32_t tmem_base)
{
    constexpr bool kPairMode = kPair == 2;
    const uint32_t rank = cluster_ctarank();
    if (kPairMode && (rank & 1u)) {
        for (int32_t it = 0;; ++it) {
            const int32_t slot = it % kSchedDepth;
            if (!wait_bar(&c->sfull[slot], (it / kSchedDepth) & 1, c, p, true, true))
                return;
            if (take_item(c, slot).stage < 0)
                return;
        }
    }
    // the peer's accumulator barriers (shared::cluster), for the leader's second commit
    const uint32_t tfull_peer0 = kPairMode ? map_to_rank(&c->tfull[0], rank | 1u) : 0u;
    const int32_t num_pipe = p.num_pipe;
    const uint32_t stage_bytes = p.stage_bytes;
    const uint32_t acc_stride = static_cast<uint32_t>(p.acc_stride);
    const uint32_t sub_stride = static_cast<uint32_t>(p.sub_stride);
    const bool split2 = p.acc_split == 2;
    const bool lamport = p.pipelined && p.lamport;
    const int32_t bm = p.bm;
    const uint32_t a_bytes = p.a_bytes;
    int32_t ps = 0;
    uint32_t pph = 0;
    uint32_t local_tiles = 0;
    bool issued = false;
    for (int32_t it = 0;; ++it) {
        const int32_t slot = it % kSchedDepth;
        if (!wait_bar(&c->sfull[slot], (it / kSchedDepth) & 1, c, p, true, true))
            break;
        const Item item = take_item(c, slot);
        if (item.stage < 0)
            break;
        if (item.tile < 0)
            continue;
        const StageParams &spr = p.st[item.stage];
        const uint32_t BN = static_cast<uint32_t>(spr.BN);
        const bool gated = spr.gated != 0;
        const bool b_kmajor = spr.b_kmajor != 0;
        const uint32_t b_swz = static_cast<uint32_t>(spr.b_swz);
        int32_t kb0, kb1;
        slice_range(spr.k_blocks, spr.kb_per_split, kslice_of<kPair>(item.split), kb0, kb1);
        const uint32_t acc = local_tiles & 1;
        const uint32_t acc_ph = (local_tiles >> 1) & 1;
        // (a pair's accumulator is released by both CTAs' epilogue warps: remote arrivals)
        if (!wait_bar(&c->tempty[acc], acc_ph ^ 1, c, p, true, kPairMode))
            break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * acc_stride;
        // A gated tile's gate and up weight tiles lie back to back in the slot, laid out exactly
        // like one B tile twice as wide, so one MMA of N = 2 BN fills both accumulators (gate in
        // columns [0, BN), up in [BN, 2 BN)): an MMA costs the same for any N <= 256.
        const uint32_t idesc = idesc_bf16_f32(static_cast<uint32_t>(kPair * bm), gated ? 2u * BN : BN, b_kmajor ? 0u : 1u);
        const uint32_t b_code = b_swz == 128 ? 2u : (b_swz == 64 ? 4u : 6u);
        bool ok = true;
        if (!lamport && !split2) {
            // The common case, kept free of per-k-block branches and address arithmetic: one
            // thread issues this loop back to back, so every instruction in it is on the path.
            // Descriptors are built once for ring slot 0; a slot's (and a 16-deep k step's)
            // offset adds to the 14-bit start-address field in 16-byte units, which cannot
            // carry out of it (shared memory is below 2^18 bytes).
            const uint32_t ring_base = smem_u32(ring);
            const uint64_t ad0 = smem_desc(ring_base, 16u, 1024u, 2u);
            const uint64_t bd0 = b_kmajor ? smem_desc(ring_base + a_bytes, 16u, 1024u, 2u)
                                          : smem_desc(ring_base + a_bytes, kBK * b_swz, 8u * b_swz, b_code);
            const uint64_t bstep = b_kmajor ? 2u : b_swz;   // 16-byte units per 16-deep k step
            const uint64_t slot16 = stage_bytes >> 4;
            uint32_t accum = 0;
            if (spr.kpf == 2) {
                // Two k blocks per fill: A tiles of blocks kb, kb + 1, then their B tiles (role_tma).
                const uint32_t box_cols = b_swz / 2u;
                const uint32_t b_tile = b_kmajor ? static_cast<uint32_t>(kBK) * BN * 2u
                                                 : (BN + box_cols - 1u) / box_cols * static_cast<uint32_t>(kBK) * b_swz;
                const uint64_t bd2 = b_kmajor ? smem_desc(ring_base + 2u * a_bytes, 16u, 1024u, 2u)
                                              : smem_desc(ring_base + 2u * a_bytes, kBK * b_swz, 8u * b_swz, b_code);
                const uint64_t a16 = a_bytes >> 4, b16 = b_tile >> 4;
                for (int32_t kb = kb0; kb < kb1; kb += 2) {
                    if (!wait_bar(&c->full[ps], pph, c, p, true, kPairMode)) {
                        ok = false;
                        break;
                    }
                    const uint64_t off = static_cast<uint64_t>(ps) * slot16;
#pragma unroll
                    for (uint32_t f = 0; f < 2; ++f)
#pragma unroll
                        for (uint32_t kk = 0; kk < kBK / 16; ++kk) {
                            mma_bf16_ss_g<kPair>(d_tmem, ad0 + off + f * a16 + 2u * kk, bd2 + off + f * b16 + bstep * kk,
                                                 idesc, accum);
                            accum = 1u;
                        }
                    issued = true;
                    mma_commit_g<kPair>(smem_u32(&c->empty[ps]));
                    if (++ps == num_pipe) {
                        ps = 0;
                        pph ^= 1;
                    }
                }
            } else
            for (int32_t kb = kb0; kb < kb1; ++kb) {
                // (a pair's fill also completes through the peer's copies: acquire at cluster scope)
                if (!wait_bar(&c->full[ps], pph, c, p, true, kPairMode)) {
                    ok = false;
                    break;
                }
                const uint64_t off = static_cast<uint64_t>(ps) * slot16;
#pragma unroll
                for (uint32_t kk = 0; kk < kBK / 16; ++kk) {
                    mma_bf16_ss_g<kPair>(d_tmem, ad0 + off + 2u * kk, bd0 + off + bstep * kk, idesc, accum);
                    accum = 1u;   // the slice's first k step overwrites the accumulator
                }
                issued = true;
                mma_commit_g<kPair>(smem_u32(&c->empty[ps]));
                if (++ps == num_pipe) {
                    ps = 0;
                    pph ^= 1;
                }
            }
        } else
        for (int32_t kb = kb0; kb < kb1; ++kb) {
            // TMA fills and tcgen05.mma reads are both async-proxy operations ordered by the
            // mbarrier's transaction count: no tcgen05 fence is needed per k block.
            if (!wait_bar(lamport ? &c->valid[ps] : &c->full[ps], pph, c, p)) {
                ok = false;
                break;
            }
            if (lamport)   // the slot reached this thread through warp 3, not through its copies
                tc_fence_after();
            const uint32_t a_addr = smem_u32(ring + static_cast<size_t>(ps) * stage_bytes);
            const uint32_t b_addr = a_addr + a_bytes;
#pragma unroll
            for (uint32_t kk = 0; kk < kBK / 16; ++kk) {
                // A: K-major, 128B swizzle; a 16-wide k step is 32 bytes along the row.
                const uint64_t ad = smem_desc(a_addr + kk * 32u, 16u, 1024u, 2u);
                // B stored K x N: MN-major; a 16-deep k step is 16 rows of b_swz bytes.  LBO: next
                // block of b_swz/2 columns (one TMA box of 64 rows); SBO: next group of 8 rows.
                // B stored N x K: K-major like A, BN rows of 128 bytes.
                const uint64_t bd = b_kmajor ? smem_desc(b_addr + kk * 32u, 16u, 1024u, 2u)
                                             : smem_desc(b_addr + kk * 16u * b_swz, kBK * b_swz, 8u * b_swz, b_code);
                // k step j of the slice goes to sub-accumulator j % acc_split; its first step
                // overwrites.
                const uint32_t j = static_cast<uint32_t>(kb - kb0) * (kBK / 16) + kk;
                const uint32_t sub = split2 ? (j & 1u) : 0u;
                const uint32_t accum = j >= (split2 ? 2u : 1u) ? 1u : 0u;
                mma_bf16_ss_g<kPair>(d_tmem + sub * sub_stride, ad, bd, idesc, accum);
            }
            issued = true;
            mma_commit_g<kPair>(smem_u32(&c->empty[ps]));   // frees the ring slot once these MMAs have read it
            if (++ps == num_pipe) {
                ps = 0;
                pph ^= 1;
            }
        }
        if (!ok)
            break;
        mma_commit_g<kPair>(smem_u32(&c->tfull[acc]));     // accumulator ready for the epilogue
        if (kPairMode)                                       // ... of both CTAs of the pair
            mma_commit_g<kPair>(tfull_peer0 + acc * 8u);
        ++local_tiles;
    }
    if (c->abort_flag && issued) {
        mma_commit_g<kPair>(smem_u32(&c->drain));
        wait_bar(&c->drain, 0, c, p, false);
    }
}

// ------------------------------------------------------------------ Lamport validation --
// The sentinel a Lamport run pre-fills every intermediate with: bf16 -0.0.  Producers of such a
// run write +0.0 for an exact negative zero, so no output value equals it.
constexpr uint32_t kSentinel = 0x8000u;

// True on every lane if any of the bf16 values of the A tile at `a` (a_bytes: 8 or 16 KB) is the
// sentinel.
// A half equals the sentinel exactly when it is zero after an XOR with the sentinel, so the
// scan keeps a running per-half unsigned minimum of w ^ sentinel (two operations per word) and
// tests it once.  Volatile shared loads (the tile is rewritten by TMA between two scans),
// eight in flight before any is used.
__device__ __forceinline__ bool tile_has_sentinel(const uint8_t *a, uint32_t a_bytes, int32_t lane)
{
    const uint32_t base = smem_u32(a) + static_cast<uint32_t>(lane) * 16u;
    const uint32_t flip = kSentinel | (kSentinel << 16);
    uint32_t m = 0xffffffffu;
#pragma unroll 1
    for (int b = 0; b < static_cast<int>(a_bytes / 512); b += 8) {
        uint32_t w[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[i][0]), "=r"(w[i][1]), "=r"(w[i][2]), "=r"(w[i][3])
                         : "r"(base + static_cast<uint32_t>(b + i) * 512u));
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                m = __vminu2(m, w[i][e] ^ flip);
    }
    return __any_sync(0xffffffffu, (m & 0xffffu) == 0u || (m >> 16) == 0u);
}

// Lamport mode only (warp 3, all lanes): the fence-free variant of the protocol (section V,
// Lamport synchronisation).  Producers publish without fences, so a consumer's A tile (the
// previous stage's output) may be read before all of it has landed.  For every k block the MMA
// warp will consume, this warp waits for the slot's copies, scans a consumer stage's A tile for
// the sentinel, re-loads the tile until it holds none (with a deadline), and only then hands the
// slot to the MMA warp through valid[slot].  First-stage tiles read the chain input and pass.
__device__ __forceinline__ void role_validate(const ChainParams &p, Ctrl *c, uint8_t *ring)
{
    const int32_t lane = threadIdx.x & 31;
    const int32_t num_pipe = p.num_pipe;
    const uint32_t stage_bytes = p.stage_bytes;
    const uint64_t pol_act = policy_evict_last();
    int32_t ps = 0;
    uint32_t pph = 0;
    uint32_t rl_phase = 0;     // bit i: parity of reload[i]'s next phase
    uint32_t rl_pending = 0;   // bit i: a reload into slot i is in flight
    bool ok = true;
    for (int32_t it = 0; ok; ++it) {
        const int32_t slot = it % kSchedDepth;
        if (!warp_wait_bar(&c->sfull[slot], (it / kSchedDepth) & 1, c, p, true))
            break;
        Item item{0, 0, 0};
        if (lane == 0)
            item = take_item(c, slot);
        item.stage = __shfl_sync(0xffffffffu, item.stage, 0);
        item.tile = __shfl_sync(0xffffffffu, item.tile, 0);
        item.split = __shfl_sync(0xffffffffu, item.split, 0);
        if (item.stage < 0)
            break;
        if (item.tile < 0)
            continue;
        const int32_t s = item.stage;
        const bool check = s > 0;
        int32_t tile = item.tile;
        if (check) {   // the queue slot names the tile (the TMA warp of this CTA polled it first)
            int32_t t = 0;
            if (lane == 0)
                t = resolve_queue_slot(p, c, s, item.tile, false);
            tile = __shfl_sync(0xffffffffu, t, 0);
            if (tile < 0)
                break;
        }
        const StageParams &spr = p.st[s];
        int32_t kb0, kb1;
        slice_range(spr.k_blocks, spr.kb_per_split, item.split, kb0, kb1);
        const int32_t m0 = (tile / spr.tiles_n) * p.bm;
        for (int32_t kb = kb0; kb < kb1 && ok; ++kb) {
            if (!warp_wait_bar(&c->full[ps], pph, c, p)) {
                ok = false;
                break;
            }
            mbar_try_wait(&c->full[ps], pph);   // every lane acquires the completed phase
            if (check) {
                uint8_t *a = ring + static_cast<size_t>(ps) * stage_bytes;
                bool force = p.force_reload != 0;
                uint64_t t0 = 0;
                while (force || tile_has_sentinel(a, p.a_bytes, lane)) {
                    force = false;
                    const uint64_t now = globaltimer_ns();
                    if (t0 == 0) {
                        t0 = now;
                    } else if (now - t0 > p.timeout_ns) {
                        if (lane == 0) {
                            atomicCAS(p.status, 0u, kStatusTimeout);
                            c->abort_flag = 1;
                        }
                        ok = false;
                        break;
                    }
                    // this warp's reads of the tile come before the copy that overwrites it
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&c->reload[ps], p.a_bytes);
                        tma_load_2d(a, &p.mapA[s], &c->reload[ps], kb * kBK, m0, pol_act);
                    }
                    rl_pending |= 1u << ps;
                    if (!warp_wait_bar(&c->reload[ps], (rl_phase >> ps) & 1u, c, p)) {
                        ok = false;
                        break;
                    }
                    mbar_try_wait(&c->reload[ps], (rl_phase >> ps) & 1u);
                    rl_pending &= ~(1u << ps);
                    rl_phase ^= 1u << ps;
                }
                if (!ok)
                    break;
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&c->valid[ps]);
            if (++ps == num_pipe) {
                ps = 0;
                pph ^= 1;
            }
        }
    }
    // after an abort, a reload still in flight lands before the CTA's shared memory goes away
    if (lane == 0)
        for (int32_t i = 0; i < kMaxPipe; ++i)
            if (rl_pending & (1u << i))
                wait_bar(&c->reload[i], (rl_phase >> i) & 1u, c, p, false);
}

// -------------------------------------------------------------------------------- epilogue --
// Two fp32 values to packed bf16 (lo in the low half), rounded to nearest even by one
// cvt.rn.bf16x2.f32 (its first source fills the upper half); NaN stays a (quiet) NaN.  A
// bit-pattern rounding in integer arithmetic took ten instructions per pair on the epilogue's
// critical path.
__device__ __forceinline__ uint32_t pack_bf16x2_rne(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Byte offset of 16-byte segment `seg` (0..3) of row `row` (0..31) in a warp's staging buffer;
// the XOR keeps the eight rows a quarter-warp touches on distinct banks.
__device__ __forceinline__ uint32_t stage_off(int row, int seg)
{
    return static_cast<uint32_t>(row * 64 + ((seg ^ ((row >> 1) & 3)) * 16));
}

// One warp stores a 32-row x 32-column chunk of the output.  Lane l holds the fp32 values of
// row row0 + l (TMEM hands each thread one row); the chunk goes through the warp's staging
// buffer so that global stores and residual loads touch whole 64-byte row segments.
// Output of a stage, copied into registers once per tile.
struct OutDesc {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *residual;
    int32_t M, N, gelu;
    int32_t canon;   // Lamport producer: store +0.0 for -0.0, so no output equals the sentinel
};

// Both bf16 halves of w with -0.0 replaced by +0.0.
__device__ __forceinline__ uint32_t canon_neg_zero(uint32_t w)
{
    if ((w & 0xffffu) == 0x8000u)
        w &= 0xffff0000u;
    if ((w >> 16) == 0x8000u)
        w &= 0x0000ffffu;
    return w;
}

// Rows row0 .. row_lim - 1 are stored (row_lim <= M; a warp of a 64-row tile holds 16 rows).
template <bool kGelu>
__device__ __forceinline__ void store_chunk_warp_t(const OutDesc sp, int32_t row0, int32_t row_lim, int32_t n,
                                                   const uint32_t (&r)[32], uint8_t *stage, int32_t lane)
{
    float v[32];
#pragma unroll
    for (int e = 0; e < 32; ++e)
        v[e] = __uint_as_float(r[e]);
    if (kGelu) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
            v[e] = gelu_tanh_f32(v[e]);
    }
    if (sp.residual) {
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int rr = it * 8 + (lane >> 2), sg = lane & 3;
            const int32_t gm = row0 + rr, gn = n + sg * 8;
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (gm < row_lim && gn < sp.N)
                x = *reinterpret_cast<const uint4 *>(sp.residual + static_cast<size_t>(gm) * sp.N + gn);
            *reinterpret_cast<uint4 *>(stage + stage_off(rr, sg)) = x;
        }
        __syncwarp();
#pragma unroll
        for (int sg = 0; sg < 4; ++sg) {
            const uint4 x = *reinterpret_cast<const uint4 *>(stage + stage_off(lane, sg));
            const __nv_bfloat162 *xb = reinterpret_cast<const __nv_bfloat162 *>(&x);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(xb[e]);
                v[sg * 8 + 2 * e] += f.x;
                v[sg * 8 + 2 * e + 1] += f.y;
            }
        }
        __syncwarp();
    }
#pragma unroll
    for (int sg = 0; sg < 4; ++sg) {
        uint4 o = make_uint4(pack_bf16x2_rne(v[sg * 8], v[sg * 8 + 1]), pack_bf16x2_rne(v[sg * 8 + 2], v[sg * 8 + 3]),
                             pack_bf16x2_rne(v[sg * 8 + 4], v[sg * 8 + 5]), pack_bf16x2_rne(v[sg * 8 + 6], v[sg * 8 + 7]));
        if (sp.canon) {
            o.x = canon_neg_zero(o.x);
            o.y = canon_neg_zero(o.y);
            o.z = canon_neg_zero(o.z);
            o.w = canon_neg_zero(o.w);
        }
        *reinterpret_cast<uint4 *>(stage + stage_off(lane, sg)) = o;
    }
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int rr = it * 8 + (lane >> 2), sg = lane & 3;
        const int32_t gm = row0 + rr, gn = n + sg * 8;
        if (gm < row_lim && gn < sp.N)   // N is a multiple of 8: a segment is all in or all out
            *reinterpret_cast<uint4 *>(sp.out + static_cast<size_t>(gm) * sp.N + gn) =
                *reinterpret_cast<const uint4 *>(stage + stage_off(rr, sg));
    }
    __syncwarp();
}

// GeLU is chosen once per call by a uniform branch, so the plain path carries no tanh code
// (a per-element test inside the unrolled loop could be if-converted into evaluating it always).
__device__ __forceinline__ void store_chunk_warp(const OutDesc sp, int32_t row0, int32_t row_lim, int32_t n,
                                                 const uint32_t (&r)[32], uint8_t *stage, int32_t lane)
{
    if (sp.gelu)
        store_chunk_warp_t<true>(sp, row0, row_lim, n, r, stage, lane);
    else
        store_chunk_warp_t<false>(sp, row0, row_lim, n, r, stage, lane);
}

// 32 accumulator columns of this thread's TMEM lane (sub-accumulators summed, even + odd).
__device__ __forceinline__ void load_acc(bool split2, uint32_t sub_stride, uint32_t taddr, uint32_t (&r)[32])
{
    tmem_ld_32x32b_x32(taddr, r);
    if (split2) {
        uint32_t r2[32];
        tmem_ld_32x32b_x32(taddr + sub_stride, r2);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e)
            r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(r2[e]));
    } else {
        tmem_ld_wait();
    }
}

// What the release of one producer tile reads from the dependency tables, loaded while the
// tile's mainloop still runs so that the release itself is one atomic add, one queue reservation
// and the stores.  Filled in full when the tile feeds exactly one group (a GEMM chain's row
// panel); `ne` is the number of groups it feeds.  Lane i holds members i and 32 + i.
struct ReleasePlan {
    int32_t ne, g, init, m0, n, mem0, mem1;
};

__device__ __forceinline__ ReleasePlan plan_release(const ChainParams &p, int32_t s, int32_t tile, int32_t lane)
{
    const BoundaryParams &bd = p.bd[s];
    ReleasePlan r{0, -1, 0, 0, 0, -1, -1};
    const int32_t e0 = bd.pg_off[tile];
    r.ne = bd.pg_off[tile + 1] - e0;
    if (r.ne == 1) {
        r.g = bd.pg_tgt[e0];
        r.init = bd.grp_init[r.g];
        r.m0 = bd.grp_off[r.g];
        r.n = bd.grp_off[r.g + 1] - r.m0;
        if (lane < r.n)
            r.mem0 = bd.grp_mem[r.m0 + lane];
        if (lane + 32 < r.n)
            r.mem1 = bd.grp_mem[r.m0 + 32 + lane];
    }
    return r;
}

// Producer side of the protocol for the rows one epilogue warp stored of a finished tile (or of
// one split-K slice of it): count one release on every group counter the tile feeds.  A group
// waits for grp_init = producer tiles x S x kEpiWarps releases per run; counters accumulate over
// the handle's runs, so run e is complete at grp_init x (e + 1) and nothing is re-armed.  The
// add that completes the count publishes the group's members on the work-queue.  Called by the
// whole warp right after a fence.acq_rel.gpu that follows its stores.
__device__ __forceinline__ void release_tile(const ChainParams &p, Ctrl *c, int32_t s, int32_t tile, int32_t lane,
                                             const ReleasePlan &pl)
{
    const BoundaryParams &bd = p.bd[s];
    if (bd.queue_free) {   // the caller's fence and these relaxed adds are the release; no push
        if (pl.ne == 1) {
            if (lane == 0)
                red_add_relaxed_gpu(bd.count + pl.g, 1u);
        } else {
            for (int32_t e = bd.pg_off[tile] + lane; e < bd.pg_off[tile + 1]; e += 32)
                red_add_relaxed_gpu(bd.count + bd.pg_tgt[e], 1u);
        }
        return;
    }
    if (pl.ne == 1) {
        // One group: lane 0 counts this release (the caller's fence and this relaxed add are the
        // release); the add that completes the run's count reserves the group's queue slots.
        uint32_t q0 = 0, fire = 0;
        if (lane == 0) {
            const uint32_t old = atom_add_relaxed_gpu(bd.count + pl.g, 1u);
            if (release_completes(old, run_target(pl.init, c->epoch))) {
                fire = 1;
                q0 = run_relative(atom_add_relaxed_gpu(bd.tail, static_cast<uint32_t>(pl.n)), c->epoch,
                                  bd.slots_per_run);
            }
        }
        if (!__shfl_sync(0xffffffffu, fire, 0))
            return;
        q0 = __shfl_sync(0xffffffffu, q0, 0);
        // No fence: a consumer that finds its entry acquires the group counter before it reads
        // a byte of the producers' output (resolve_queue_slot).
        if (lane < pl.n)
            st_relaxed_gpu_u64(bd.queue + q0 + lane, queue_entry(c->epoch, pl.mem0));
        if (lane + 32 < pl.n)
            st_relaxed_gpu_u64(bd.queue + q0 + 32 + lane, queue_entry(c->epoch, pl.mem1));
        for (int32_t i = lane + 64; i < pl.n; i += 32)
            st_relaxed_gpu_u64(bd.queue + q0 + i, queue_entry(c->epoch, bd.grp_mem[pl.m0 + i]));
        return;
    }
    const int32_t e0 = bd.pg_off[tile], e1 = bd.pg_off[tile + 1];
    for (int32_t eb = e0; eb < e1; eb += 32) {
        const int32_t e = eb + lane;
        int32_t g = -1;
        bool fire = false;
        if (e < e1) {
            g = bd.pg_tgt[e];
            // The caller's fence.acq_rel.gpu and this relaxed add form the release of the warp's
            // stores; consumers acquire them through the counter.
            const uint32_t old = atom_add_relaxed_gpu(bd.count + g, 1u);
            fire = release_completes(old, run_target(bd.grp_init[g], c->epoch));
        }
        // Every group this warp completed is published by the whole warp with relaxed stores (the
        // consumers' acquire is on the group counter, see resolve_queue_slot).
        uint32_t todo = __ballot_sync(0xffffffffu, fire);
        while (todo) {
            const int32_t src = __ffs(todo) - 1;
            todo &= todo - 1;
            const int32_t gg = __shfl_sync(0xffffffffu, g, src);
            const int32_t m0 = bd.grp_off[gg], n = bd.grp_off[gg + 1] - m0;
            uint32_t q0 = 0;
            if (lane == src)
                q0 = run_relative(atom_add_relaxed_gpu(bd.tail, static_cast<uint32_t>(n)), c->epoch, bd.slots_per_run);
            q0 = __shfl_sync(0xffffffffu, q0, src);
            for (int32_t i = lane; i < n; i += 32)
                st_relaxed_gpu_u64(bd.queue + q0 + i, queue_entry(c->epoch, bd.grp_mem[m0 + i]));
        }
    }
}

__device__ __forceinline__ void log_end(const ChainParams &p, int32_t s, int32_t tile)
{
    EventRec *e = p.events + p.tile_base[s] + tile;
    e->seq_end = atom_add_relaxed_gpu(p.seq, 1u);
    e->t_end = globaltimer_ns();
}

// Injected epilogue of a finished tile or split-K slice, run by each epilogue warp for the 32
// rows it stored.  The caller has fenced the warp's stores at gpu scope (after the warp's last
// __syncwarp, so the fence is cumulative over all its lanes); that fence and the relaxed add in
// release_tile form the release.  Each of the four warps of each of the S slices releases once
// (a group counts producer tiles x S x 4 releases per run), so no warp waits for another.
__device__ __forceinline__ void publish(const ChainParams &p, Ctrl *c, int32_t s, int32_t tile, bool log_it,
                                        bool producer, int32_t warp, int32_t lane, const ReleasePlan &pl)
{
    if (log_it && warp == 4 && lane == 0)
        log_end(p, s, tile);
    __syncwarp();
    if (!producer || (s == 0 && tile == p.drop_tile))
        return;
    if (p.kwait) {   // K-granular mode: count this warp's release on the producer tile itself
        if (lane == 0)
            red_add_relaxed_gpu(p.bd[s].ready + tile, 1u);
        return;
    }
    release_tile(p, c, s, tile, lane, pl);
}

// With a CTA pair each CTA stores the rows its TMEM holds (the leader the tile's first bm rows, the
// peer the rest) and releases them; the accumulator goes back to the leader's MMA thread through
// the leader's tempty barrier, which counts both CTAs' epilogue warps.
template <int kPair>
__device__ __forceinline__ void role_epilogue(const ChainParams &p, Ctrl *c, uint32_t tmem_base, uint32_t rank,
                                              uint8_t *staging, uint8_t *recv)
{
    constexpr bool kPairMode = kPair == 2;
    const int32_t half = kPairMode ? static_cast<int32_t>(rank & 1u) : 0;
    const uint32_t tempty_lead0 = kPairMode ? map_to_rank(&c->tempty[0], rank & ~1u) : 0u;
    const uint32_t recv_u32 = smem_u32(recv);
    const int32_t warp = threadIdx.x / 32;
    const int32_t lane = threadIdx.x & 31;
    const int32_t quad = warp & 3;              // TMEM lanes 32*quad .. 32*quad+31
    // Accumulator rows of this warp's TMEM sub-partition: with M = 128 lane l of sub-partition q
    // holds row 32q + l; with M = 64 its first 16 lanes hold rows 16q .. 16q+15 (the tcgen05
    // data-path layout of a 64-row MMA) and lanes 16 .. 31 hold nothing.
    const int32_t bm = p.bm;
    const int32_t rpw = bm / 4;                 // rows per warp
    const int32_t row = quad * rpw + lane;      // this lane's row of the tile (valid if lane < rpw)
    const bool row_ok = lane < rpw;
    uint8_t *stage = staging + quad * kEpiStageBytes;
    // kernel-uniform parameters in registers (see role_tma)
    const uint32_t acc_stride = static_cast<uint32_t>(p.acc_stride);
    const uint32_t sub_stride = static_cast<uint32_t>(p.sub_stride);
    const bool split2 = p.acc_split == 2;
    const int32_t cs = p.cs;
    const size_t partial_floats = static_cast<size_t>(p.partial_floats);
    const bool pipelined = p.pipelined != 0;
    const bool kwait = pipelined && p.kwait != 0;
    const bool lamport = pipelined && p.lamport != 0;
    const int32_t num_stages = p.num_stages;
    const bool logging = p.events != nullptr;
    const size_t cbase = static_cast<size_t>(cluster_id_x()) * cs;
    uint32_t local_tiles = 0;
    uint32_t nsplit = 0;                        // split-K tiles this CTA took part in
    bool have_epoch = false;
    for (int32_t it = 0;; ++it) {
        const int32_t slot = it % kSchedDepth;
        if (!warp_wait_bar(&c->sfull[slot], (it / kSchedDepth) & 1, c, p, true))
            break;
        Item item{0, 0, 0};
        if (lane == 0)
            item = take_item(c, slot);
        item.stage = __shfl_sync(0xffffffffu, item.stage, 0);
        item.tile = __shfl_sync(0xffffffffu, item.tile, 0);
        item.split = __shfl_sync(0xffffffffu, item.split, 0);
        if (item.stage < 0)
            break;
        if (item.tile < 0)
            continue;
        const int32_t s = item.stage;
        int32_t tile = item.tile;
        if (pipelined && !have_epoch) {   // queue slots, releases and pushes carry the run's epoch
            if (!warp_wait_bar_all(&c->epoch_bar, 0, c, p))
                break;
            have_epoch = true;
        }
        if (pipelined && s > 0 && !kwait) {   // the TMA warp of this CTA polled the same slot first
            int32_t t = 0;
            if (lane == 0)
                t = resolve_queue_slot(p, c, s, item.tile, false);   // reads no producer data
            tile = __shfl_sync(0xffffffffu, t, 0);
            if (tile < 0)
                break;
        }
        const StageParams &spr = p.st[s];
        const int32_t BN = spr.BN, tiles_n = spr.tiles_n, S = kPairMode ? spr.split / 2 : spr.split;   // k-slices
        const bool dsmem = spr.dsmem_reduce != 0;
        float *const partials = spr.partials;
        const bool producer = pipelined && s + 1 < num_stages;
        const OutDesc od{spr.out, spr.residual, spr.M, spr.N, spr.gelu, lamport && producer};
        const uint32_t acc = local_tiles & 1;
        const uint32_t acc_ph = (local_tiles >> 1) & 1;
        ReleasePlan pl{0, -1, 0, 0, 0, -1, -1};
        if (producer && !kwait)
            pl = plan_release(p, s, tile, lane);
        if (!warp_wait_bar(&c->tfull[acc], acc_ph, c, p, kPairMode))   // (a pair's: the leader's commit)
            break;
        tc_fence_after();
        if (logging && warp == 4 && lane == 0 && item.split == 0)
            p.events[p.tile_base[s] + tile].t_acc = globaltimer_ns();
        const int32_t row0 = (tile / tiles_n) * (kPair * bm) + half * bm + quad * rpw;   // this warp's first row
        const int32_t row_lim = min(spr.M, row0 + rpw);
        const int32_t n0 = (tile % tiles_n) * BN;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * acc_stride;

        if (S == 1) {
            for (int32_t c0 = 0; c0 < BN; c0 += 32) {
                uint32_t r[32];
                load_acc(split2, sub_stride, taddr + c0, r);
                if (spr.gated) {   // SwiGLU: SiLU(gate) * up, both fp32, rounded once below
                    uint32_t u[32];
                    tmem_ld_32x32b_x32(taddr + BN + c0, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float g = __uint_as_float(r[e]);
                        r[e] = __float_as_uint(__fdividef(g, 1.0f + __expf(-g)) * __uint_as_float(u[e]));
                    }
                }
                store_chunk_warp(od, row0, row_lim, n0 + c0, r, stage, lane);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {   // the MMA warp may reuse this accumulator
                if (kPairMode)
                    mbar_arrive_cluster(tempty_lead0 + acc * 8u);
                else
                    mbar_arrive(&c->tempty[acc]);
            }
            ++local_tiles;
            if (producer || (pipelined && logging)) {
                if (!lamport)   // this warp's stores, released at gpu scope for the consumers
                    fence_acq_rel_gpu();
                publish(p, c, s, tile, logging && half == 0, producer, warp, lane, pl);
            }
            continue;
        }

        // ---- split-K tile: S siblings each hold a k-slice partial of the same rows: ranks
        // g0 .. g0+S-1, or with CTA pairs the same half of each slice's pair, g0 + 2 q + half ----
        const uint32_t g0 = rank - static_cast<uint32_t>(item.split);      // the tile's first rank
        const uint32_t weight = static_cast<uint32_t>(cs / S);             // arrivals per sibling warp
        const int32_t ks = kslice_of<kPair>(item.split);                   // my k-slice
        auto sibling = [&](int32_t q) {
            return g0 + static_cast<uint32_t>(kPairMode ? 2 * q + half : q);
        };
        if (spr.xsplit) {
            // The slices run on separate clusters.  Each keeps its partial in a buffer of its own
            // (tile, slice, half), written once per run, so no sibling waits before overwriting
            // one; the same halves of the tile's slices count their releases on one counter.
            // Layout and order of the sum as below.
            const size_t tile_buf = static_cast<size_t>(tile) * S * kPair;
            auto buf = [&](int32_t q) { return partials + (tile_buf + static_cast<size_t>(q) * kPair + half) * partial_floats; };
            const int32_t slice = BN / S;
            const int32_t col0 = ks * slice;
            float *mine = buf(ks);
            for (int32_t c0 = 0; c0 < BN; c0 += 32) {
                if (c0 >= col0 && c0 < col0 + slice)
                    continue;
                uint32_t r[32];
                load_acc(split2, sub_stride, taddr + c0, r);
                float4 *dst = reinterpret_cast<float4 *>(mine) + (c0 / 32) * 8 * bm + row;
                if (row_ok)
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        dst[v * bm] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                                  __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
            }
            fence_acq_rel_gpu();   // these stores, released at gpu scope by the add below
            __syncwarp();
            uint32_t *cnt = spr.xcount + static_cast<size_t>(tile) * kPair + half;
            uint32_t ok = 1;
            if (lane == 0) {
                red_add_relaxed_gpu(cnt, 1u);
                // every epilogue warp of every slice of this half: S x kEpiWarps releases per run
                const uint32_t want = run_target(S * kEpiWarps, c->epoch);
                const uint64_t t0 = globaltimer_ns();
                while (!count_reached(ld_acquire_gpu_u32(cnt), want)) {
                    if (c->abort_flag || globaltimer_ns() - t0 > p.timeout_ns) {
                        if (!c->abort_flag)
                            atomicCAS(p.status, 0u, kStatusTimeout);
                        c->abort_flag = 1;
                        ok = 0;
                        break;
                    }
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0))
                break;
            for (int32_t c0 = col0; c0 < col0 + slice; c0 += 32) {
                uint32_t own[32];
                load_acc(split2, sub_stride, taddr + c0, own);
                float acc_v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    acc_v[e] = 0.0f;
                const size_t off = static_cast<size_t>((c0 / 32) * 8 * bm + row);   // in float4
                for (int32_t q = 0; q < S && row_ok; ++q) {
                    if (q == ks) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            acc_v[e] += __uint_as_float(own[e]);
                        continue;
                    }
                    const float4 *src = reinterpret_cast<const float4 *>(buf(q)) + off;
                    float4 v[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        v[i] = __ldcg(src + i * bm);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        acc_v[4 * i] += v[i].x;
                        acc_v[4 * i + 1] += v[i].y;
                        acc_v[4 * i + 2] += v[i].z;
                        acc_v[4 * i + 3] += v[i].w;
                    }
                }
                uint32_t r[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    r[e] = __float_as_uint(acc_v[e]);
                store_chunk_warp(od, row0, row_lim, n0 + c0, r, stage, lane);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {   // the MMA warp may reuse this accumulator
                if (kPairMode)
                    mbar_arrive_cluster(tempty_lead0 + acc * 8u);
                else
                    mbar_arrive(&c->tempty[acc]);
            }
            ++local_tiles;
            fence_acq_rel_gpu();   // the slice stores, released at gpu scope for the consumers
            __syncwarp();
            if (producer || (pipelined && logging))
                publish(p, c, s, tile, logging && item.split == 0, producer, warp, lane, pl);
            continue;
        }
        if (dsmem && !kPairMode) {
            // Sibling q owns columns [q*BN/S, (q+1)*BN/S).  Every CTA sends each owner its part of
            // that slice straight from TMEM into the owner's receive buffer, laid out
            // [source split][chunk of the slice][vector][128 rows][4 floats] (a warp writes 512
            // contiguous bytes), then the owner adds the S parts in source order.
            const int32_t cpo = BN / S / 32;   // 32-column chunks per owner
            if (nsplit > 0 && !warp_wait_bar(&c->done_bar, (nsplit - 1) & 1, c, p, true))
                break;   // every owner has finished reading its buffer from the previous tile
            for (int32_t ch = 0; ch < BN / 32; ++ch) {
                uint32_t r[32];
                load_acc(split2, sub_stride, taddr + ch * 32, r);
                const int32_t owner = ch / cpo, oc = ch % cpo;
                const uint32_t dst = map_to_rank(recv, g0 + owner) +
                                     static_cast<uint32_t>((((item.split * cpo + oc) * 8) * bm + row) * 16);
                if (row_ok)
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        st_cluster_v4_f32(dst + v * bm * 16, __uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                          __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&c->tempty[acc]);
            ++local_tiles;
            fence_acq_rel_cluster();
            __syncwarp();
            if (lane == 0)
                for (int32_t q = 0; q < S; ++q)
                    arrive_rank_relaxed(&c->red_bar, g0 + q, weight);
            if (!warp_wait_bar(&c->red_bar, nsplit & 1, c, p, true))
                break;
            for (int32_t oc = 0; oc < cpo; ++oc) {
                float acc_v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    acc_v[e] = 0.0f;
                for (int32_t q = 0; q < S && row_ok; ++q) {
                    const uint32_t src = recv_u32 + static_cast<uint32_t>((((q * cpo + oc) * 8) * bm + row) * 16);
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        const float4 x = ld_shared_v4_f32(src + v * bm * 16);
                        acc_v[4 * v] += x.x;
                        acc_v[4 * v + 1] += x.y;
                        acc_v[4 * v + 2] += x.z;
                        acc_v[4 * v + 3] += x.w;
                    }
                }
                uint32_t r[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    r[e] = __float_as_uint(acc_v[e]);
                store_chunk_warp(od, row0, row_lim, n0 + (item.split * cpo + oc) * 32, r, stage, lane);
            }
            if (lamport)           // (a Lamport run publishes the slice without a release)
                fence_acq_rel_cluster();
            else                   // the slice stores, released at gpu scope for the consumers
                fence_acq_rel_gpu();
            __syncwarp();
            if (lane == 0)         // my receive buffer is read: siblings may send the next tile
                for (int32_t q = 0; q < S; ++q)
                    arrive_rank_relaxed(&c->done_bar, g0 + q, weight);
            ++nsplit;
            // Each sibling publishes its own column slice; the tile's consumers wait for all S.
            if (producer || (pipelined && logging))
                publish(p, c, s, tile, logging && item.split == 0, producer, warp, lane, pl);
            continue;
        }
        // Through global memory.  Partial layout: [BN/32 chunks][8 vectors][bm rows][4 floats]:
        // for a fixed vector the warp's lanes (rows) touch 512 contiguous bytes, so stores and
        // loads coalesce.  Only the chunks other siblings own are written; my own column slice
        // stays in TMEM until I have added the S parts, so the accumulator is handed back to the
        // MMA warp after the reduction.
        float *mine = partials + (cbase + rank) * partial_floats;
        const int32_t slice = BN / S;
        const int32_t col0 = ks * slice;
        // my previous partial must have been read by every sibling of that tile
        if (nsplit > 0 && !warp_wait_bar(&c->done_bar, (nsplit - 1) & 1, c, p, true))
            break;
        for (int32_t c0 = 0; c0 < BN; c0 += 32) {
            if (c0 >= col0 && c0 < col0 + slice)
                continue;
            uint32_t r[32];
            load_acc(split2, sub_stride, taddr + c0, r);
            float4 *dst = reinterpret_cast<float4 *>(mine) + (c0 / 32) * 8 * bm + row;
            if (row_ok)
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    dst[v * bm] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                              __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
        }
        fence_acq_rel_cluster();
        __syncwarp();
        if (lane == 0)
            for (int32_t q = 0; q < S; ++q)
                arrive_rank_relaxed(&c->red_bar, sibling(q), weight);
        if (!warp_wait_bar(&c->red_bar, nsplit & 1, c, p, true))
            break;
        // Reduce my column slice over the S partials in sibling order (mine from TMEM), then the
        // epilogue.  Loads of two partials are issued before either is added.
        for (int32_t c0 = col0; c0 < col0 + slice; c0 += 32) {
            uint32_t own[32];
            load_acc(split2, sub_stride, taddr + c0, own);
            float acc_v[32];
#pragma unroll
            for (int e = 0; e < 32; ++e)
                acc_v[e] = 0.0f;
            const size_t off = static_cast<size_t>((c0 / 32) * 8 * bm + row);   // in float4
            for (int32_t qb = 0; qb < S && row_ok; qb += 2) {
                float4 v[2][8];
#pragma unroll
                for (int qq = 0; qq < 2; ++qq)
                    if (qb + qq < S && qb + qq != ks) {
                        const float4 *src =
                            reinterpret_cast<const float4 *>(partials + (cbase + sibling(qb + qq)) * partial_floats) + off;
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            v[qq][i] = __ldcg(src + i * bm);
                    }
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    if (qb + qq >= S)
                        continue;
                    if (qb + qq == ks) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            acc_v[e] += __uint_as_float(own[e]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            acc_v[4 * i] += v[qq][i].x;
                            acc_v[4 * i + 1] += v[qq][i].y;
                            acc_v[4 * i + 2] += v[qq][i].z;
                            acc_v[4 * i + 3] += v[qq][i].w;
                        }
                    }
                }
            }
            uint32_t r[32];
#pragma unroll
            for (int e = 0; e < 32; ++e)
                r[e] = __float_as_uint(acc_v[e]);
            store_chunk_warp(od, row0, row_lim, n0 + c0, r, stage, lane);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {   // the MMA warp may reuse this accumulator
            if (kPairMode)
                mbar_arrive_cluster(tempty_lead0 + acc * 8u);
            else
                mbar_arrive(&c->tempty[acc]);
        }
        ++local_tiles;
        if (lamport)
            fence_acq_rel_cluster();
        else                   // the slice stores, released at gpu scope for the consumers
            fence_acq_rel_gpu();
        __syncwarp();
        if (lane == 0)         // the siblings' partials are read: they may overwrite them
            for (int32_t q = 0; q < S; ++q)
                arrive_rank_relaxed(&c->done_bar, sibling(q), weight);
        ++nsplit;
        if (producer || (pipelined && logging))
            publish(p, c, s, tile, logging && item.split == 0, producer, warp, lane, pl);
    }
}

// ------------------------------------------------------------------------------ the kernel --
// kPair = 1: one CTA per tile (tcgen05 cta_group::1).  kPair = 2: clusters of CTA pairs, each pair
// computing 2 bm-row tiles with cta_group::2 MMAs (every tcgen05 allocation, MMA and commit of a
// kernel uses one CTA group, hence two instantiations).
template <int kPair>
__global__ void __launch_bounds__(kThreads, 1) chain_kernel(const __grid_constant__ ChainParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + (((base + 1023u) & ~1023u) - base);
    Ctrl *c = reinterpret_cast<Ctrl *>(ring + ctrl_offset(p.num_pipe, p.stage_bytes, p.recv_bytes));
    const int32_t warp = threadIdx.x / 32;
    const int32_t lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    // a pipelined run's event log also records each CTA's lifetime: entry, set-up done, exit
    EventRec *const cta_rec = (p.pipelined && p.events) ? p.events + p.tile_base[p.num_stages] + blockIdx.x : nullptr;
    if (cta_rec && threadIdx.x == 0)
        cta_rec->t_start = globaltimer_ns();

    if (warp == 3 && lane == 0) {   // (otherwise idle now) the tensor maps, while warp 0 sets up
        for (int i = 0; i < p.num_stages; ++i) {
            prefetch_tensormap(&p.mapA[i]);
            prefetch_tensormap(&p.mapB[i]);
        }
        if (p.st[0].gated)
            prefetch_tensormap(&p.mapU);
    }
    if (warp == 0) {
        // The status read goes out first, so its latency overlaps the barrier set-up below; the
        // warp's lanes initialise the ring's barriers side by side.
        const uint32_t status0 = lane == 0 ? ld_relaxed_gpu_u32(p.status) : 0u;
        for (int i = lane; i < p.num_pipe; i += 32) {
            mbar_init(&c->full[i], 1);
            mbar_init(&c->empty[i], 1);
            mbar_init(&c->valid[i], 1);
            mbar_init(&c->reload[i], 1);
        }
        if (lane < 2) {
            mbar_init(&c->tfull[lane], 1);
            mbar_init(&c->tempty[lane], 4 * kPair);   // a pair's: both CTAs' epilogue warps
        }
        for (int i = lane; i < kSchedDepth; i += 32) {
            mbar_init(&c->sfull[i], 1);
            // TMA + MMA + 4 epilogue warps of every rank (+ the Lamport validator)
            mbar_init(&c->sempty[i], (p.pipelined && p.lamport ? 7 : 6) * p.cs);
        }
        if (lane == 2) {
            mbar_init(&c->drain, 1);
            mbar_init(&c->want_next, 1);
            mbar_init(&c->red_bar, 4 * p.cs);          // 4 warps x S siblings, each arriving cs/S times
            mbar_init(&c->done_bar, 4 * p.cs);
            mbar_init(&c->epoch_bar, 1);
        }
        if (lane == 0) {
            // the cluster's first item needs no ticket and no broadcast: write it into slot 0 here
            int32_t ntiles = 0, slice = -1;
            int32_t tiles[kMaxCluster];
            const int32_t stage = item_tiles(p, static_cast<int32_t>(cluster_id_x()), ntiles, tiles, slice);
            int32_t tile0, split0;
            item_member(p, stage, ntiles, tiles, slice, stage >= 0 ? p.st[stage].split : 1, static_cast<int32_t>(rank),
                        tile0, split0);
            c->item_stage[0] = stage;
            c->item_tile[0] = tile0;
            c->item_split[0] = split0;
            c->abort_flag = 0;
            c->skip = status0 != 0;   // sticky error: do nothing
            c->epoch = 0;
        }
        fence_barrier_init();   // (each lane orders its own initialisations)
        if (lane == 0)
            mbar_arrive(&c->sfull[0]);   // item 0 is in place (a local arrival, before any remote one)
    }
    if (warp == 1) {
        tmem_alloc_g<kPair>(&c->tmem_base, p.tmem_cols);   // with a pair: one warp in each CTA, together
        tmem_relinquish_g<kPair>();
    }
    tc_fence_before();
    cluster_sync_all();   // every barrier of the cluster is initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = c->tmem_base;
    if (cta_rec && threadIdx.x == 0)
        cta_rec->t_acc = globaltimer_ns();
    if (p.pdl_trigger && threadIdx.x == 0)
        griddep_launch_dependents();   // the next GEMM's CTAs may take SMs as this grid's retire

    if (!c->skip) {
        if (warp == 0) {
            if (lane == 0)
                role_tma<kPair>(p, c, ring, rank == 0);
        } else if (warp == 1) {
            if (lane == 0)
                role_mma<kPair>(p, c, ring, tmem_base);
            __syncwarp();
        } else if (warp == 2) {
            if (lane == 0 && rank == 0)
                role_scheduler(p, c);
        } else if (warp == 3) {
            // The run's epoch, from the launch counter every CTA adds 1 to (protocol.h): taken
            // here, after the set-up, so its round trip delays no first load; every role that
            // needs it waits for epoch_bar first.
            if (lane == 0) {
                if (p.pipelined)
                    c->epoch = epoch_of_launch(atom_add_relaxed_gpu_u64(p.launches, 1ull), gridDim.x);
                mbar_arrive(&c->epoch_bar);
            }
            // The protocol's few kilobytes of state are cold after whatever ran before (the
            // release and the consumer prologue would each pay HBM misses in sequence), so the
            // otherwise idle warp pulls them into L2 now, spread over the grid.
            const uint32_t step = gridDim.x * 32u * 128u;
            for (uint32_t off = (blockIdx.x * 32u + static_cast<uint32_t>(lane)) * 128u; off < p.meta_bytes; off += step)
                prefetch_l2_keep(p.meta + off);
            if (p.pipelined && p.lamport)
                role_validate(p, c, ring);
        } else if (warp >= 4) {
            role_epilogue<kPair>(p, c, tmem_base, rank, ring + staging_offset(p.num_pipe, p.stage_bytes),
                          ring + recv_offset(p.num_pipe, p.stage_bytes));
        }
    }
    tc_fence_before();
    // A pair frees its TMEM together, and only once the leader's MMAs (which write the peer's
    // TMEM) and both CTAs' epilogues are done.
    if constexpr (kPair == 2)
        cluster_sync_all();
    else
        __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_g<kPair>(tmem_base, p.tmem_cols);
    }
    // Nothing is reset for the next run: scoreboard counters, the ticket, the queue tails and the
    // launch counter all accumulate over runs (protocol.h), and queue slots carry the run's epoch.
    cluster_sync_all();   // no CTA leaves while a peer may still write to its shared memory
    if (cta_rec && threadIdx.x == 0) {
        cta_rec->stage = -1;
        cta_rec->tile = static_cast<int32_t>(blockIdx.x);
        cta_rec->smid = static_cast<int32_t>(smid());
        cta_rec->cta = static_cast<int32_t>(blockIdx.x);
        cta_rec->t_end = globaltimer_ns();
    }
}

}  // namespace mlpc
