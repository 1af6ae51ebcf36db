// chain_kernel.cuh -- the persistent, warp-specialised tcgen05 kernel that runs a GEMM chain
// with the CTA-pipelining protocol of "CTA-Pipelining: A Latency-Oriented Spatial Scaling
// Method for Multi-GPU Systems" (arXiv 2607.07862).
//
// Warp roles (256 threads, one CTA per SM):
//   warp 0      TMA producer: streams A (activations, K-major) and B (weights, MN-major) tiles
//               into an NS-deep shared-memory ring.
//   warp 1      MMA issuer: one thread issues tcgen05.mma into a double-buffered TMEM
//               accumulator; warp 1 also owns the TMEM allocation.
//   warp 2      scheduler: takes tickets and, for consumer stages, polls the work-queue (the
//               injected prologue of section III-A, Fig. 1; "fetch the work-queue value and
//               broadcast it" of section III-C, Fig. 2b, here a shared-memory ring + mbarrier).
//   warps 4-7   epilogue: TMEM -> registers -> (GeLU) -> bf16 -> global, then the injected
//               epilogue: fence, scoreboard decrements and queue pushes (section III-A; the
//               fence placement follows the memory-consistency discussion of section V).
// Because the scheduler and epilogue warps would otherwise wait at pipeline barriers, the
// protocol work overlaps the next tile's mainloop, which is how the pages hide it in
// warp-specialised persistent kernels (section III-C, Fig. 2b).
#pragma once

#include <cuda_bf16.h>

#include "protocol.h"
#include "ptx.cuh"

namespace mlpc {

constexpr int kMaxStages = 4;
constexpr int kBM = 128;          // rows per tile = TMEM lanes
constexpr int kBK = 64;           // 64 bf16 = 128 bytes = one 128B-swizzle row
constexpr int kThreads = 256;
constexpr int kSchedDepth = 4;
constexpr int kMaxPipe = 16;
constexpr int kTicketLead = 4;    // k-blocks before the end of a tile at which the next ticket is taken
constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KB

// Device status codes (match mlp_status).
constexpr uint32_t kStatusTimeout = 5;
constexpr uint32_t kStatusBadTile = 7;

struct StageParams {
    int32_t M, K, N;
    int32_t BN;            // tile width (32, 64, 128, 256)
    int32_t tiles_m, tiles_n;
    int32_t k_blocks;
    int32_t b_swz;         // bytes of one B swizzle row: 128 (BN >= 64) or 64 (BN = 32)
    __nv_bfloat16 *out;    // M x N row-major
    const __nv_bfloat16 *residual;  // M x N (the chain input) or null
    int32_t gelu;
    int32_t b_kmajor;      // 1: weights stored N x K, B tile is K-major (one box of BN rows)
};

// Stage boundary s -> s+1.  The scoreboard holds one counter per group of consumer tiles with
// identical producer sets (a row panel for GEMM chains); see dep_groups.h.
struct BoundaryParams {
    const int32_t *pg_off;     // producer tile -> groups it feeds (CSR)
    const int32_t *pg_tgt;
    const int32_t *grp_off;    // group -> member consumer tiles (CSR)
    const int32_t *grp_mem;
    const int32_t *grp_init;   // producers each group waits for
    uint32_t *count;           // one counter per group
    unsigned long long *queue; // one slot per consumer tile
    uint32_t *tail;
};

struct EventRec {
    int32_t stage, tile, smid, cta;
    uint64_t t_start, t_end;
    uint32_t seq_start, seq_end;
};

struct ChainParams {
    CUtensorMap mapA[kMaxStages];
    CUtensorMap mapB[kMaxStages];
    StageParams st[kMaxStages];
    BoundaryParams bd[kMaxStages - 1];
    int32_t num_stages;
    int32_t pipelined;
    int32_t first_stage;                 // non-pipelined launches run this single stage
    int32_t m_tile_begin, m_tile_end;    // ... over these row tiles
    int32_t stage_base[kMaxStages + 1];  // pipelined: first ticket of each stage
    int32_t raster_group;
    int32_t num_pipe;                    // shared-memory ring depth
    uint32_t stage_bytes;                // bytes of one ring slot (A + B)
    uint32_t tmem_cols;
    int32_t acc_stride;                  // TMEM columns between the two accumulator buffers
    int32_t acc_split;                   // 1, or 2: k16 steps alternate between two sub-accumulators
    int32_t sub_stride;                  // TMEM columns between the sub-accumulators of a buffer
    int32_t drop_tile;                   // fault injection (-1: off)
    uint64_t timeout_ns;
    uint32_t *ticket;
    uint32_t *done;
    uint32_t *epoch;
    uint32_t *status;
    uint32_t *seq;
    EventRec *events;                    // null: no event log
};

struct __align__(8) Ctrl {
    uint64_t full[kMaxPipe], empty[kMaxPipe];
    uint64_t tfull[2], tempty[2];
    uint64_t sfull[kSchedDepth], sempty[kSchedDepth];
    uint64_t drain;
    uint64_t epi_sync;
    uint64_t want_next;   // TMA -> scheduler: take the next ticket now
    int32_t item_stage[kSchedDepth], item_tile[kSchedDepth];
    uint32_t tmem_base;
    volatile int32_t abort_flag;
    int32_t skip;
    uint32_t epoch;
};

__host__ __device__ inline uint32_t ctrl_offset(int num_pipe, uint32_t stage_bytes)
{
    return static_cast<uint32_t>(num_pipe) * stage_bytes;
}

__host__ inline size_t chain_smem_bytes(int num_pipe, uint32_t stage_bytes)
{
    return 1024 + ctrl_offset(num_pipe, stage_bytes) + sizeof(Ctrl);
}

// ------------------------------------------------------------------------ bounded waits --
// Every wait has a deadline.  On expiry the waiter records kStatusTimeout (first error wins)
// and raises the CTA's abort flag so the other roles stop too.  Returns false on abort.
// Drain waits (after an abort, for this CTA's own copies and MMAs in flight) ignore the abort
// flag and use a short fixed limit.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, Ctrl *c, const ChainParams &p,
                                         bool honor_abort = true)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    const uint64_t limit = honor_abort ? 2 * p.timeout_ns + 1000000000ull : 200000000ull;
    while (true) {
        if (mbar_try_wait(bar, parity))
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
__device__ __forceinline__ bool warp_wait_bar(uint64_t *bar, uint32_t parity, Ctrl *c, const ChainParams &p)
{
    uint32_t ok = 0;
    if ((threadIdx.x & 31) == 0)
        ok = wait_bar(bar, parity, c, p) ? 1u : 0u;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
}

__device__ __forceinline__ float gelu_tanh_f32(float x)
{
    const float k0 = 0.7978845608028654f;  // sqrt(2 / pi)
    const float k1 = 0.044715f;
    return 0.5f * x * (1.0f + tanhf(k0 * (x + k1 * x * x * x)));
}

// ------------------------------------------------------------------------------ scheduler --
__device__ __forceinline__ void role_scheduler(const ChainParams &p, Ctrl *c)
{
    const int32_t total = p.pipelined ? p.stage_base[p.num_stages] : 0;
    for (int32_t it = 0;; ++it) {
        const int32_t slot = it % kSchedDepth;
        const uint32_t ph = (it / kSchedDepth) & 1;
        if (!wait_bar(&c->sempty[slot], ph ^ 1, c, p))
            return;
        // Take tickets just in time: a ticket taken early would sit in this CTA while other
        // CTAs idle, so wait until the TMA warp is about to finish its current tile.
        if (it > 0 && !wait_bar(&c->want_next, (it - 1) & 1, c, p))
            return;
        int32_t stage = -1, tile = 0;
        if (p.pipelined) {
            const int32_t t = static_cast<int32_t>(atom_add_relaxed_gpu(p.ticket, 1u));
            if (t < total) {
                int32_t s = 0;
                s = stage_of_ticket(p.stage_base, t);
                const int32_t local = t - p.stage_base[s];
                if (s == 0) {
                    tile = raster_tile(local, p.st[0].tiles_m, p.st[0].tiles_n, p.raster_group);
                    stage = 0;
                } else {
                    // Consumer prologue: poll queue slot `local` until this run's entry lands.
                    const unsigned long long *q = p.bd[s - 1].queue + local;
                    uint64_t v = ld_acquire_gpu_u64(q);
                    if (!queue_entry_ready(v, c->epoch)) {
                        const uint64_t t0 = globaltimer_ns();
                        uint32_t backoff = 32;
                        while (true) {
                            __nanosleep(backoff);
                            backoff = backoff < 256 ? backoff * 2 : 256;
                            v = ld_acquire_gpu_u64(q);
                            if (queue_entry_ready(v, c->epoch))
                                break;
                            if (ld_relaxed_gpu_u32(p.status) != 0 || c->abort_flag) {
                                v = 0;
                                break;
                            }
                            if (globaltimer_ns() - t0 > p.timeout_ns) {
                                atomicCAS(p.status, 0u, kStatusTimeout);
                                v = 0;
                                break;
                            }
                        }
                    }
                    if (queue_entry_ready(v, c->epoch)) {
                        tile = queue_entry_tile(v);
                        if (tile < 0 || tile >= p.st[s].tiles_m * p.st[s].tiles_n) {
                            atomicCAS(p.status, 0u, kStatusBadTile);
                        } else {
                            stage = s;
                            // Later TMA (async proxy) reads of the producers' output must not
                            // be ordered before this acquire.
                            fence_proxy_async_global();
                        }
                    }
                }
                if (stage >= 0 && p.events) {
                    EventRec *e = p.events + p.stage_base[stage] + tile;
                    e->stage = stage;
                    e->tile = tile;
                    e->smid = static_cast<int32_t>(smid());
                    e->cta = static_cast<int32_t>(blockIdx.x);
                    e->seq_start = atom_add_relaxed_gpu(p.seq, 1u);
                    e->t_start = globaltimer_ns();
                }
            }
        } else {
            const int32_t tn = p.st[p.first_stage].tiles_n;
            const int32_t n_local = (p.m_tile_end - p.m_tile_begin) * tn;
            const int32_t local = static_cast<int32_t>(blockIdx.x) + it * static_cast<int32_t>(gridDim.x);
            if (local < n_local) {
                stage = p.first_stage;
                tile = p.m_tile_begin * tn + local;
            }
        }
        c->item_stage[slot] = stage;
        c->item_tile[slot] = tile;
        mbar_arrive(&c->sfull[slot]);
        if (stage < 0)
            return;
    }
}

// ---------------------------------------------------------------------------- TMA producer --
__device__ __forceinline__ void role_tma(const ChainParams &p, Ctrl *c, uint8_t *ring)
{
    const uint64_t pol_act = policy_evict_last();    // activations are re-read by many tiles
    const uint64_t pol_w = policy_evict_first();     // each weight tile is read by one row panel
    int32_t ps = 0;
    uint32_t pph = 0;
    uint32_t fills[kMaxPipe];
    for (int i = 0; i < kMaxPipe; ++i)
        fills[i] = 0;
    for (int32_t it = 0;; ++it) {
        const int32_t slot = it % kSchedDepth;
        if (!wait_bar(&c->sfull[slot], (it / kSchedDepth) & 1, c, p))
            break;
        const int32_t s = c->item_stage[slot];
        const int32_t tile = c->item_tile[slot];
        mbar_arrive(&c->sempty[slot]);
        if (s < 0)
            break;
        if (s > 0)
            fence_proxy_async_global();
        const StageParams &sp = p.st[s];
        const int32_t m0 = (tile / sp.tiles_n) * kBM;
        const int32_t n0 = (tile % sp.tiles_n) * sp.BN;
        const int32_t box_cols = sp.b_swz / 2;
        const uint32_t box_bytes = kBK * sp.b_swz;
        const int32_t nbox = sp.BN / box_cols;
        const uint32_t bytes = kABytes + static_cast<uint32_t>(kBK * sp.BN * 2);
        const int32_t lead_kb = sp.k_blocks > kTicketLead ? sp.k_blocks - kTicketLead : 0;
        bool ok = true;
        for (int32_t kb = 0; kb < sp.k_blocks; ++kb) {
            if (kb == lead_kb)
                mbar_arrive(&c->want_next);
            if (!wait_bar(&c->empty[ps], pph ^ 1, c, p)) {
                ok = false;
                break;
            }
            uint8_t *a = ring + static_cast<size_t>(ps) * p.stage_bytes;
            uint8_t *b = a + kABytes;
            mbar_arrive_expect_tx(&c->full[ps], bytes);
            tma_load_2d(a, &p.mapA[s], &c->full[ps], kb * kBK, m0, pol_act);
            if (sp.b_kmajor) {
                tma_load_2d(b, &p.mapB[s], &c->full[ps], kb * kBK, n0, pol_w);
            } else {
                for (int32_t j = 0; j < nbox; ++j)
                    tma_load_2d(b + j * box_bytes, &p.mapB[s], &c->full[ps], n0 + j * box_cols, kb * kBK, pol_w);
            }
            ++fills[ps];
            if (++ps == p.num_pipe) {
                ps = 0;
                pph ^= 1;
            }
        }
        if (!ok)
            break;
    }
    if (c->abort_flag) {
        // Let every copy this thread issued land before the CTA's shared memory goes away.
        for (int32_t i = 0; i < p.num_pipe; ++i)
            if (fills[i] > 0)
                wait_bar(&c->full[i], (fills[i] - 1) & 1, c, p, false);
    }
}

// ------------------------------------------------------------------------------ MMA issuer --
__device__ __forceinline__ void role_mma(const ChainParams &p, Ctrl *c, uint8_t *ring, uint32_t tmem_base)
{
    int32_t ps = 0;
    uint32_t pph = 0;
    uint32_t local_tiles = 0;
    bool issued = false;
    for (int32_t it = 0;; ++it) {
        const int32_t slot = it % kSchedDepth;
        if (!wait_bar(&c->sfull[slot], (it / kSchedDepth) & 1, c, p))
            break;
        const int32_t s = c->item_stage[slot];
        mbar_arrive(&c->sempty[slot]);
        if (s < 0)
            break;
        const StageParams &sp = p.st[s];
        const uint32_t acc = local_tiles & 1;
        const uint32_t acc_ph = (local_tiles >> 1) & 1;
        if (!wait_bar(&c->tempty[acc], acc_ph ^ 1, c, p))
            break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * static_cast<uint32_t>(p.acc_stride);
        const uint32_t idesc = idesc_bf16_f32(kBM, static_cast<uint32_t>(sp.BN), sp.b_kmajor ? 0u : 1u);
        const uint32_t b_swz = static_cast<uint32_t>(sp.b_swz);
        const uint32_t b_code = b_swz == 128 ? 2u : (b_swz == 64 ? 4u : 6u);
        const bool split2 = p.acc_split == 2;
        bool ok = true;
        for (int32_t kb = 0; kb < sp.k_blocks; ++kb) {
            // TMA fills and tcgen05.mma reads are both async-proxy operations ordered by the
            // mbarrier's transaction count: no tcgen05 fence is needed per k block.
            if (!wait_bar(&c->full[ps], pph, c, p)) {
                ok = false;
                break;
            }
            const uint32_t a_addr = smem_u32(ring + static_cast<size_t>(ps) * p.stage_bytes);
            const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
            for (uint32_t kk = 0; kk < kBK / 16; ++kk) {
                // A: K-major, 128B swizzle; a 16-wide k step is 32 bytes along the row.
                const uint64_t ad = smem_desc(a_addr + kk * 32u, 16u, 1024u, 2u);
                // B: MN-major; a 16-deep k step is 16 rows of b_swz bytes.  LBO: next block of
                // b_swz/2 columns (one TMA box of 64 rows); SBO: next group of 8 rows.
                // B stored N x K: K-major like A, BN rows of 128 bytes.
                const uint64_t bd = sp.b_kmajor
                                        ? smem_desc(b_addr + kk * 32u, 16u, 1024u, 2u)
                                        : smem_desc(b_addr + kk * 16u * b_swz, kBK * b_swz, 8u * b_swz, b_code);
                // k step j goes to sub-accumulator j % acc_split; its first step overwrites.
                const uint32_t j = static_cast<uint32_t>(kb) * (kBK / 16) + kk;
                const uint32_t sub = split2 ? (j & 1u) : 0u;
                mma_bf16_ss(d_tmem + sub * static_cast<uint32_t>(p.sub_stride), ad, bd, idesc,
                            j >= (split2 ? 2u : 1u) ? 1u : 0u);
            }
            issued = true;
            mma_commit(&c->empty[ps]);  // frees the ring slot once these MMAs have read it
            if (++ps == p.num_pipe) {
                ps = 0;
                pph ^= 1;
            }
        }
        if (!ok)
            break;
        mma_commit(&c->tfull[acc]);     // accumulator ready for the epilogue
        ++local_tiles;
    }
    if (c->abort_flag && issued) {
        mma_commit(&c->drain);
        wait_bar(&c->drain, 0, c, p, false);
    }
}

// -------------------------------------------------------------------------------- epilogue --
__device__ __forceinline__ void store_chunk(const StageParams &sp, int32_t m, int32_t n, const uint32_t (&r)[32])
{
    if (m >= sp.M)
        return;
    const __nv_bfloat16 *res = sp.residual ? sp.residual + static_cast<size_t>(m) * sp.N + n : nullptr;
    __nv_bfloat16 *dst = sp.out + static_cast<size_t>(m) * sp.N + n;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (n + 8 * j >= sp.N)
            break;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            v[e] = __uint_as_float(r[8 * j + e]);
            if (sp.gelu)
                v[e] = gelu_tanh_f32(v[e]);
        }
        if (res) {
            const uint4 rv = *reinterpret_cast<const uint4 *>(res + 8 * j);
            const __nv_bfloat162 *rb = reinterpret_cast<const __nv_bfloat162 *>(&rv);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(rb[e]);
                v[2 * e] += f.x;
                v[2 * e + 1] += f.y;
            }
        }
        uint4 o;
        __nv_bfloat162 *ob = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            ob[e] = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
        *reinterpret_cast<uint4 *>(dst + 8 * j) = o;
    }
}

__device__ __forceinline__ void role_epilogue(const ChainParams &p, Ctrl *c, uint32_t tmem_base)
{
    const int32_t warp = threadIdx.x / 32;
    const int32_t lane = threadIdx.x & 31;
    const int32_t quad = warp & 3;              // TMEM lanes 32*quad .. 32*quad+31
    const int32_t row = quad * 32 + lane;
    uint32_t local_tiles = 0;
    uint32_t epi_phase = 0;
    for (int32_t it = 0;; ++it) {
        const int32_t slot = it % kSchedDepth;
        if (!warp_wait_bar(&c->sfull[slot], (it / kSchedDepth) & 1, c, p))
            break;
        int32_t s = 0, tile = 0;
        if (lane == 0) {
            s = c->item_stage[slot];
            tile = c->item_tile[slot];
            mbar_arrive(&c->sempty[slot]);
        }
        s = __shfl_sync(0xffffffffu, s, 0);
        tile = __shfl_sync(0xffffffffu, tile, 0);
        if (s < 0)
            break;
        const StageParams &sp = p.st[s];
        const uint32_t acc = local_tiles & 1;
        const uint32_t acc_ph = (local_tiles >> 1) & 1;
        if (!warp_wait_bar(&c->tfull[acc], acc_ph, c, p))
            break;
        tc_fence_after();
        const int32_t m = (tile / sp.tiles_n) * kBM + row;
        const int32_t n0 = (tile % sp.tiles_n) * sp.BN;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * p.acc_stride;
        for (int32_t c0 = 0; c0 < sp.BN; c0 += 32) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + c0, r);
            if (p.acc_split == 2) {
                uint32_t r2[32];
                tmem_ld_32x32b_x32(taddr + p.sub_stride + c0, r2);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e)   // even k steps + odd k steps, in that order
                    r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(r2[e]));
            } else {
                tmem_ld_wait();
            }
            store_chunk(sp, m, n0 + c0, r);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&c->tempty[acc]);   // the MMA warp may reuse this accumulator
        ++local_tiles;

        const bool producer = p.pipelined && s + 1 < p.num_stages;
        if (producer || (p.pipelined && p.events)) {
            // Injected epilogue: every thread orders its stores, the four warps meet (a bounded
            // mbarrier rather than bar.sync, so an aborting warp cannot strand the others), then
            // one warp releases and decrements the scoreboard.
            fence_acq_rel_gpu();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&c->epi_sync);
            if (!warp_wait_bar(&c->epi_sync, epi_phase, c, p))
                break;
            epi_phase ^= 1;
            if (warp == 4) {
                if (lane == 0 && p.events) {
                    EventRec *e = p.events + p.stage_base[s] + tile;
                    e->seq_end = atom_add_relaxed_gpu(p.seq, 1u);
                    e->t_end = globaltimer_ns();
                }
                __syncwarp();
                const bool dropped = (s == 0 && tile == p.drop_tile);
                if (producer && !dropped) {
                    const BoundaryParams &bd = p.bd[s];
                    const int32_t e0 = bd.pg_off[tile], e1 = bd.pg_off[tile + 1];
                    for (int32_t eb = e0; eb < e1; eb += 32) {
                        const int32_t e = eb + lane;
                        int32_t g = -1;
                        bool fire = false;
                        if (e < e1) {
                            g = bd.pg_tgt[e];
                            fence_acq_rel_gpu();
                            const uint32_t old = atom_add_acq_rel_gpu(bd.count + g, 0xffffffffu);
                            fire = (old == 1u);
                            if (fire)   // re-arm for the next run; no producer touches it again
                                bd.count[g] = static_cast<uint32_t>(bd.grp_init[g]);
                        }
                        // Every group this warp completed is published by the whole warp: the
                        // lane whose acq_rel decrement reached zero acquired every earlier
                        // producer's release; __syncwarp orders that before each lane's release
                        // fence, which makes its relaxed queue stores carry the release.
                        uint32_t todo = __ballot_sync(0xffffffffu, fire);
                        while (todo) {
                            const int32_t src = __ffs(todo) - 1;
                            todo &= todo - 1;
                            const int32_t gg = __shfl_sync(0xffffffffu, g, src);
                            const int32_t m0 = bd.grp_off[gg], n = bd.grp_off[gg + 1] - m0;
                            uint32_t q0 = 0;
                            if (lane == src)
                                q0 = atom_add_relaxed_gpu(bd.tail, static_cast<uint32_t>(n));
                            q0 = __shfl_sync(0xffffffffu, q0, src);
                            __syncwarp();
                            fence_acq_rel_gpu();
                            for (int32_t i = lane; i < n; i += 32)
                                st_relaxed_gpu_u64(bd.queue + q0 + i, queue_entry(c->epoch, bd.grp_mem[m0 + i]));
                        }
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------------------------------ the kernel --
__global__ void __launch_bounds__(kThreads, 1) chain_kernel(const __grid_constant__ ChainParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + (((base + 1023u) & ~1023u) - base);
    Ctrl *c = reinterpret_cast<Ctrl *>(ring + ctrl_offset(p.num_pipe, p.stage_bytes));
    const int32_t warp = threadIdx.x / 32;
    const int32_t lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.num_pipe; ++i) {
            mbar_init(&c->full[i], 1);
            mbar_init(&c->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&c->tfull[i], 1);
            mbar_init(&c->tempty[i], 4);
        }
        for (int i = 0; i < kSchedDepth; ++i) {
            mbar_init(&c->sfull[i], 1);
            mbar_init(&c->sempty[i], 6);   // TMA + MMA + 4 epilogue warps
        }
        mbar_init(&c->drain, 1);
        mbar_init(&c->epi_sync, 4);
        mbar_init(&c->want_next, 1);
        c->abort_flag = 0;
        c->skip = ld_relaxed_gpu_u32(p.status) != 0;   // sticky error: do nothing
        c->epoch = p.pipelined ? ld_relaxed_gpu_u32(p.epoch) : 0u;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&p.mapA[0]);
        prefetch_tensormap(&p.mapB[0]);
    }
    if (warp == 1) {
        tmem_alloc(&c->tmem_base, p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = c->tmem_base;

    if (!c->skip) {
        if (warp == 0) {
            if (lane == 0)
                role_tma(p, c, ring);
        } else if (warp == 1) {
            if (lane == 0)
                role_mma(p, c, ring, tmem_base);
            __syncwarp();
        } else if (warp == 2) {
            if (lane == 0)
                role_scheduler(p, c);
        } else if (warp >= 4) {
            role_epilogue(p, c, tmem_base);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
    if (threadIdx.x == 0 && p.pipelined && !c->skip) {
        // The last CTA out re-arms the run-wide counters for the next run.  Scoreboard counters
        // were re-armed by their last producer; queue slots carry the run's epoch instead of
        // being cleared.
        fence_acq_rel_gpu();
        const uint32_t old = atom_add_acq_rel_gpu(p.done, 1u);
        if (old == gridDim.x - 1) {
            *p.ticket = 0;
            for (int b = 0; b + 1 < p.num_stages; ++b)
                *p.bd[b].tail = 0;
            *p.done = 0;
            *p.epoch = c->epoch + 1;
            fence_acq_rel_gpu();
        }
    }
}

}  // namespace mlpc
