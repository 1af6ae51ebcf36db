// protocol.h -- the pure (host + device) arithmetic of the CTA-pipelining protocol: ticket to
// stage, first-stage raster order, the epoch-tagged work-queue entry and the run targets of the
// accumulating scoreboard counters.  The CUDA kernel and
// the host-thread protocol model both use these, so the model exercises the kernel's logic.
//
// Work-queue entry (one 64-bit word per slot): high 32 bits = run epoch + 1, low 32 bits = the
// ready consumer tile id.  A slot holds "this run's" entry exactly when its high word equals
// the current epoch + 1, so slots never need clearing between runs (the pages' queue is a
// plain list of ready CTA ids, section III-A; the epoch tag is this library's addition).
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define MLPC_HD __host__ __device__ __forceinline__
#else
#define MLPC_HD inline
#endif

namespace mlpc {

MLPC_HD uint64_t queue_entry(uint32_t epoch, int32_t tile)
{
    return ((static_cast<uint64_t>(epoch) + 1u) << 32) | static_cast<uint32_t>(tile);
}

MLPC_HD bool queue_entry_ready(uint64_t v, uint32_t epoch)
{
    return (v >> 32) == static_cast<uint64_t>(epoch) + 1u;
}

MLPC_HD int32_t queue_entry_tile(uint64_t v) { return static_cast<int32_t>(v & 0xffffffffu); }

// Scoreboard counters count releases and are never re-armed: a counter accumulates over all
// runs of a handle, so a group that waits for `per_run` releases in every run has completed run
// `epoch` (0, 1, ...) once its count reaches per_run x (epoch + 1).
MLPC_HD uint32_t run_target(int32_t per_run, uint32_t epoch)
{
    return static_cast<uint32_t>(per_run) * (epoch + 1u);
}

// The release that took the count from `old` to old + 1 completed the run (and so publishes the
// group's members on the work-queue).
MLPC_HD bool release_completes(uint32_t old, uint32_t target) { return old + 1u == target; }

// A count read by a waiter has reached the run's target (wrap-safe comparison).
MLPC_HD bool count_reached(uint32_t v, uint32_t target) { return static_cast<int32_t>(v - target) >= 0; }

// Run-wide counters are never reset either.  Every CTA of a pipelined launch adds 1 to a 64-bit
// launch counter once, at its start, so run e's CTAs read e x ctas .. e x ctas + ctas - 1: the
// run's epoch is that value divided by the CTA count.
MLPC_HD uint32_t epoch_of_launch(uint64_t old, uint32_t ctas) { return static_cast<uint32_t>(old / ctas); }

// A run takes exactly `per_run` increments of the ticket counter (one per cluster item: every
// valid ticket once, plus one past the end per cluster that had a first item) and of each stage
// boundary's queue tail (one per consumer tile), so run e's own count is the raw value minus
// per_run x e (mod 2^32, so the counters may wrap).
MLPC_HD uint32_t run_relative(uint32_t raw, uint32_t epoch, uint32_t per_run) { return raw - per_run * epoch; }

// Tickets are issued stage by stage: [base[0], base[1]) are first-stage tiles, ...
MLPC_HD int32_t stage_of_ticket(const int32_t *base, int32_t t)
{
    int32_t s = 0;
    while (t >= base[s + 1])
        ++s;
    return s;
}

// First-stage raster: ticket -> tile id (row-major over a tiles_m x tiles_n grid).
// g <= 1: whole row panels in order, so consumer row panels become ready as early as possible.
// g > 1: groups of g row panels, column-major inside a group (better L2 reuse of weight columns;
// the panels of one group finish together).
MLPC_HD int32_t raster_tile(int32_t local, int32_t tiles_m, int32_t tiles_n, int32_t g)
{
    if (g <= 1)
        return local;
    const int32_t per_group = g * tiles_n;
    const int32_t grp = local / per_group;
    const int32_t rem = tiles_m - grp * g;
    const int32_t rows = rem < g ? rem : g;
    const int32_t idx = local - grp * per_group;
    const int32_t n = idx / rows;
    const int32_t m = grp * g + idx % rows;
    return m * tiles_n + n;
}

}  // namespace mlpc
