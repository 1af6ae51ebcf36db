// dep_groups.h -- host-side compression of a dependency array into scoreboard groups.
//
// Consumer tiles whose producer sets are identical become ready at the same moment, so they
// can share one scoreboard counter: the counter of a group starts at the group's in-degree,
// each producer decrements every group it feeds once, and the decrement that reaches zero
// pushes all members of the group onto the work-queue.  Readiness is exactly that of one
// counter per consumer tile (section III-A of the CTA-pipelining paper), with O(P) instead of
// O(P * consumers-per-panel) atomics.  For a GEMM chain with equal row tiles a group is the set
// of consumer tiles of one row panel.
#pragma once

#include <cstdint>
#include <vector>

namespace mlpc {

struct DepGroups {
    std::vector<int32_t> pg_off, pg_tgt;    // producer -> groups it feeds (ascending)
    std::vector<int32_t> grp_off, grp_mem;  // group -> member consumer tiles (ascending)
    std::vector<int32_t> grp_init;          // producers each group waits for
    std::vector<int32_t> cons_grp;          // consumer tile -> its group
};

// prod_off[P+1] / prod_tgt: producer -> consumers CSR (consumer ids ascending per producer).
DepGroups build_groups(const int32_t *prod_off, const int32_t *prod_tgt, int32_t P, int32_t C);

// One group per run of `g` consecutive consumer row panels (consumer tile c lies in row panel
// c / tiles_n).  A merged group waits for the union of its members' producers, so it is never
// ready before any of its members would have been; when the producers finish those panels
// together (the first stage's raster walks g panels column by column) it costs nothing.  Its
// members are listed column by column -- all of its panels at n = 0, then n = 1, ... -- so that
// consecutive queue slots read the same weight column slab and share it in L2.
DepGroups merge_groups_by_panel(const int32_t *prod_off, const int32_t *prod_tgt, int32_t P, int32_t C,
                                int32_t tiles_n, int32_t g);

// The scoreboard groups of one stage boundary, as mlp_chain_create uploads them: row-panel
// groups merged per raster group of g > 1 panels, else classes of identical producer sets.
DepGroups scoreboard_groups(const int32_t *prod_off, const int32_t *prod_tgt, int32_t P, int32_t C,
                            int32_t tiles_n, int32_t g);

}  // namespace mlpc
