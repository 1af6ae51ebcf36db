// host_protocol.cpp -- host-only parts of the library: the dependency-array builder used by
// mlp_chain_create, and a host-thread model of the scoreboard / work-queue protocol.
//
// Dependency array (section III-A of "CTA-Pipelining: A Latency-Oriented Spatial Scaling
// Method for Multi-GPU Systems": built from the static tile dataflow; a consumer CTA consumes
// one or more input tiles and produces one output tile).  A consumer tile of GEMM s+1 reads a
// band of rows of GEMM s's output across all of its columns (that is GEMM s+1's reduction
// dimension), so it depends on every producer tile whose row range overlaps its own.  This
// builder works on row intervals; the oracle enumerates elements instead.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdint>
#include <map>
#include <random>
#include <thread>
#include <vector>

#include "../../include/mlp_chain.h"
#include "dep_groups.h"
#include "protocol.h"

extern "C" int64_t mlp_deps_build(int64_t M, int64_t n_out, int64_t n_next, int32_t bm_p, int32_t bn_p,
                                  int32_t bm_c, int32_t bn_c, int32_t *prod_off, int32_t *prod_tgt,
                                  int64_t tgt_cap, int32_t *init_count)
{
    if (M <= 0 || n_out <= 0 || n_next <= 0 || bm_p <= 0 || bn_p <= 0 || bm_c <= 0 || bn_c <= 0)
        return -1;
    const int64_t Pm = (M + bm_p - 1) / bm_p, Pn = (n_out + bn_p - 1) / bn_p;
    const int64_t Cm = (M + bm_c - 1) / bm_c, Cn = (n_next + bn_c - 1) / bn_c;
    if (Pm * Pn >= INT32_MAX || Cm * Cn >= INT32_MAX)
        return -1;
    // in-degree: producer row tiles overlapping the consumer's rows, times all producer columns
    int64_t nnz = 0;
    for (int64_t mc = 0; mc < Cm; ++mc) {
        const int64_t r0 = mc * bm_c, r1 = std::min<int64_t>(M, (mc + 1) * bm_c);
        const int64_t deg = ((r1 - 1) / bm_p - r0 / bm_p + 1) * Pn;
        for (int64_t nc = 0; nc < Cn; ++nc)
            if (init_count)
                init_count[mc * Cn + nc] = static_cast<int32_t>(deg);
        nnz += deg * Cn;
    }
    if (!prod_off || !prod_tgt)
        return nnz;
    if (nnz > tgt_cap || nnz >= INT32_MAX)
        return -1;
    int64_t e = 0;
    for (int64_t mp = 0; mp < Pm; ++mp) {
        const int64_t r0 = mp * bm_p, r1 = std::min<int64_t>(M, (mp + 1) * bm_p);
        const int64_t mc0 = r0 / bm_c, mc1 = (r1 - 1) / bm_c;  // consumer row tiles it feeds
        for (int64_t np = 0; np < Pn; ++np) {
            prod_off[mp * Pn + np] = static_cast<int32_t>(e);
            for (int64_t mc = mc0; mc <= mc1; ++mc)
                for (int64_t nc = 0; nc < Cn; ++nc)
                    prod_tgt[e++] = static_cast<int32_t>(mc * Cn + nc);
        }
    }
    prod_off[Pm * Pn] = static_cast<int32_t>(e);
    return e;
}

mlpc::DepGroups mlpc::build_groups(const int32_t *prod_off, const int32_t *prod_tgt, int32_t P, int32_t C)
{
    // producers of each consumer, ascending (producers are visited in ascending order)
    std::vector<std::vector<int32_t>> in(static_cast<size_t>(C));
    for (int32_t p = 0; p < P; ++p)
        for (int32_t e = prod_off[p]; e < prod_off[p + 1]; ++e)
            in[static_cast<size_t>(prod_tgt[e])].push_back(p);
    std::map<std::vector<int32_t>, int32_t> id;
    std::vector<int32_t> group_of(static_cast<size_t>(C));
    std::vector<std::vector<int32_t>> members;
    DepGroups g;
    for (int32_t c = 0; c < C; ++c) {
        auto it = id.find(in[c]);
        int32_t gid;
        if (it == id.end()) {
            gid = static_cast<int32_t>(members.size());
            id.emplace(in[c], gid);
            members.emplace_back();
            g.grp_init.push_back(static_cast<int32_t>(in[c].size()));
        } else {
            gid = it->second;
        }
        group_of[c] = gid;
        members[gid].push_back(c);
    }
    g.cons_grp = group_of;
    g.grp_off.push_back(0);
    for (auto &m : members) {
        g.grp_mem.insert(g.grp_mem.end(), m.begin(), m.end());
        g.grp_off.push_back(static_cast<int32_t>(g.grp_mem.size()));
    }
    g.pg_off.push_back(0);
    for (int32_t p = 0; p < P; ++p) {
        std::vector<int32_t> gs;
        for (int32_t e = prod_off[p]; e < prod_off[p + 1]; ++e)
            gs.push_back(group_of[prod_tgt[e]]);
        std::sort(gs.begin(), gs.end());
        gs.erase(std::unique(gs.begin(), gs.end()), gs.end());
        g.pg_tgt.insert(g.pg_tgt.end(), gs.begin(), gs.end());
        g.pg_off.push_back(static_cast<int32_t>(g.pg_tgt.size()));
    }
    return g;
}

mlpc::DepGroups mlpc::merge_groups_by_panel(const int32_t *prod_off, const int32_t *prod_tgt, int32_t P, int32_t C,
                                            int32_t tiles_n, int32_t g)
{
    const int32_t panels = (C + tiles_n - 1) / tiles_n;
    const int32_t supers = (panels + g - 1) / g;
    std::vector<std::vector<int32_t>> in(static_cast<size_t>(C));
    for (int32_t p = 0; p < P; ++p)
        for (int32_t e = prod_off[p]; e < prod_off[p + 1]; ++e)
            in[static_cast<size_t>(prod_tgt[e])].push_back(p);
    DepGroups r;
    r.cons_grp.assign(static_cast<size_t>(C), 0);
    r.grp_off.push_back(0);
    for (int32_t sg = 0; sg < supers; ++sg) {
        const int32_t m0 = sg * g, m1 = std::min(panels, m0 + g);
        std::vector<int32_t> producers;
        for (int32_t n = 0; n < tiles_n; ++n)
            for (int32_t m = m0; m < m1; ++m) {
                const int32_t c = m * tiles_n + n;
                if (c >= C)
                    continue;
                r.grp_mem.push_back(c);
                r.cons_grp[static_cast<size_t>(c)] = sg;
                producers.insert(producers.end(), in[static_cast<size_t>(c)].begin(), in[static_cast<size_t>(c)].end());
            }
        std::sort(producers.begin(), producers.end());
        producers.erase(std::unique(producers.begin(), producers.end()), producers.end());
        r.grp_init.push_back(static_cast<int32_t>(producers.size()));
        r.grp_off.push_back(static_cast<int32_t>(r.grp_mem.size()));
    }
    r.pg_off.push_back(0);
    for (int32_t p = 0; p < P; ++p) {
        std::vector<int32_t> gs;
        for (int32_t e = prod_off[p]; e < prod_off[p + 1]; ++e)
            gs.push_back(r.cons_grp[static_cast<size_t>(prod_tgt[e])]);
        std::sort(gs.begin(), gs.end());
        gs.erase(std::unique(gs.begin(), gs.end()), gs.end());
        r.pg_tgt.insert(r.pg_tgt.end(), gs.begin(), gs.end());
        r.pg_off.push_back(static_cast<int32_t>(r.pg_tgt.size()));
    }
    return r;
}

mlpc::DepGroups mlpc::scoreboard_groups(const int32_t *prod_off, const int32_t *prod_tgt, int32_t P, int32_t C,
                                        int32_t tiles_n, int32_t g)
{
    return g > 1 ? merge_groups_by_panel(prod_off, prod_tgt, P, C, tiles_n, g) : build_groups(prod_off, prod_tgt, P, C);
}

extern "C" mlp_status mlp_scoreboard_build(int64_t M, int64_t n_out, int64_t n_next, int32_t bm, int32_t bn_p,
                                           int32_t bn_c, int32_t raster_group, int32_t releases_per_producer,
                                           mlp_scoreboard *sb)
{
    if (!sb || releases_per_producer < 1)
        return MLP_ERR_INVALID_ARG;
    const int64_t nnz = mlp_deps_build(M, n_out, n_next, bm, bn_p, bm, bn_c, nullptr, nullptr, 0, nullptr);
    if (nnz < 0)
        return MLP_ERR_INVALID_ARG;
    const int64_t P = ((M + bm - 1) / bm) * ((n_out + bn_p - 1) / bn_p);
    const int64_t C = ((M + bm - 1) / bm) * ((n_next + bn_c - 1) / bn_c);
    std::vector<int32_t> off(static_cast<size_t>(P + 1)), tgt(static_cast<size_t>(std::max<int64_t>(nnz, 1))),
        init(static_cast<size_t>(C));
    mlp_deps_build(M, n_out, n_next, bm, bn_p, bm, bn_c, off.data(), tgt.data(), nnz, init.data());
    const int32_t tiles_n = static_cast<int32_t>((n_next + bn_c - 1) / bn_c);
    const mlpc::DepGroups G = mlpc::scoreboard_groups(off.data(), tgt.data(), static_cast<int32_t>(P),
                                                static_cast<int32_t>(C), tiles_n, raster_group);
    sb->producers = static_cast<int32_t>(P);
    sb->consumers = static_cast<int32_t>(C);
    sb->groups = static_cast<int32_t>(G.grp_init.size());
    sb->edges = static_cast<int32_t>(G.pg_tgt.size());
    sb->releases_per_producer = releases_per_producer;
    if (!sb->pg_off || !sb->pg_tgt || !sb->grp_off || !sb->grp_mem || !sb->grp_target || !sb->cons_grp)
        return MLP_OK;
    std::copy(G.pg_off.begin(), G.pg_off.end(), sb->pg_off);
    std::copy(G.pg_tgt.begin(), G.pg_tgt.end(), sb->pg_tgt);
    std::copy(G.grp_off.begin(), G.grp_off.end(), sb->grp_off);
    std::copy(G.grp_mem.begin(), G.grp_mem.end(), sb->grp_mem);
    std::copy(G.cons_grp.begin(), G.cons_grp.end(), sb->cons_grp);
    for (size_t g = 0; g < G.grp_init.size(); ++g)
        sb->grp_target[g] = G.grp_init[g] * releases_per_producer;
    return MLP_OK;
}

// ------------------------------------------------------------------------------------------
// Host model of the protocol: `threads` host threads play the persistent CTAs and run the
// kernel's protocol steps on std::atomic state, with the kernel's tables and arithmetic:
//   - every thread takes its run's epoch from a launch counter it adds 1 to at its start, has a
//     static first ticket (its own index) and takes the rest from a ticket counter, in stage
//     order; first-stage tickets map to tiles through raster_tile(rg);
//   - scoreboard groups from scoreboard_groups() (merged per rg row panels, members column by
//     column), each waiting for grp_init x R releases per run, R = releases one producer tile
//     makes (split-K slices x epilogue warps on the device);
//   - a finished tile makes R releases, each after writing its own part of the tile's output:
//     one acq_rel add of +1 on every group it feeds (on the device: fence.acq_rel.gpu + a
//     relaxed add, the PTX form of a release RMW); the add that completes the run's target,
//     run_target(init, epoch), reserves the group's queue slots on the tail and stores the
//     members there with relaxed stores, tagged with the epoch (a queue-free boundary, one group
//     or no more consumer tiles than threads, pushes nothing: its consumer slot q is the q-th
//     member of the groups in group order, as on the device);
//   - a consumer ticket polls its queue slot with relaxed loads until this run's entry lands,
//     then acquires the named tile's group counter until it reaches the run's target, and only
//     then reads the producers' output (plain, non-atomic reads: a missing happens-before edge is
//     a data race that ThreadSanitizer reports, and a stale value fails the run);
//   - a stage may split each tile into k-slices that run as items of their own (the device's
//     slices on separate clusters): slice j of a tile is the ticket after slice j-1, makes R / S
//     of the tile's releases, and first exchanges partial sums with its siblings: each of its
//     releases writes its own partial rows and adds 1 to the tile's exchange counter (acq_rel),
//     then the slice acquires that counter until it holds this run's S x R/S adds and reads the
//     siblings' rows (plain reads again).  Siblings wait on one another, so such a stage must fit
//     one wave (items <= threads), as on the device;
//   - nothing is reset between three back-to-back runs (epochs 0, 1, 2): scoreboard counters,
//     the exchange counters, the ticket, the queue tails and the launch counter accumulate, and
//     each run reads its own share of them relative to its epoch (protocol.h).
// ------------------------------------------------------------------------------------------
namespace {

struct ModelBoundary {
    std::vector<int32_t> off, tgt, init;
    mlpc::DepGroups grp;
    std::vector<int32_t> target;                 // releases per run, per group
    std::vector<std::vector<int32_t>> in;        // consumer -> its producers
    std::vector<std::atomic<uint32_t>> count;    // one per group, accumulating over runs
    std::vector<std::atomic<uint64_t>> queue;
    std::atomic<uint32_t> tail{0};
    std::vector<uint32_t> data;                  // producer output: R parts per producer tile
    bool queue_free = false;                     // consumers skip the queue (as on the device)
};

}  // namespace

extern "C" mlp_status mlp_protocol_model_slices(int32_t num_gemms, int32_t tiles_m, const int32_t *tiles_n,
                                                const int32_t *slices, int32_t raster_group,
                                                int32_t releases_per_tile, int32_t threads, uint64_t seed,
                                                int32_t drop_tile, int32_t drop_exchange, uint32_t timeout_ms,
                                                int32_t *order_out)
{
    if (num_gemms < 1 || num_gemms > MLP_MAX_GEMMS || tiles_m < 1 || !tiles_n || threads < 1 || threads > 512 ||
        raster_group < 0 || releases_per_tile < 1 || releases_per_tile > 64)
        return MLP_ERR_INVALID_ARG;
    const int S = num_gemms;
    const int32_t R = releases_per_tile;
    int32_t X[MLP_MAX_GEMMS];   // k-slices per tile, each an item of its own
    for (int s = 0; s < S; ++s) {
        X[s] = slices ? slices[s] : 1;
        if (tiles_n[s] < 1 || X[s] < 1 || R % X[s] != 0)
            return MLP_ERR_INVALID_ARG;
        // siblings wait on one another, so a sliced stage must fit one wave of threads
        if (X[s] > 1 && static_cast<int64_t>(tiles_m) * tiles_n[s] * X[s] > threads)
            return MLP_ERR_INVALID_ARG;
    }
    if (drop_exchange >= 0 && (X[0] == 1 || drop_exchange >= tiles_m * tiles_n[0]))
        return MLP_ERR_INVALID_ARG;
    int32_t base[MLP_MAX_GEMMS + 1], ibase[MLP_MAX_GEMMS + 1];   // per stage: first tile, first item (ticket)
    base[0] = ibase[0] = 0;
    for (int s = 0; s < S; ++s) {
        base[s + 1] = base[s] + tiles_m * tiles_n[s];
        ibase[s + 1] = ibase[s] + tiles_m * tiles_n[s] * X[s];
    }
    const int32_t total = base[S], items = ibase[S];
    // the slices' exchange: one partial per (tile, slice, release) and one counter per tile
    std::vector<std::vector<uint32_t>> part(static_cast<size_t>(S));
    std::vector<std::vector<std::atomic<uint32_t>>> xcount(static_cast<size_t>(S));
    for (int s = 0; s < S; ++s)
        if (X[s] > 1) {
            part[s].assign(static_cast<size_t>(tiles_m) * tiles_n[s] * R, 0u);
            xcount[s] = std::vector<std::atomic<uint32_t>>(static_cast<size_t>(tiles_m) * tiles_n[s]);
            for (auto &c : xcount[s])
                c.store(0);
        }

    std::vector<ModelBoundary> bd(S > 1 ? S - 1 : 0);
    for (int b = 0; b + 1 < S; ++b) {
        // tiles as unit cells: a tiles_m x tiles_n[b] producer grid, tiles_m x tiles_n[b+1] consumers
        ModelBoundary &B = bd[b];
        const int64_t nnz = mlp_deps_build(tiles_m, tiles_n[b], tiles_n[b + 1], 1, 1, 1, 1, nullptr, nullptr, 0, nullptr);
        B.off.resize(static_cast<size_t>(tiles_m) * tiles_n[b] + 1);
        B.tgt.resize(static_cast<size_t>(nnz));
        B.init.resize(static_cast<size_t>(tiles_m) * tiles_n[b + 1]);
        mlp_deps_build(tiles_m, tiles_n[b], tiles_n[b + 1], 1, 1, 1, 1, B.off.data(), B.tgt.data(), nnz, B.init.data());
        const int32_t P = static_cast<int32_t>(B.off.size() - 1), C = static_cast<int32_t>(B.init.size());
        B.grp = mlpc::scoreboard_groups(B.off.data(), B.tgt.data(), P, C, tiles_n[b + 1], raster_group);
        for (int32_t v : B.grp.grp_init)
            B.target.push_back(v * R);
        B.in.assign(static_cast<size_t>(C), {});
        for (int32_t p = 0; p < P; ++p)
            for (int32_t e = B.off[p]; e < B.off[p + 1]; ++e)
                B.in[static_cast<size_t>(B.tgt[e])].push_back(p);
        B.count = std::vector<std::atomic<uint32_t>>(B.grp.grp_init.size());
        B.queue = std::vector<std::atomic<uint64_t>>(static_cast<size_t>(C));
        for (auto &c : B.count)
            c.store(0);
        for (auto &q : B.queue)
            q.store(0);
        B.data.assign(static_cast<size_t>(P) * R, 0u);
        // one group, or no more consumer tiles than threads (each consumer gets a thread of its own)
        B.queue_free = B.grp.grp_init.size() == 1 || C <= threads;
    }

    std::atomic<uint32_t> ticket{0}, seq{0}, status{0};
    std::atomic<uint64_t> launches{0};
    // per tile: the first start and the last end over its slices, and how many slices ran
    std::vector<std::atomic<uint32_t>> start_seq(total), end_seq(total), runs(total);
    std::atomic<int32_t> order_pos{0};
    const auto timeout = std::chrono::milliseconds(timeout_ms ? timeout_ms : 2000);
    auto fail = [&](uint32_t code) {
        uint32_t z = 0;
        status.compare_exchange_strong(z, code);
    };

    for (uint32_t epoch = 0; epoch < 3; ++epoch) {
        for (int32_t i = 0; i < total; ++i) {
            start_seq[i].store(UINT32_MAX);
            end_seq[i].store(0);
            runs[i].store(0);
        }
        auto worker = [&](int tid) {
            std::mt19937_64 rng(seed * 7919u + static_cast<uint64_t>(tid) * 104729u + epoch);
            std::uniform_int_distribution<int> delay(0, 40);
            const uint32_t run = mlpc::epoch_of_launch(launches.fetch_add(1, std::memory_order_relaxed),
                                                       static_cast<uint32_t>(threads));
            if (run != epoch) {
                fail(MLP_ERR_DEVICE_STATE);
                return;
            }
            for (int32_t t = tid; t < items;
                 t = threads + static_cast<int32_t>(mlpc::run_relative(ticket.fetch_add(1, std::memory_order_relaxed),
                                                                       run, static_cast<uint32_t>(items)))) {
                const int32_t s = mlpc::stage_of_ticket(ibase, t);
                // a sliced stage's item is one k-slice of one tile; its siblings are the neighbouring tickets
                const int32_t local = (t - ibase[s]) / X[s], slice = (t - ibase[s]) % X[s];
                const auto t0 = std::chrono::steady_clock::now();
                auto expired = [&]() {
                    if (status.load(std::memory_order_relaxed) != 0)
                        return true;
                    if (std::chrono::steady_clock::now() - t0 > timeout) {
                        fail(MLP_ERR_TIMEOUT);
                        return true;
                    }
                    std::this_thread::yield();
                    return false;
                };
                int32_t tile;
                if (s == 0) {
                    tile = mlpc::raster_tile(local, tiles_m, tiles_n[0], raster_group);
                } else {
                    ModelBoundary &B = bd[s - 1];
                    // relaxed polls of the queue slot: the entry only names the tile (a queue-free
                    // boundary has none: slot q is the q-th member of the groups in group order)
                    uint64_t v;
                    if (B.queue_free)
                        v = mlpc::queue_entry(epoch, B.grp.grp_mem[static_cast<size_t>(local)]);
                    else
                        while (!mlpc::queue_entry_ready(v = B.queue[local].load(std::memory_order_relaxed), epoch))
                            if (expired())
                                return;
                    tile = mlpc::queue_entry_tile(v);
                    if (tile < 0 || tile >= tiles_m * tiles_n[s]) {
                        fail(MLP_ERR_BAD_TILE);
                        return;
                    }
                    // the acquire that makes every producer's output visible
                    const int32_t g = B.grp.cons_grp[static_cast<size_t>(tile)];
                    const uint32_t want = mlpc::run_target(B.target[static_cast<size_t>(g)], epoch);
                    while (!mlpc::count_reached(B.count[static_cast<size_t>(g)].load(std::memory_order_acquire), want))
                        if (expired())
                            return;
                    for (int32_t p : B.in[static_cast<size_t>(tile)])
                        for (int32_t r = 0; r < R; ++r)
                            if (B.data[static_cast<size_t>(p) * R + r] != epoch + 1u) {
                                fail(MLP_ERR_DEVICE_STATE);
                                return;
                            }
                }
                const int32_t id = base[s] + tile;
                uint32_t st = seq.fetch_add(1) + 1, cur = start_seq[id].load();
                while (st < cur && !start_seq[id].compare_exchange_weak(cur, st)) {
                }
                std::this_thread::sleep_for(std::chrono::microseconds(delay(rng)));
                const int32_t Rs = R / X[s];   // releases this item makes (its epilogue warps)
                if (X[s] > 1) {
                    // the slices' exchange: each release writes its own partial rows, then adds 1 to the
                    // tile's counter (on the device: fence.acq_rel.gpu + a relaxed add); every slice waits
                    // for all S x Rs adds of this run and reads its siblings' rows of the same release
                    std::vector<uint32_t> &P = part[s];
                    for (int32_t w = 0; w < Rs; ++w) {
                        P[(static_cast<size_t>(tile) * X[s] + slice) * Rs + w] = epoch + 1u;
                        if (s == 0 && tile == drop_exchange && slice == X[s] - 1)
                            continue;   // fault injection: the partial lands, its add never comes
                        xcount[s][static_cast<size_t>(tile)].fetch_add(1, std::memory_order_acq_rel);
                    }
                    const uint32_t want = mlpc::run_target(static_cast<uint32_t>(R), epoch);
                    while (!mlpc::count_reached(xcount[s][static_cast<size_t>(tile)].load(std::memory_order_acquire), want))
                        if (expired())
                            return;
                    for (int32_t w = 0; w < Rs; ++w)
                        for (int32_t q = 0; q < X[s]; ++q)
                            if (q != slice && P[(static_cast<size_t>(tile) * X[s] + q) * Rs + w] != epoch + 1u) {
                                fail(MLP_ERR_DEVICE_STATE);
                                return;
                            }
                }
                runs[id].fetch_add(1);
                const uint32_t en = seq.fetch_add(1) + 1;
                cur = end_seq[id].load();
                while (en > cur && !end_seq[id].compare_exchange_weak(cur, en)) {
                }
                if (order_out && epoch == 0)
                    order_out[order_pos.fetch_add(1)] = (s << 24) | tile;
                if (s + 1 >= S)
                    continue;
                ModelBoundary &B = bd[s];
                const mlpc::DepGroups &G = B.grp;
                for (int32_t r = slice * Rs; r < (slice + 1) * Rs; ++r) {   // this item's epilogue warps
                    B.data[static_cast<size_t>(tile) * R + r] = epoch + 1u;   // this release's rows
                    if (s == 0 && tile == drop_tile)
                        continue;   // fault injection: the stores land, the releases never come
                    if (delay(rng) < 8)
                        std::this_thread::yield();
                    for (int32_t e = G.pg_off[tile]; e < G.pg_off[tile + 1]; ++e) {
                        const int32_t g = G.pg_tgt[e];
                        const uint32_t old = B.count[static_cast<size_t>(g)].fetch_add(1, std::memory_order_acq_rel);
                        if (B.queue_free ||
                            !mlpc::release_completes(old, mlpc::run_target(B.target[static_cast<size_t>(g)], epoch)))
                            continue;   // (a queue-free boundary pushes nothing)
                        const int32_t m0 = G.grp_off[g], n = G.grp_off[g + 1] - m0;
                        const uint32_t q0 = mlpc::run_relative(B.tail.fetch_add(static_cast<uint32_t>(n), std::memory_order_relaxed),
                                                               run, static_cast<uint32_t>(B.queue.size()));
                        for (int32_t i = 0; i < n; ++i)
                            B.queue[q0 + i].store(mlpc::queue_entry(epoch, G.grp_mem[m0 + i]), std::memory_order_relaxed);
                    }
                }
            }
        };
        std::vector<std::thread> pool;
        for (int i = 0; i < threads; ++i)
            pool.emplace_back(worker, i);
        for (auto &th : pool)
            th.join();
        if (status.load() != 0)
            return static_cast<mlp_status>(status.load());
        // every slice of every tile ran once, after all of its producers' slices had finished
        for (int s = 0; s < S; ++s)
            for (int32_t i = base[s]; i < base[s + 1]; ++i)
                if (runs[i].load() != static_cast<uint32_t>(X[s]))
                    return MLP_ERR_DEVICE_STATE;
        for (int b = 0; b + 1 < S; ++b) {
            for (int32_t p = 0; p + 1 < static_cast<int32_t>(bd[b].off.size()); ++p)
                for (int32_t e = bd[b].off[p]; e < bd[b].off[p + 1]; ++e)
                    if (!(end_seq[base[b] + p].load() < start_seq[base[b + 1] + bd[b].tgt[e]].load()))
                        return MLP_ERR_DEVICE_STATE;
            // every counter sits exactly at this run's target: nothing lost, nothing counted twice
            for (size_t g = 0; g < bd[b].count.size(); ++g)
                if (bd[b].count[g].load() != mlpc::run_target(bd[b].target[g], epoch))
                    return MLP_ERR_DEVICE_STATE;
        }
        for (int s = 0; s < S; ++s)
            for (auto &c : xcount[s])
                if (c.load() != mlpc::run_target(static_cast<uint32_t>(R), epoch))
                    return MLP_ERR_DEVICE_STATE;
    }
    return MLP_OK;
}

extern "C" mlp_status mlp_protocol_model(int32_t num_gemms, int32_t tiles_m, const int32_t *tiles_n,
                                         int32_t raster_group, int32_t releases_per_tile, int32_t threads,
                                         uint64_t seed, int32_t drop_tile, uint32_t timeout_ms, int32_t *order_out)
{
    return mlp_protocol_model_slices(num_gemms, tiles_m, tiles_n, nullptr, raster_group, releases_per_tile, threads,
                                     seed, drop_tile, -1, timeout_ms, order_out);
}
