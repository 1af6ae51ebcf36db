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

// ------------------------------------------------------------------------------------------
// Host model of the protocol: `threads` host threads play the persistent CTAs.  Each takes
// tickets in stage order; first-stage tickets map to tiles through raster_tile(); later-stage
// tickets poll the matching work-queue slot (acquire) until this run's entry lands; a tile's
// "work" is a seeded random sleep; its epilogue decrements (acq_rel) the counters of its
// consumers and the decrement that reaches zero re-arms the counter and pushes (release).
// Two runs are played back to back (epochs 0 and 1) to exercise the re-arm and epoch tags.
// ------------------------------------------------------------------------------------------
namespace {

struct ModelBoundary {
    std::vector<int32_t> off, tgt, init;
    mlpc::DepGroups grp;
    std::vector<std::atomic<uint32_t>> count;   // one per group
    std::vector<std::atomic<uint64_t>> queue;
    std::atomic<uint32_t> tail{0};
};

}  // namespace

extern "C" mlp_status mlp_protocol_model(int32_t num_gemms, int32_t tiles_m, const int32_t *tiles_n,
                                         int32_t threads, uint64_t seed, int32_t drop_tile,
                                         uint32_t timeout_ms, int32_t *order_out)
{
    if (num_gemms < 1 || num_gemms > MLP_MAX_GEMMS || tiles_m < 1 || !tiles_n || threads < 1 || threads > 512)
        return MLP_ERR_INVALID_ARG;
    for (int s = 0; s < num_gemms; ++s)
        if (tiles_n[s] < 1)
            return MLP_ERR_INVALID_ARG;
    const int S = num_gemms;
    int32_t base[MLP_MAX_GEMMS + 1];
    base[0] = 0;
    for (int s = 0; s < S; ++s)
        base[s + 1] = base[s] + tiles_m * tiles_n[s];
    const int32_t total = base[S];

    std::vector<ModelBoundary> bd(S > 1 ? S - 1 : 0);
    for (int b = 0; b + 1 < S; ++b) {
        // tiles as unit cells: a tiles_m x tiles_n[b] producer grid, tiles_m x tiles_n[b+1] consumers
        const int64_t nnz = mlp_deps_build(tiles_m, tiles_n[b], tiles_n[b + 1], 1, 1, 1, 1, nullptr, nullptr, 0, nullptr);
        bd[b].off.resize(static_cast<size_t>(tiles_m) * tiles_n[b] + 1);
        bd[b].tgt.resize(static_cast<size_t>(nnz));
        bd[b].init.resize(static_cast<size_t>(tiles_m) * tiles_n[b + 1]);
        mlp_deps_build(tiles_m, tiles_n[b], tiles_n[b + 1], 1, 1, 1, 1, bd[b].off.data(), bd[b].tgt.data(), nnz,
                       bd[b].init.data());
        bd[b].grp = mlpc::build_groups(bd[b].off.data(), bd[b].tgt.data(),
                                       static_cast<int32_t>(bd[b].off.size() - 1),
                                       static_cast<int32_t>(bd[b].init.size()));
        bd[b].count = std::vector<std::atomic<uint32_t>>(bd[b].grp.grp_init.size());
        bd[b].queue = std::vector<std::atomic<uint64_t>>(bd[b].init.size());
        for (size_t i = 0; i < bd[b].grp.grp_init.size(); ++i)
            bd[b].count[i].store(static_cast<uint32_t>(bd[b].grp.grp_init[i]));
        for (size_t i = 0; i < bd[b].init.size(); ++i)
            bd[b].queue[i].store(0);
    }

    std::atomic<uint32_t> ticket{0}, seq{0}, status{0};
    std::vector<std::atomic<uint32_t>> start_seq(total), end_seq(total), runs(total);
    std::atomic<int32_t> order_pos{0};
    const auto timeout = std::chrono::milliseconds(timeout_ms ? timeout_ms : 2000);

    for (uint32_t epoch = 0; epoch < 2; ++epoch) {
        for (int32_t i = 0; i < total; ++i) {
            start_seq[i].store(0);
            end_seq[i].store(0);
            runs[i].store(0);
        }
        auto worker = [&](int tid) {
            std::mt19937_64 rng(seed * 7919u + static_cast<uint64_t>(tid) * 104729u + epoch);
            std::uniform_int_distribution<int> delay(0, 40);
            while (true) {
                const int32_t t = static_cast<int32_t>(ticket.fetch_add(1, std::memory_order_relaxed));
                if (t >= total)
                    return;
                const int32_t s = mlpc::stage_of_ticket(base, t);
                const int32_t local = t - base[s];
                int32_t tile;
                if (s == 0) {
                    tile = mlpc::raster_tile(local, tiles_m, tiles_n[0], 1);
                } else {
                    const auto t0 = std::chrono::steady_clock::now();
                    uint64_t v;
                    while (true) {
                        v = bd[s - 1].queue[local].load(std::memory_order_acquire);
                        if (mlpc::queue_entry_ready(v, epoch))
                            break;
                        if (status.load(std::memory_order_relaxed) != 0)
                            return;
                        if (std::chrono::steady_clock::now() - t0 > timeout) {
                            uint32_t z = 0;
                            status.compare_exchange_strong(z, MLP_ERR_TIMEOUT);
                            return;
                        }
                        std::this_thread::yield();
                    }
                    tile = mlpc::queue_entry_tile(v);
                    if (tile < 0 || tile >= tiles_m * tiles_n[s]) {
                        uint32_t z = 0;
                        status.compare_exchange_strong(z, MLP_ERR_BAD_TILE);
                        return;
                    }
                }
                const int32_t id = base[s] + tile;
                start_seq[id].store(seq.fetch_add(1) + 1);
                std::this_thread::sleep_for(std::chrono::microseconds(delay(rng)));
                runs[id].fetch_add(1);
                end_seq[id].store(seq.fetch_add(1) + 1);
                if (order_out && epoch == 0)
                    order_out[order_pos.fetch_add(1)] = (s << 24) | tile;
                if (s + 1 < S && !(s == 0 && tile == drop_tile)) {
                    ModelBoundary &b = bd[s];
                    const mlpc::DepGroups &G = b.grp;
                    for (int32_t e = G.pg_off[tile]; e < G.pg_off[tile + 1]; ++e) {
                        const int32_t g = G.pg_tgt[e];
                        const uint32_t old = b.count[g].fetch_sub(1, std::memory_order_acq_rel);
                        if (old == 1u) {
                            b.count[g].store(static_cast<uint32_t>(G.grp_init[g]), std::memory_order_relaxed);
                            const int32_t n = G.grp_off[g + 1] - G.grp_off[g];
                            const uint32_t slot0 = b.tail.fetch_add(static_cast<uint32_t>(n), std::memory_order_relaxed);
                            for (int32_t i = 0; i < n; ++i)
                                b.queue[slot0 + i].store(mlpc::queue_entry(epoch, G.grp_mem[G.grp_off[g] + i]),
                                                         std::memory_order_release);
                        }
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
        // every tile ran once, after all of its producers had finished
        for (int32_t i = 0; i < total; ++i)
            if (runs[i].load() != 1)
                return MLP_ERR_DEVICE_STATE;
        for (int b = 0; b + 1 < S; ++b)
            for (int32_t p = 0; p + 1 < static_cast<int32_t>(bd[b].off.size()); ++p)
                for (int32_t e = bd[b].off[p]; e < bd[b].off[p + 1]; ++e)
                    if (!(end_seq[base[b] + p].load() < start_seq[base[b + 1] + bd[b].tgt[e]].load()))
                        return MLP_ERR_DEVICE_STATE;
        // what the last CTA out does on the device
        ticket.store(0);
        for (auto &b : bd)
            b.tail.store(0);
    }
    return MLP_OK;
}
