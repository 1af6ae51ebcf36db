// drive_host.cpp -- exercises the library's host-only code (dependency builder, grouped
// scoreboard tables, host-thread protocol model) under a sanitizer: AddressSanitizer +
// UndefinedBehaviorSanitizer, or ThreadSanitizer for the protocol model's threads.  Exit status
// 0 when every call behaves as the header says and the sanitizer reports nothing.
#include <cstdint>
#include <cstdio>
#include <vector>

#include "mlp_chain.h"

int main()
{
    int fails = 0;
    const int64_t shapes[3][7] = {{64, 256, 256, 64, 64, 128, 64}, {300, 384, 512, 128, 64, 128, 128},
                                  {2048, 8192, 8192, 128, 256, 128, 256}};
    for (const auto &d : shapes) {
        const int64_t P = ((d[0] + d[3] - 1) / d[3]) * ((d[1] + d[4] - 1) / d[4]);
        const int64_t C = ((d[0] + d[5] - 1) / d[5]) * ((d[2] + d[6] - 1) / d[6]);
        std::vector<int32_t> init(static_cast<size_t>(C));
        const int64_t nnz = mlp_deps_build(d[0], d[1], d[2], static_cast<int32_t>(d[3]), static_cast<int32_t>(d[4]),
                                           static_cast<int32_t>(d[5]), static_cast<int32_t>(d[6]), nullptr, nullptr, 0,
                                           init.data());
        std::vector<int32_t> off(static_cast<size_t>(P + 1)), tgt(static_cast<size_t>(nnz > 0 ? nnz : 1));
        fails += nnz < 0 || mlp_deps_build(d[0], d[1], d[2], static_cast<int32_t>(d[3]), static_cast<int32_t>(d[4]),
                                           static_cast<int32_t>(d[5]), static_cast<int32_t>(d[6]), off.data(), tgt.data(),
                                           nnz, init.data()) != nnz;
    }
    const int32_t tn2[2] = {4, 4}, tn4[4] = {3, 5, 2, 4}, tn3[3] = {3, 2, 3}, tn5[2] = {3, 2};
    for (uint64_t seed = 1; seed <= 3; ++seed) {
        std::vector<int32_t> order(64 * 16);
        fails += mlp_protocol_model(2, 4, tn2, 1, 4, 8, seed, -1, 2000, order.data()) != MLP_OK;
        fails += mlp_protocol_model(4, 3, tn4, 1, 16, 6, seed, -1, 2000, order.data()) != MLP_OK;
        fails += mlp_protocol_model(3, 17, tn3, 8, 8, 12, seed, -1, 2000, order.data()) != MLP_OK;   // merged groups
        fails += mlp_protocol_model(2, 4, tn5, 1, 4, 8, seed, -1, 2000, order.data()) != MLP_OK;    // queue-free groups
    }
    fails += mlp_protocol_model(2, 2, tn2, 1, 4, 4, 5, 1, 200, nullptr) != MLP_ERR_TIMEOUT;   // withheld release
    // k-slices on separate threads: each slice exchanges its partials with its siblings through a
    // per-tile counter before its own releases
    const int32_t sl_first[2] = {2, 1}, sl_cons[2] = {1, 4}, sl3[3] = {2, 4, 1}, tn8[2] = {8, 4}, tn3b[3] = {4, 2, 4};
    for (uint64_t seed = 1; seed <= 3; ++seed) {
        std::vector<int32_t> order(64 * 16);
        fails += mlp_protocol_model_slices(2, 2, tn2, sl_first, 1, 8, 16, seed, -1, -1, 2000, order.data()) != MLP_OK;
        fails += mlp_protocol_model_slices(2, 1, tn8, sl_cons, 1, 8, 16, seed, -1, -1, 2000, order.data()) != MLP_OK;
        fails += mlp_protocol_model_slices(3, 2, tn3b, sl3, 2, 8, 16, seed, -1, -1, 2000, order.data()) != MLP_OK;
    }
    fails += mlp_protocol_model_slices(2, 2, tn2, sl_first, 1, 8, 16, 7, -1, 3, 200, nullptr) !=
             MLP_ERR_TIMEOUT;   // withheld exchange add
    for (int32_t rg : {1, 3, 8}) {   // the grouped scoreboard tables, sizes first
        mlp_scoreboard sb{};
        fails += mlp_scoreboard_build(1000, 512, 384, 128, 128, 64, rg, 4, &sb) != MLP_OK;
        std::vector<int32_t> pg_off(sb.producers + 1), pg_tgt(sb.edges), grp_off(sb.groups + 1), grp_mem(sb.consumers),
            grp_target(sb.groups), cons_grp(sb.consumers);
        sb.pg_off = pg_off.data();
        sb.pg_tgt = pg_tgt.data();
        sb.grp_off = grp_off.data();
        sb.grp_mem = grp_mem.data();
        sb.grp_target = grp_target.data();
        sb.cons_grp = cons_grp.data();
        fails += mlp_scoreboard_build(1000, 512, 384, 128, 128, 64, rg, 4, &sb) != MLP_OK;
        fails += grp_off[sb.groups] != sb.consumers;
    }
    std::printf("host driver: %d failures\n", fails);
    return fails != 0;
}
