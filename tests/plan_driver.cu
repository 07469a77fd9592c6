// Test driver (host code only): prints the fp32 schedule planners' choices
// (splits, spread, tile shape, K chunks; the workspace split "priced lower"
// against the cluster split alone; stream-K's CTAs and whether stream-K is the
// workspace entry's choice over both) for the shapes given on the command
// line as M,N,K triples, for a 152-SM GPU whose
// cluster-split CTAs fit 76 clusters of 2, 36 of 4 and 15 of 8 at one CTA per
// SM (the occupancy the library queries on GB300); with "pair" first, the
// CTA-pair kernel's K-split choice instead, with "longk" first the K-split of
// the 128-wide streaming tensor-core kernels. Built and run by
// tests/test_plan_host.py; no GPU is needed.
#include <cstdio>
#include <cstdlib>
#include <string>

#include "kernels.h"

int main(int argc, char **argv)
{
    if (argc > 1 && std::string(argv[1]) == "longk") {
        // longk tiles K sms ...: the K-split of the 128-wide streaming kernels
        for (int i = 2; i + 2 < argc; i += 3)
            std::printf("%s %s %s splits %d\n", argv[i], argv[i + 1], argv[i + 2],
                        rtm::long_k_splits(std::atoll(argv[i]), std::atoll(argv[i + 1]),
                                           std::atoi(argv[i + 2])));
        return 0;
    }
    if (argc > 1 && std::string(argv[1]) == "pair") {
        // pair ntiles pairs kblocks c_vec ...: the CTA-pair kernel's first split tile
        for (int i = 2; i + 3 < argc; i += 4)
            std::printf("%s %s %s %s split_from %lld\n", argv[i], argv[i + 1], argv[i + 2], argv[i + 3],
                        rtm::pair_split_from(std::atoll(argv[i]), std::atoi(argv[i + 1]),
                                             std::atoi(argv[i + 2]), std::atoi(argv[i + 3]) != 0));
        return 0;
    }
    const int sms = 152;
    const int resident[3] = {76, 36, 15};
    for (int i = 1; i + 2 < argc; i += 3) {
        const int M = std::atoi(argv[i]), N = std::atoi(argv[i + 1]), K = std::atoi(argv[i + 2]);
        double cluster_est = 0;
        const rtm::SplitK c = rtm::sgemm_cluster_plan(M, N, K, sms, resident, &cluster_est);
        const rtm::SplitK w = rtm::sgemm_splitk_plan(M, N, K, sms);
        const double w_est = rtm::sgemm_workspace_estimate(M, N, K, sms, w);
        const bool ws_wins = w.splits > 1 && !(cluster_est < w_est);
        const rtm::TailPlan t = rtm::sgemm_tail_plan(M, N, K, sms);
        const rtm::SimtTile tile = rtm::simt_resolve_tile(c.tile, M, N);
        double sk_est = 0;
        const int sk = rtm::sgemm_streamk_plan(M, N, K, sms, &sk_est);
        const bool sk_wins = sk > 0 && sk_est < cluster_est && (!ws_wins || sk_est < w_est);
        std::printf("%d %d %d cluster %d %d workspace %d %d tail %lld %d tile %d %d "
                    "chunks %d %d %d streamk %d %d\n",
                    M, N, K, c.splits, c.spread ? 1 : 0, w.splits, ws_wins ? 1 : 0,
                    t.plain_tiles, t.tail.splits, tile.m, tile.n, c.kchunk, w.kchunk,
                    t.tail.kchunk, sk, sk_wins ? 1 : 0);
    }
    return 0;
}
