// Host-side schedule of the CTA-pair tensor-core kernel (gemm_tc2.cu): which
// 256 x 256 tiles split K in two. Kept apart from the kernel so the choice can
// be tested without a GPU.
#include "kernels.h"

namespace rtm {

// A tile split in two adds each K half into a zeroed C with TMA reduce-adds
// (two partials: the same sum in either order). Split when C rows are 16-byte
// aligned (the TMA-store epilogue), both halves keep at least 32 K-blocks, and
// either all tiles fill at most half the pairs (256 x 8192 x 8192: 45.1 ->
// 37.2 us), or the persistent loop's last round is at most half full: its
// tiles then run as two half-length units each (8192^3: 13 rounds of 76 tiles,
// then 36 tiles on 72 pairs for half a round; 579.1 -> 569.9 us).
long long pair_split_from(long long ntiles, int pairs, int kblocks, bool c_vec)
{
    if (!c_vec || kblocks < 64 || pairs <= 0)
        return ntiles;
    if (2 * ntiles <= pairs)
        return 0;
    const long long tail = ntiles % pairs;
    if (ntiles > pairs && tail > 0 && 2 * tail <= pairs)
        return ntiles - tail;
    return ntiles;
}

} // namespace rtm
