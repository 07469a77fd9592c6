// Host-side schedules of the tensor-core kernels, kept apart from the kernels
// so the choices can be tested without a GPU: which 256 x 256 tiles of the
// CTA-pair kernel (gemm_tc2.cu) split K in two, and the K-split of the kernels
// that stream one operand through 128-wide tiles (gemm_tc_t.cu,
// gemm_tc_any_t.cu).
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

// 0 unless K has at least 32 64-deep blocks and the `tiles` fit on the SMs at
// once; otherwise the largest S (1, 2, 4 or 8) that keeps at most one CTA per
// SM and at least 16 blocks per CTA. Whole blocks, so that K = 4094 splits
// like K = 4096 (64 x 4094 x 4094 on the load-and-swizzle kernel: S 2 -> 4,
// 26.9 -> 17.9 us).
int long_k_splits(long long tiles, long long K, int sms)
{
    const long long kblocks = (K + 63) / 64;
    if (kblocks < 32 || tiles > sms)
        return 0;
    int splits = 1;
    while (splits < 8 && tiles * splits * 2 <= sms && kblocks / (splits * 2) >= 16)
        splits *= 2;
    return splits;
}

} // namespace rtm
