// Host-side schedule of the SIMT FP32 product: how many K chunks (split-K)
// a product with few C tiles is cut into. Kept apart from the kernels so a
// change of schedule leaves the kernel sources untouched.
#include "kernels.h"

namespace rtm {

using namespace simt_tiles;

// Schedule model for the split: an SM retires CTA-slices (one BK-deep slice
// of one tile) at about the same rate whether one or two CTAs are resident (a
// lone CTA runs about twice as fast), so T equal CTAs of c slices each take
// about ceil(T / SMs) * c slice-times. A split into s partial products adds a
// reduction launch (about 2 slice-times) and, per partial product, writing and
// re-reading M x N floats (about M * N / 2.1e6 slice-times at HBM bandwidth).
// The plan minimises that estimate; a sweep of every split on GB300 (shapes
// from 256^3 to 2048^2 x 8192) put its choice within 1.2 % of the fastest on
// average. Products with more tiles than SMs are not split (every SM already
// has work; the gain measured there was 4-9 % at most), nor are splits kept
// that the model prices within 3 % of the plain product.
SplitK sgemm_splitk_plan(int M, int N, int K, int sm_count)
{
    SplitK p{1, K};
    const int tile_n = N <= kNarrowN ? kNarrowN : kTileN;
    const int tile_m = M <= kShortTileM ? kShortTileM : kTileM;
    const long long tiles = (long long)((M + tile_m - 1) / tile_m) * ((N + tile_n - 1) / tile_n);
    if (sm_count <= 0 || tiles > sm_count)
        return p;
    const long long kslices = (K + kSliceK - 1) / kSliceK;
    // Tiles of half the area: less work per slice.
    const double slice_time = (tile_n == kNarrowN || tile_m == kShortTileM) ? 0.8 : 1.0;
    const double per_partial = (double)M * N / 2.1e6;
    const double plain = (double)((tiles + sm_count - 1) / sm_count) * kslices * slice_time;
    double best = plain;
    for (int s = 2; s <= 32; ++s) {
        const long long chunk = (kslices + s - 1) / s;
        const int splits = (int)((kslices + chunk - 1) / chunk);
        if (splits < 2)
            continue;
        const double est = (double)((tiles * splits + sm_count - 1) / sm_count) * chunk * slice_time +
                           2.0 + per_partial * splits;
        if (est < best) {
            best = est;
            p = SplitK{splits, (int)(chunk * kSliceK)};
        }
    }
    if (p.splits > 1 && best > 0.97 * plain)
        p = SplitK{1, K};
    return p;
}

} // namespace rtm
