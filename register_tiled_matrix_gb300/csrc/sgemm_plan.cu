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

namespace {

// Comparable run-time estimates (in slice-times) for the split schedules,
// fitted to a sweep of 18 shapes on GB300 (256^3 to 64 x 8192 x 8192, every
// cluster size and the workspace plan): each wave of CTAs costs its chunk plus
// kCtaOverhead slice-times (start-up, pipeline fill, epilogue); two CTAs
// sharing an SM finish a wave in kPackedRate x twice a lone CTA's time.
constexpr double kCtaOverhead = 0.7;
constexpr double kPackedRate = 0.9;
constexpr double kClusterReduce = 1.0;  // per wave: partials parked, cluster barriers, DSMEM adds

struct ShapeCost {
    long long tiles, kslices;
    double slice_time;
};

// Slice-times of one slice of each tile shape. 256 x 64 and 64 x 256 take
// 1.35, fitted on GB300 to tall, narrow products (8192 x 64 x 4096 to 16384 x
// 64 x 8192) and to products of 40 to 64 rows (64 x 2048 x 8192 to 64 x 16384
// x 8192), K split 1 to 8 ways: the same area as a 128 x 128 tile, but with
// 16 x 4 or 4 x 16 outputs per thread the loop reads shared memory 5 times
// per 64 FMA against 4. A 128 x 64 or 64 x 128 tile's slice (8 x 4 or 4 x 8
// per thread, 6 reads per 64 FMA) takes 0.8 for half the area, a 64 x 64
// tile's (4 x 4 per thread, 8 reads per 64 FMA) 0.45 for a quarter: with it
// the plan picked the fastest tile and split measured on GB300 for 256^3,
// 384^3, 512^3 and 256 x 256 x 1024.
ShapeCost shape_cost(int M, int N, int K, SimtTile shape = SimtTile{})
{
    const SimtTile t = simt_resolve_tile(shape, M, N);
    ShapeCost c;
    c.tiles = (long long)((M + t.m - 1) / t.m) * ((N + t.n - 1) / t.n);
    c.kslices = (K + kSliceK - 1) / kSliceK;
    const int area = t.m * t.n;
    c.slice_time = t.m == kTallTileM || t.n == kWideTileN ? 1.35
                   : area == kTileM * kTileN              ? 1.0
                   : area == kTileM * kNarrowN            ? 0.8
                                                          : 0.45;
    return c;
}

// `ctas` CTAs of `chunk` slices each; `alone`: every CTA has an SM to itself.
double waves_time(const ShapeCost &c, long long ctas, long long chunk, int sms, bool alone,
                  double per_wave)
{
    const double waves = alone ? 1.0 : kPackedRate * (double)((ctas + sms - 1) / sms < 2
                                                                  ? 2
                                                                  : (ctas + sms - 1) / sms);
    return waves * ((chunk + kCtaOverhead) * c.slice_time + per_wave);
}

} // namespace

double sgemm_workspace_estimate(int M, int N, int K, int sm_count, const SplitK &plan)
{
    const ShapeCost c = shape_cost(M, N, K);
    if (plan.splits <= 1 || sm_count <= 0)
        return 1e300;
    const long long chunk = (plan.kchunk + kSliceK - 1) / kSliceK;
    const long long ctas = c.tiles * plan.splits;
    return waves_time(c, ctas, chunk, sm_count, ctas <= sm_count, 0.0) + 2.0 +
           (double)M * N / 2.1e6 * plan.splits;
}

// The split over one cluster's CTAs: S in {2, 4, 8} (S must divide the tile
// height), no reduction launch and no partial products in HBM; the partial
// tiles are added through distributed shared memory. Left to itself the GPU
// places the CTAs of a cluster of 8 two to an SM (measured on GB300: 512 x
// 512 x 8192 at S = 8 ran each slice 1.9x slower than at S = 4), so when every
// CTA can have an SM of its own the plan asks for one CTA per SM (`spread`),
// provided all the clusters fit at once that way; otherwise it prices the
// split as packed two to an SM.
namespace {

// The cluster plan for one tile shape; *est_out: its estimate (the plain
// product's when not split, priced as waves of CTAs two to an SM where there
// are more tiles than SMs).
SplitK cluster_plan_for(const ShapeCost &c, int K, int sm_count, const int (&resident_spread)[3],
                        double *est_out)
{
    SplitK p{1, K};
    const bool few = c.tiles <= sm_count;
    const double plain = waves_time(c, c.tiles, c.kslices, sm_count, few, 0.0);
    *est_out = plain;
    if (!few)
        return p;
    double best = plain;
    for (int i = 0, s = 2; s <= 8; ++i, s *= 2) {
        const long long chunk = (c.kslices + s - 1) / s;
        if ((long long)s * chunk - c.kslices >= chunk)
            break;  // a chunk would be empty: K too short for this many
        const long long ctas = c.tiles * s;
        // Clusters of 2 and 4 land one CTA per SM by themselves when they fit.
        const bool spread = ctas <= sm_count && c.tiles <= resident_spread[i];
        const bool alone = ctas <= sm_count && (spread || s < 8);
        const double est = waves_time(c, ctas, chunk, sm_count, alone, kClusterReduce);
        if (est < best) {
            best = est;
            p = SplitK{s, (int)(chunk * kSliceK), spread && s == 8};
        }
    }
    if (p.splits > 1 && best > 0.97 * plain)
        p = SplitK{1, K};
    *est_out = p.splits > 1 ? best : plain;
    return p;
}

} // namespace

SplitK sgemm_cluster_plan(int M, int N, int K, int sm_count, const int (&resident_spread)[3],
                          double *est_out)
{
    if (est_out)
        *est_out = 1e300;
    if (sm_count <= 0)
        return SplitK{1, K};
    double est = 0;
    SplitK p = cluster_plan_for(shape_cost(M, N, K), K, sm_count, resident_spread, &est);
    // Other tile shapes, split or not, where they price lower: tall, narrow
    // (256 x 64) or short (64 x 256) tiles; and for products with few tiles,
    // 64-row and 64-column tiles, whose smaller CTAs spread the work over
    // more SMs. Tall, unsplit, on GB300: 65536 x 64 x 256 59.5 -> 53.4 us,
    // 65536 x 64 x 2048 441.8 -> 389.9 us, 131072 x 64 x 1024 the same; with K
    // of one or two slices the longer CTAs lost (131072 x 16 x 64 30.9 -> 33.0
    // us), so K of three slices or fewer keeps the standard tiles. Smaller
    // tiles, against 128 x 128 split over clusters: 256^3 10.3 -> 8.2 us
    // (64 x 64, split 4), 384^3 16.4 -> 8.8 (64 x 64, split 4), 512^3 18.5 ->
    // 12.4 (64 x 128, split 4), 256 x 256 x 1024 18.5 -> 12.5 (64 x 128, split 8).
    const SimtTile std_tile = simt_standard_tile(M, N);
    SimtTile alts[4];
    int n_alt = 0;
    if (K > 3 * kSliceK) {
        if (N <= kNarrowN && M > kTileM)
            alts[n_alt++] = SimtTile{kTallTileM, kNarrowN};
        else if (M <= kShortTileM && N > kNarrowN)
            alts[n_alt++] = SimtTile{kShortTileM, kWideTileN};
    }
    if (M > kShortTileM)
        alts[n_alt++] = SimtTile{kShortTileM, std_tile.n};
    if (N > kNarrowN)
        alts[n_alt++] = SimtTile{std_tile.m, kNarrowN};
    if (M > kShortTileM && N > kNarrowN)
        alts[n_alt++] = SimtTile{kShortTileM, kNarrowN};
    for (int i = 0; i < n_alt; ++i) {
        const ShapeCost c = shape_cost(M, N, K, alts[i]);
        const bool tall_or_wide = alts[i].m == kTallTileM || alts[i].n == kWideTileN;
        if (!tall_or_wide && c.tiles > sm_count)
            continue;  // smaller tiles only where they all fit at once
        double est_alt = 0;
        SplitK t = cluster_plan_for(c, K, sm_count, resident_spread, &est_alt);
        if (est_alt < est) {
            t.tile = alts[i];
            p = t;
            est = est_alt;
        }
    }
    if (est_out)
        *est_out = est;
    return p;
}

// Stream-K over 128 x 128 tiles (sgemm_tma.cu), for products with at most one
// tile per SM: the CTAs take equal ranges of the tiles x K-slices iterations,
// so every SM works the same time instead of the cluster split's whole CTAs
// that leave some SMs with two and others with one; split tiles are added by
// a fixup kernel. Two CTAs per SM where that leaves each at least 4 slices,
// else one. Priced in slice-times like the other schedules (0.9 x twice a lone
// CTA's time for two per SM), x 0.95 for the packed-FMA loop, plus a fixed
// cost for the prologue, the partial tiles and the fixup (kStreamKFixed),
// fitted on GB300 to 1024^3, 512^2 x 8192, 640^2 x 4096 and 1280^2 x 1024
// (4.1-5.1; 48.5, 83.9, 68.1, 71.1 us at 304 CTAs against 49.8, 92.5 (the
// workspace split), 94.3 and 74.2 before). Only for K % 4 == 0 and N % 4 == 0:
// the TMA loads need rows on 16-byte boundaries.
constexpr double kStreamKFixed = 4.4;
constexpr double kPackedLoop = 0.95;

int sgemm_streamk_plan(int M, int N, int K, int sm_count, double *est)
{
    if (est)
        *est = 1e300;
    if (M <= kShortTileM || N <= kNarrowN || sm_count <= 0 || K % 4 != 0 || N % 4 != 0)
        return 0;
    const long long tiles = (long long)((M + kTileM - 1) / kTileM) * ((N + kTileN - 1) / kTileN);
    if (tiles > sm_count)
        return 0;
    const long long iters = tiles * ((K + kSliceK - 1) / kSliceK);
    if (iters >= (1LL << 31))
        return 0;
    const bool two = iters >= 8LL * sm_count;
    const int ctas = two ? 2 * sm_count : (int)(iters < sm_count ? iters : sm_count);
    const long long chunk = (iters + ctas - 1) / ctas;
    if (est)
        *est = (two ? kPackedRate * 2.0 : 1.0) * (double)chunk * kPackedLoop + kStreamKFixed;
    return ctas;
}

// Products with more 128 x 128 tiles than SMs: the whole waves of CTA slots
// (2 per SM) run as the plain product, and the ragged last wave can run as a
// second launch with K split over clusters of 4 CTAs. Measured on GB300 (plain
// against prefix + split tail): 4097 x 3001 x 1023 601.9 -> 550.8 us, 3072 x 2048
// x 4096 1015.5 -> 955.1, 2048 x 2048 x 4096 679.2 -> 622.9, 6144^2 x 2048
// 2611.1 -> 2550.8; but 4096^3 2310.8 -> 2357.0, 8192^2 x 2048 and 5000^2 x 1000
// slower too: after several full waves a tail of at most one tile per SM
// already runs one CTA per SM and the second launch loses the overlap of the
// last wave with the one before. So the tail is split only when it holds more
// tiles than SMs or the product has fewer than two full waves, the tail fills
// at most 85 % of the slots (2048 x 2304 x 512, 288 tiles: 90.0 -> 110.8 us) and
// every chunk keeps at least 8 K-slices. Products of fewer than two waves
// gain most: 2048 x 1536 x 1024 173.5 -> 147.6 us, 2304^2 x 4096 (304 + 20
// tiles) 997.4 -> 779.2 us.
TailPlan sgemm_tail_plan(int M, int N, int K, int sm_count)
{
    TailPlan t{0, SplitK{1, K}};
    if (M <= kShortTileM || N <= kNarrowN || sm_count <= 0)
        return t;  // the tail schedule is measured for 128 x 128 tiles only
    const long long tiles = (long long)((M + kTileM - 1) / kTileM) * ((N + kTileN - 1) / kTileN);
    const long long slots = 2LL * sm_count;
    if (tiles <= sm_count)
        return t;  // sgemm_cluster_plan's case
    const long long plain = tiles / slots * slots;
    const long long tail = tiles - plain;
    const long long kslices = (K + kSliceK - 1) / kSliceK;
    constexpr int S = 4;
    const long long chunk = (kslices + S - 1) / S;
    if (tail == 0 || !(tail > sm_count || tiles < 2 * slots) || tail * 100 > slots * 85 ||
        chunk < 8 || (long long)S * chunk - kslices >= chunk)
        return t;
    t.plain_tiles = plain;
    t.tail = SplitK{S, (int)(chunk * kSliceK)};
    return t;
}

} // namespace rtm
