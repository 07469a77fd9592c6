"""CPU tests of the schedule planners (host code in sgemm_plan.cu and
tc_plan.cu): a driver built from tests/plan_driver.cu prints each planner's
choice for a 152-SM GB300, and the choices the GB300 sweeps justified are
checked here: which fp32 products split K over clusters and into how many
CTAs, when the workspace split is priced below the cluster split, when the
ragged last wave of a larger product is split, which tile shape a product
takes (256 x 64 and 64 x 256 for tall and short ones, 64-row and 64-column
tiles for products with few tiles), and which tiles of the bf16 CTA-pair
kernel split K in two."""

import os
import shutil
import subprocess

import pytest

import register_tiled_matrix_gb300 as rtm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "register_tiled_matrix_gb300", "csrc")

# (M, N, K): (cluster splits, spread, workspace splits, workspace priced lower,
#             unsplit tiles before the tail, tail splits, CTA tile rows x columns)
EXPECT = {
    (256, 256, 256): (4, 0, 8, 0, 0, 1, (64, 64)),       # 10.3 -> 8.2 us against 128 x 128 split 8
    (384, 384, 384): (4, 0, 12, 0, 0, 1, (64, 64)),      # 16.4 -> 8.8 us
    (512, 512, 512): (4, 0, 8, 0, 0, 1, (64, 128)),      # 18.5 -> 12.4 us
    (256, 256, 1024): (8, 1, 32, 1, 0, 1, (64, 128)),    # 18.5 -> 12.5 us
    (1024, 1024, 1024): (4, 0, 2, 0, 0, 1, (128, 128)),  # 52.8 us split 4, 55.4 with the workspace
    (1000, 1000, 999): (4, 0, 2, 0, 0, 1, (128, 128)),
    (512, 512, 8192): (8, 0, 9, 1, 0, 1, (64, 128)),     # 182.2 -> 115.0 us; the workspace wins
    (64, 4096, 8192): (8, 0, 19, 1, 0, 1, (64, 128)),    # 64-row tiles: the workspace wins
    (2048, 1024, 1024): (1, 0, 1, 0, 0, 1, (128, 128)),  # 128 tiles: split was no faster
    (4096, 4096, 4096): (1, 0, 1, 0, 0, 1, (128, 128)),  # 3 waves + 112 tiles: tail left alone
    (4097, 3001, 1023): (1, 0, 1, 0, 608, 4, (128, 128)),  # 608 tiles + a 184-tile tail split
    (2304, 2304, 4096): (1, 0, 1, 0, 304, 4, (128, 128)),  # one wave + 20 tiles
    (2048, 1536, 1024): (1, 0, 1, 0, 0, 4, (128, 128)),  # 192 tiles, under two waves
    (2048, 2304, 512): (1, 0, 1, 0, 0, 1, (128, 128)),   # 4-slice chunks, 95 % of the slots
    (300, 3000, 700): (2, 0, 2, 0, 0, 1, (128, 128)),
    # Tall, narrow (N <= 64): 256 x 64 tiles against 128 x 64, fastest on GB300 in
    # each row (us): 117.6 for 128 x 64 split 4 against 106.1 here; 230.4 (split 8)
    # against 196.7; 227.4 against 198.8; 62.7 here against 100.5; 2048 x 64 x 8192
    # on 64 x 64 tiles 77.1 through gemm_f32 against 105.2 on 256 x 64.
    (8192, 64, 4096): (8, 0, 7, 0, 0, 1, (256, 64)),
    (16384, 64, 4096): (4, 0, 8, 0, 0, 1, (256, 64)),
    (8192, 64, 8192): (8, 0, 7, 0, 0, 1, (256, 64)),
    (4096, 64, 4096): (8, 0, 19, 0, 0, 1, (128, 64)),    # 16 tall tiles would pack two to an SM
    (2048, 64, 8192): (8, 0, 19, 1, 0, 1, (64, 64)),
    (32768, 64, 512): (1, 0, 1, 0, 0, 1, (256, 64)),     # 128 tall tiles unsplit
    (200, 64, 8192): (8, 1, 32, 1, 0, 1, (64, 64)),
    (131072, 16, 64): (1, 0, 1, 0, 0, 1, (128, 64)),     # two K slices: 128 x 64 tiles
    # 33 to 64 rows: 64 x 256 tiles against 64 x 128, fastest on GB300 in each
    # row (us): 220.0 for 64 x 128 split 4 against 199.0 here; 114.7 (split 2)
    # against 104.5; 434.9 (split 8) against 385.5; 120.4 against 111.3; 64.5
    # here against 108.8 (16 wide tiles); 20.6 here against 30.9; 64 x 2048 x
    # 8192 on 64 x 64 tiles 76.6 through gemm_f32 against 105.2 on 64 x 256.
    (64, 8192, 8192): (8, 0, 7, 0, 0, 1, (64, 256)),
    (64, 16384, 2048): (4, 0, 1, 0, 0, 1, (64, 256)),
    (64, 16384, 8192): (4, 0, 7, 0, 0, 1, (64, 256)),
    (40, 8192, 4096): (8, 0, 7, 0, 0, 1, (64, 256)),
    (48, 4096, 4096): (8, 0, 19, 0, 0, 1, (64, 128)),
    (64, 4096, 1024): (4, 0, 4, 0, 0, 1, (64, 128)),
    (64, 2048, 8192): (8, 0, 19, 1, 0, 1, (64, 64)),
    (64, 65536, 512): (1, 0, 1, 0, 0, 1, (64, 256)),     # 256 wide tiles unsplit
}


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out = str(tmp_path_factory.mktemp("plan") / "plan_driver")
    cmd = [nvcc, "-std=c++17", "-O2", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "plan_driver.cu"), os.path.join(CSRC, "sgemm_plan.cu"),
           os.path.join(CSRC, "tc_plan.cu"), "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    return out


def test_planner_choices(driver):
    args = [str(x) for shape in EXPECT for x in shape]
    r = subprocess.run([driver, *args], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    got = {}
    for line in r.stdout.splitlines():
        f = line.split()
        got[(int(f[0]), int(f[1]), int(f[2]))] = (int(f[4]), int(f[5]), int(f[7]), int(f[8]),
                                                   int(f[10]), int(f[11]), (int(f[13]), int(f[14])))
    for shape, want in EXPECT.items():
        assert got[shape] == want, (shape, got[shape], want)


# Stream-K (gemm_f32_ws, TMA-fed 128 x 128 tiles): (CTAs, chosen over the
# cluster and workspace splits). Measured on GB300 (us, graph replay, scalar
# loop): 1024^3 48.5 against 49.8 for the cluster split; 512^2 x 8192 83.9
# against 92.5 for the workspace split; 640^2 x 4096 68.1 against 94.3;
# 2048 x 1024 x 1024 88.3 against 93.6 unsplit; 256^2 x 2048 keeps the
# workspace split (13.2 against 15.1); K % 4 != 0 cannot be loaded by TMA.
STREAMK_EXPECT = {
    (1024, 1024, 1024): (304, 1),
    (512, 512, 8192): (304, 1),
    (640, 640, 4096): (304, 1),
    (2048, 1024, 1024): (304, 1),
    (256, 256, 2048): (152, 0),
    (1000, 1000, 999): (0, 0),
    (200, 300, 4096): (152, 0),
    (64, 4096, 8192): (0, 0),      # 64-row tiles: not a stream-K shape
    (4096, 4096, 4096): (0, 0),    # more tiles than SMs
}


def test_streamk_choices(driver):
    args = [str(x) for shape in STREAMK_EXPECT for x in shape]
    r = subprocess.run([driver, *args], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    got = {}
    for line in r.stdout.splitlines():
        f = line.split()
        got[(int(f[0]), int(f[1]), int(f[2]))] = (int(f[20]), int(f[21]))
    for shape, want in STREAMK_EXPECT.items():
        assert got[shape] == want, (shape, got[shape], want)


def _shape_grid():
    dims = [1, 7, 33, 64, 65, 100, 128, 129, 200, 256, 257, 500, 1000, 1024, 2047, 4096, 8192,
            20000]
    ks = [1, 31, 32, 33, 96, 97, 200, 1000, 4096, 8193]
    return [(m, n, k) for m in dims for n in dims for k in ks]


def test_planner_invariants_over_a_grid(driver):
    """Every plan the fp32 planners make over a grid of 3240 shapes is one the
    launchers accept: a cluster size of 1, 2, 4 or 8 that divides the tile
    height, a tile shape the kernel is built for (256 x 64 only for N <= 64,
    64 x 256 only for M <= 64), K chunks of whole 32-deep slices that cover K
    with none empty, one CTA per SM only for clusters of 8, at most 32
    workspace chunks, and a tail split only after whole waves of 304 slots."""
    shapes = _shape_grid()
    args = [str(x) for shape in shapes for x in shape]
    r = subprocess.run([driver, *args], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    lines = r.stdout.splitlines()
    assert len(lines) == len(shapes)
    shapes_ok = {(128, 128), (128, 64), (64, 128), (64, 64), (256, 64), (64, 256)}

    def chunks_ok(splits, chunk, K):
        if splits == 1:
            return True
        return chunk % 32 == 0 and splits * chunk >= K and (splits - 1) * chunk < K

    for line in lines:
        f = line.split()
        M, N, K = int(f[0]), int(f[1]), int(f[2])
        cs, spread, ws, plain_tiles, ts = int(f[4]), int(f[5]), int(f[7]), int(f[10]), int(f[11])
        tm, tn = int(f[13]), int(f[14])
        cchunk, wchunk, tchunk = int(f[16]), int(f[17]), int(f[18])
        where = f"{M}x{N}x{K}: {line}"
        assert cs in (1, 2, 4, 8) and tm % cs == 0, where
        assert (tm, tn) in shapes_ok, where
        assert tm != 256 or N <= 64, where
        assert tn != 256 or M <= 64, where
        assert chunks_ok(cs, cchunk, K), where
        assert spread == 0 or cs == 8, where
        assert 1 <= ws <= 32 and chunks_ok(ws, wchunk, K), where
        assert ts in (1, 4), where
        if ts == 4:
            assert plain_tiles % 304 == 0 and chunks_ok(ts, tchunk, K) and M > 64 and N > 64, where


# CTA-pair kernel (bf16/fp16, M > 128): (tiles, resident pairs, 64-deep K blocks,
# C rows on 16-byte boundaries) -> first tile whose K is split in two.
PAIR_EXPECT = {
    (1024, 76, 128, 1): 988,   # 8192^3: 13 rounds + 36 tiles split for half a round
    (256, 76, 64, 1): 228,     # 4096^3: 3 rounds + 28 tiles
    (576, 76, 64, 1): 576,     # 6144^2 x 4096: last round 44 tiles, more than half full
    (128, 76, 128, 1): 128,    # 1024 x 8192^2: last round 52 tiles
    (32, 76, 128, 1): 0,       # 256 x 8192^2: every tile split
    (38, 76, 64, 1): 0,        # exactly half the pairs
    (39, 76, 64, 1): 39,       # more than half, one round: unsplit
    (32, 76, 32, 1): 32,       # K = 2048: halves too short
    (1024, 76, 128, 0): 1024,  # C rows not 16-byte aligned: no reduce-add epilogue
}


def test_pair_split_choices(driver):
    args = ["pair"] + [str(x) for key in PAIR_EXPECT for x in key]
    r = subprocess.run([driver, *args], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    got = {tuple(int(x) for x in l.split()[:4]): int(l.split()[-1]) for l in r.stdout.splitlines()}
    assert got == PAIR_EXPECT


def test_pair_split_invariants_over_a_grid(driver):
    """For every (tiles, pairs, K-blocks, aligned C) on a grid: the split tiles
    are a suffix of the tile order; none split without aligned C or with K
    halves under 32 blocks; either every tile splits (the tiles fill at most
    half the pairs) or only the last round's tiles do, and then that round is
    at most half full, so its 2 x tail half-length units fit in one round."""
    keys = [(t, p, kb, cv) for t in list(range(1, 200)) + [255, 256, 576, 988, 1024, 4096]
            for p in (1, 38, 76) for kb in (1, 32, 63, 64, 65, 128) for cv in (0, 1)]
    args = ["pair"] + [str(x) for key in keys for x in key]
    r = subprocess.run([driver, *args], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    got = {tuple(int(x) for x in l.split()[:4]): int(l.split()[-1]) for l in r.stdout.splitlines()}
    assert len(got) == len(keys)
    for (t, p, kb, cv), sf in got.items():
        where = (t, p, kb, cv, sf)
        assert 0 <= sf <= t, where
        if not cv or kb < 64:
            assert sf == t, where
        split = t - sf
        if split and sf:
            assert sf % p == 0 and 2 * split <= p, where   # the last round only
        if split and not sf:
            assert 2 * t <= p, where                       # every tile, all at once


# (tiles, K, SMs): K-split of the 128-wide streaming tensor-core kernels
# (transposed short products, tall narrow products; TMA-fed or load-and-swizzle).
LONGK_EXPECT = {
    (64, 8190, 152): 2,     # 128 x 8190 x 8190: 64 column tiles, S = 4 would need 256 SMs
    (64, 8192, 152): 2,
    (32, 4094, 152): 4,     # 64 x 4094 x 4094: 64 K-blocks like K = 4096
    (32, 4096, 152): 4,
    (32, 4032, 152): 2,     # 63 K-blocks: 15 per CTA at S = 4
    (32, 4033, 152): 4,     # 64 K-blocks (the last one ragged)
    (8, 8192, 152): 8,      # 64 x 1024 x 8192: 16 blocks per CTA at S = 8
    (8, 16384, 152): 8,     # at most 8 CTAs per cluster
    (79, 2050, 152): 1,     # 16 x 10002 x 2050: two CTAs per tile would need 158 SMs
    (152, 8192, 152): 1,    # one tile per SM
    (153, 8192, 152): 0,    # more tiles than SMs: not this kernel
    (8, 1984, 152): 0,      # 31 K-blocks: too short
    (8, 1985, 152): 2,      # 32 K-blocks (the last one ragged): 16 per CTA at S = 2
    (8, 2048, 152): 2,
    (1, 3001, 152): 2,      # 47 blocks: 23 per CTA at S = 2, 11 at S = 4
}


def test_long_k_split_choices(driver):
    args = ["longk"] + [str(x) for key in LONGK_EXPECT for x in key]
    r = subprocess.run([driver, *args], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    got = {tuple(int(x) for x in l.split()[:3]): int(l.split()[-1]) for l in r.stdout.splitlines()}
    assert got == LONGK_EXPECT


def test_long_k_split_invariants_over_a_grid(driver):
    """For every (tiles, K) on a grid: no split below 32 K-blocks or with more
    tiles than SMs; otherwise S is 1, 2, 4 or 8, fits one CTA per SM, leaves
    every CTA at least 16 K-blocks (when S > 1), and is the largest such; and
    K values with the same number of 64-deep blocks get the same S."""
    sms = 152
    keys = [(t, k, sms) for t in (1, 2, 5, 8, 19, 20, 38, 39, 64, 76, 77, 100, 152, 153)
            for k in list(range(1900, 2200, 7)) + [4031, 4032, 4033, 4094, 4096, 8190, 8192,
                                                   16383, 16384, 65536]]
    args = ["longk"] + [str(x) for key in keys for x in key]
    r = subprocess.run([driver, *args], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    got = {tuple(int(x) for x in l.split()[:3]): int(l.split()[-1]) for l in r.stdout.splitlines()}
    assert len(got) == len(keys)
    by_blocks = {}
    for (t, k, n), s in got.items():
        kb = (k + 63) // 64
        by_blocks.setdefault((t, kb), set()).add(s)
        if kb < 32 or t > n:
            assert s == 0, (t, k, s)
            continue
        assert s in (1, 2, 4, 8), (t, k, s)
        assert t * s <= n, (t, k, s)
        assert s == 1 or kb // s >= 16, (t, k, s)
        assert s == 8 or t * 2 * s > n or kb // (2 * s) < 16, (t, k, s)  # largest
    assert all(len(v) == 1 for v in by_blocks.values())


def test_schedule_kinds_cover_the_planner_outcomes():
    """Every outcome above has a name in the binding's schedule kinds."""
    assert set(rtm.F32_KINDS.values()) >= {"tiles", "tiles+cluster-split", "tiles+workspace-split",
                                            "column-strips", "tiles+tail-cluster-split",
                                            "tall-tiles", "tall-tiles+cluster-split",
                                            "wide-tiles", "wide-tiles+cluster-split"}
