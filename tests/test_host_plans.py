"""Host-side work plans of the split-K kernels, restated here and checked
against the scratch sizes the library reports (no GPU needed: without a
device the library plans for 148 SMs; with one, for the device's count).

Every workspace starts with a fixed 64 KiB area holding the arrival counters
(no kernel's partials overlap it, so GEMMs of different shapes may share a
workspace).  Swap-AB GEMM (weights as the MMA's 128-row operand, 256-wide
k-blocks):
every CTA takes floor(tiles/grid) whole tiles, the other tiles are cut into
one contiguous run of (tile, k-block) pairs per CTA, and when those shared
tiles have fewer k-blocks than there are CTAs one round of whole tiles joins
them.  W4A16 tensor-core GEMM (the TMEM kernel, given its workspace): tiles of
128 weight rows x 16/32/64 tokens per CTA, or 256 weight rows x 128 tokens
per CTA pair, split as the swap-AB kernel without clusters (whole tiles
last, over the clusters); its scratch is the counter area, the fp32
partials [clusters][fragment slots][pair CTA][tokens padded][128] when a
tile is shared,
the f16 activations [m][k] and the fp32 row scales [m], each rounded up to
256 bytes.  The whole-MLP decode kernel plans both of its GEMM phases the
swap-AB way on one grid (the smaller of the SM count and either phase's
k-block count).  The rule that every CTA between a shared tile's first and
last owner contributes to it is checked on the restated partition, and so is
the kernels' reduction bookkeeping: the walk of each CTA (its run, then its
whole tiles), the first/last owner formula and each contributor's partial
slot, written out as the kernels compute them.
"""
import math

import pytest

import nvfp4_quantized_dense_gb300 as nv
from nvfp4_quantized_dense_gb300 import build as nvbuild


@pytest.fixture(scope="module")
def lib():
    nvbuild.build()
    return nv.load()


def sm_count():
    import torch
    if torch.cuda.is_available():
        return torch.cuda.get_device_properties(0).multi_processor_count
    return 148


# Every split-K workspace starts with a fixed 64 KiB counter area that no
# kernel's partials overlap, so calls of different shapes can share one.
COUNTER_AREA = 64 * 1024


def r256(b):
    return (b + 255) // 256 * 256


def swapab_cluster(tiles, kbt, sms):
    """Cluster size of the cluster split (1: not used): at most 8 CTAs per
    tile and one per k-block, at least 90 % of the SMs busy, every cluster
    resident at once (without a device: as many as the SMs allow)."""
    cl = min(8, sms // max(tiles, 1), kbt)
    while cl >= 2 and tiles * cl * 10 >= sms * 9:
        if sms // cl >= tiles:
            return cl
        cl -= 1
    return 1


def swapab_plan(m, n, k, sms, clusters=True):
    """clusters=False: the split the kernel uses when no cluster split fits."""
    nt = 16 if m <= 16 else 32 if m <= 32 else 64
    tiles, kbt = math.ceil(n / 128), math.ceil(k / 256)
    cl = swapab_cluster(tiles, kbt, sms) if clusters else 1
    if cl > 1:
        return dict(nt=nt, tiles=tiles, kbt=kbt, grid=tiles * cl, whole=0, split=0, ws=0, cl=cl)
    grid = min(tiles * kbt, sms)
    whole = tiles // grid
    split = tiles - whole * grid
    if whole > 0 and split > 0 and split * kbt < grid:
        whole, split = whole - 1, split + grid
    units = split * kbt
    per = math.ceil(units / grid)
    maxfrag = math.ceil(per / kbt) + 1
    shared = units % grid != 0 or (units // grid) % kbt != 0
    ws = COUNTER_AREA + grid * maxfrag * nt * 128 * 4 if shared else 0
    return dict(nt=nt, tiles=tiles, kbt=kbt, grid=grid, whole=whole, split=split, ws=ws, cl=1)


def mixed_plan(tiles, kbt, sms, nt):
    """The mixed split (whole tiles last): grid, whole tiles per CTA, split
    tiles, fragment slots and the partials' bytes (0 when no tile is
    shared)."""
    grid = min(tiles * kbt, sms)
    whole = tiles // grid
    split = tiles - whole * grid
    if whole > 0 and split > 0 and split * kbt < grid:
        whole, split = whole - 1, split + grid
    units = split * kbt
    maxfrag = math.ceil(math.ceil(units / grid) / kbt) + 1
    shared = units > 0 and (units % grid != 0 or (units // grid) % kbt != 0)
    return dict(grid=grid, whole=whole, split=split, maxfrag=maxfrag,
                part=grid * maxfrag * nt * 128 * 4 if shared else 0)


def w4a16_tiles(m, n, k, sms):
    """The W4A16 TMEM kernel's tiling: 256-wide k-blocks; token tiles of
    16/32/64 (one CTA, 128 weight rows) or 128 (a CTA pair, 256 weight rows);
    tiles = weight tiles x token tiles over the SMs' clusters."""
    nt = 16 if m <= 16 else 32 if m <= 32 else 64 if m <= 64 else 128
    cl = 2 if nt == 128 else 1
    tiles = math.ceil(n / (128 * cl)) * math.ceil(m / nt)
    return nt, cl, tiles, math.ceil(k / 256), sms // cl


def w4a16_ws(m, n, k, sms):
    """The W4A16 TMEM kernel's scratch: counters, the partials of the mixed
    split (one [tokens][128] slot per CTA of a cluster), the f16 activations
    [m][k] and the fp32 row scales [m], each rounded up to 256 bytes."""
    nt, cl, tiles, kbt, units = w4a16_tiles(m, n, k, sms)
    pl = mixed_plan(tiles, kbt, units, nt)
    return COUNTER_AREA + r256(pl["part"] * cl) + r256(m * k * 2) + r256(m * 4)


SWAP_CASES = [
    (1, 34816, 5120),     # decode gate_up H5120: 272 tiles -> one whole tile per CTA + shared tiles
    (16, 34816, 5120),
    (1, 5120, 17408),     # decode down: 40 tiles, all shared (clusters of 3 would leave 32 SMs idle)
    (16, 7168, 18432),    # DeepSeek-shaped down: 56 tiles, all shared
    (3, 2560, 2048),      # 20 tiles -> clusters of 7 CTAs, one tile each
    (40, 6144, 1280),     # 48 tiles -> clusters of 3
    (64, 36864, 7168),    # DeepSeek-shaped gate_up
    (8, 7168, 18432),
    (1, 20480, 512),      # 160 tiles of 2 k-blocks: the shared k-blocks would be fewer than CTAs
    (5, 39168, 768),
    (33, 384, 1024), (4, 1024, 256), (17, 128, 128),
]


@pytest.mark.parametrize("m,n,k", SWAP_CASES)
def test_swapab_scratch_matches_plan(lib, m, n, k):
    pl = swapab_plan(m, n, k, sm_count())
    assert nv.nvfp4_workspace_bytes(m, n, k, nv.ALGO_TC_SWAPAB) == pl["ws"]
    assert nv.nvfp4_workspace_bytes(m, n, k) == pl["ws"]          # AUTO picks swap-AB up to 64 tokens


@pytest.mark.parametrize("m,n,k", SWAP_CASES)
@pytest.mark.parametrize("sms", [148, 152, 7])
def test_swapab_partition_contributors_are_contiguous(m, n, k, sms):
    pl = swapab_plan(m, n, k, sms)
    if pl["cl"] > 1:
        # cluster split: the cl CTAs of tile t cover its k-blocks in order,
        # each at least one, as the kernel cuts them (j * kbt / cl)
        cl, kbt = pl["cl"], pl["kbt"]
        assert 2 <= cl <= 8 and pl["grid"] == pl["tiles"] * cl <= sms and 10 * pl["grid"] >= 9 * sms
        cuts = [kbt * j // cl for j in range(cl + 1)]
        assert cuts[0] == 0 and cuts[-1] == kbt and all(b > a for a, b in zip(cuts, cuts[1:]))
        return
    grid, kbt, split = pl["grid"], pl["kbt"], pl["split"]
    assert split + pl["whole"] * grid == pl["tiles"]
    units = split * kbt
    starts = [j * units // grid for j in range(grid + 1)]
    owner = {}
    for j in range(grid):
        for u in range(starts[j], starts[j + 1]):
            owner[u] = j
    assert len(owner) == units
    if units and split:
        assert units >= grid, "a CTA without a shared k-block would break the arrival count"
    for t in range(split):
        cs = sorted({owner[u] for u in range(t * kbt, (t + 1) * kbt)})
        assert cs == list(range(cs[0], cs[-1] + 1))
        # every contributor after the first starts its run inside the tile
        # (its partial sits in fragment slot 0)
        for c in cs[1:]:
            assert starts[c] // kbt == t


def mlp_decode_ws(m, hid, inter, sms):
    """Scratch of the whole-MLP decode kernel: sync words, h-slice counters
    and both phases' tile counters, then each phase's fp32 partials (every
    phase uses the swap-AB mixed partition on the same grid)."""
    nt = 16 if m <= 16 else 32 if m <= 32 else 64
    tiles = [2 * inter // 128, hid // 128]
    kbt = [math.ceil(hid / 256), math.ceil(inter / 256)]
    grid = min(tiles[0] * kbt[0], tiles[1] * kbt[1], sms)
    assert 256 + (kbt[1] + tiles[0] + tiles[1]) * 4 <= COUNTER_AREA
    ws = COUNTER_AREA
    for g in range(2):
        whole = tiles[g] // grid
        split = tiles[g] - whole * grid
        if whole > 0 and split > 0 and split * kbt[g] < grid:
            whole, split = whole - 1, split + grid
        per = math.ceil(split * kbt[g] / grid)
        ws += r256(grid * (math.ceil(per / kbt[g]) + 1) * nt * 128 * 4)
    return ws


@pytest.mark.parametrize("m,hid,inter", [(1, 5120, 17408), (16, 5120, 17408), (64, 7168, 18432), (4, 256, 512),
                                         (33, 1024, 2048), (1, 128, 64)])
def test_mlp_decode_scratch_matches_plan(lib, m, hid, inter):
    assert nv.nvfp4_mlp_decode_workspace_bytes(m, hid, inter) == mlp_decode_ws(m, hid, inter, sm_count())


@pytest.mark.parametrize("m,n,k", [(1, 34816, 5120), (16, 34816, 5120), (16, 5120, 17408), (64, 384, 2048),
                                   (33, 128, 1024), (5, 96, 320), (128, 34816, 5120), (1024, 34816, 5120),
                                   (128, 5120, 17408), (1024, 5120, 17408), (300, 4096, 512)])
def test_w4a16_scratch_matches_plan(lib, m, n, k):
    assert nv.bf16_fp4_gemm_workspace_bytes(m, n, k, nv.ALGO_TC) == w4a16_ws(m, n, k, sm_count())


def _random_shapes(count, seed):
    import numpy as np
    g = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        m = int(g.integers(1, 65))
        n = int(g.integers(1, 400)) * 32
        k = int(g.integers(1, 300)) * 64
        out.append((m, n, k))
    return out


def test_swapab_scratch_matches_plan_random_shapes(lib):
    """The restated plan and the library agree on 300 random decode shapes
    (M 1..64, N multiples of 32 up to 12768, K multiples of 64 up to 19136)."""
    sms = sm_count()
    for m, n, k in _random_shapes(300, 11):
        assert nv.nvfp4_workspace_bytes(m, n, k, nv.ALGO_TC_SWAPAB) == swapab_plan(m, n, k, sms)["ws"], (m, n, k)


def test_swapab_partition_invariants_random_shapes():
    for m, n, k in _random_shapes(300, 12):
        for sms in (148, 152):
            pl = swapab_plan(m, n, k, sms, clusters=False)
            grid, kbt, split = pl["grid"], pl["kbt"], pl["split"]
            assert split + pl["whole"] * grid == pl["tiles"]
            units = split * kbt
            if units and split:
                assert units >= grid, (m, n, k, sms)


def test_w4a16_scratch_matches_plan_random_shapes(lib):
    sms = sm_count()
    for m, n, k in _random_shapes(300, 13):
        assert nv.bf16_fp4_gemm_workspace_bytes(m, n, k, nv.ALGO_TC) == w4a16_ws(m, n, k, sms), (m, n, k)


def _mixed_fragments(kbt, grid, whole, split_tiles, j):
    """The fragments CTA j walks under the swap-AB mixed partition: its run of
    the split units (start(j) = floor(j * U / grid)), then its whole tiles
    split_tiles + j*whole + [0, whole)."""
    units = split_tiles * kbt
    x, end = j * units // grid, (j + 1) * units // grid
    out = []
    while x < end:
        tile = x // kbt
        kb0 = x - tile * kbt
        kb1 = min(kbt, kb0 + (end - x))
        out.append((tile, kb0, kb1))
        x += kb1 - kb0
    for t in range(split_tiles + j * whole, split_tiles + (j + 1) * whole):
        out.append((t, 0, kbt))
    return out


@pytest.mark.parametrize("m,n,k", SWAP_CASES + [(1, 5120, 17408), (16, 36864, 7168), (64, 7168, 18432)])
@pytest.mark.parametrize("sms", [148, 152, 7])
def test_swapab_reduction_bookkeeping(m, n, k, sms):
    """Every (tile, k-block) is covered once; for a shared tile the owner of
    its first and last k-block (cta_of = ((x + 1) * grid - 1) // U, the
    inverse of start) bracket exactly the CTAs that hold a fragment of it;
    each contributor's partial slot (f_first for the first owner, 0 for the
    others) is its fragment's index in its own walk, below maxfrag."""
    pl = swapab_plan(m, n, k, sms, clusters=False)
    grid, kbt, whole, split = pl["grid"], pl["kbt"], pl["whole"], pl["split"]
    units = split * kbt
    maxfrag = (math.ceil(math.ceil(units / grid) / kbt) + 1) if units else 1
    seen = {}
    holders = {}
    for j in range(grid):
        for f, (tile, kb0, kb1) in enumerate(_mixed_fragments(kbt, grid, whole, split, j)):
            for kb in range(kb0, kb1):
                assert (tile, kb) not in seen
                seen[(tile, kb)] = j
            if tile < split:
                holders.setdefault(tile, []).append((j, f))
    assert len(seen) == pl["tiles"] * kbt
    cta_of = lambda x: ((x + 1) * grid - 1) // units
    start = lambda j: j * units // grid
    for tile, hs in holders.items():
        c_first, c_last = cta_of(tile * kbt), cta_of(tile * kbt + kbt - 1)
        assert [c for c, _ in hs] == list(range(c_first, c_last + 1))
        f_first = tile - start(c_first) // kbt
        for c, f in hs:
            slot = f_first if c == c_first else 0
            assert slot == f and slot < maxfrag, (tile, c, f, slot)


def test_swapab_reduction_bookkeeping_random_shapes():
    for m, n, k in _random_shapes(150, 14):
        for sms in (148, 152):
            test_swapab_reduction_bookkeeping(m, n, k, sms)


@pytest.mark.parametrize("m,n,k", [(1, 34816, 5120), (16, 34816, 5120), (16, 5120, 17408), (64, 384, 2048),
                                   (33, 128, 1024), (5, 96, 320), (64, 7168, 18432), (128, 5120, 17408),
                                   (1024, 5120, 17408)])
@pytest.mark.parametrize("sms", [148, 152, 7])
def test_w4a16_reduction_bookkeeping(m, n, k, sms):
    """The W4A16 TMEM kernel's mixed split (weight tiles x token tiles,
    whole tiles last) keeps the swap-AB split's invariants: every (tile,
    k-block) covered once, a shared tile's contributors contiguous, each
    contributor's partial slot its fragment's index below maxfrag."""
    nt, cl, tiles, kbt, units = w4a16_tiles(m, n, k, sms)
    pl = mixed_plan(tiles, kbt, units, nt)
    grid, whole, split = pl["grid"], pl["whole"], pl["split"]
    units = split * kbt
    seen, holders = set(), {}
    for j in range(grid):
        for f, (tile, kb0, kb1) in enumerate(_mixed_fragments(kbt, grid, whole, split, j)):
            for kb in range(kb0, kb1):
                assert (tile, kb) not in seen
                seen.add((tile, kb))
            if tile < split:
                holders.setdefault(tile, []).append((j, f))
    assert len(seen) == tiles * kbt
    for tile, hs in holders.items():
        c_first, c_last = ((tile * kbt + 1) * grid - 1) // units, ((tile * kbt + kbt) * grid - 1) // units
        assert [c for c, _ in hs] == list(range(c_first, c_last + 1))
        f_first = tile - (c_first * units // grid) // kbt
        for c, f in hs:
            assert (f_first if c == c_first else 0) == f < pl["maxfrag"]


def _kwalk(kbt, early, u0, u1):
    """The whole-MLP kernel's walk of the units [u0, u1) of one fragment,
    written out as the kernel steps it: the early units (u with
    floor((u+1)*early/kbt) > floor(u*early/kbt)) first, then the others;
    early unit number e is k-block e, the others follow after `early`."""
    out = []
    for pass_ in (0, 1):
        eb = u0 * early // kbt
        r = u0 * early - eb * kbt
        for u in range(u0, u1):
            is_early = r + early >= kbt
            e = eb
            if is_early:
                eb += 1
                r += early - kbt
            else:
                r += early
            if is_early == (pass_ == 0):
                out.append(e if is_early else early + (u - e))
    return out


@pytest.mark.parametrize("kbt", [1, 2, 3, 20, 28, 68, 72])
def test_mlp_decode_kwalk_is_a_permutation_of_every_fragment_split(kbt):
    """Whatever contiguous pieces a tile's units are cut into, the pieces'
    walks visit every k-block exactly once, early k-blocks (0..early-1) before
    the others within each piece."""
    import numpy as np
    g = np.random.default_rng(kbt)
    for early in range(0, kbt + 1):
        assert sorted(_kwalk(kbt, early, 0, kbt)) == list(range(kbt))
        for _ in range(5):
            cuts = sorted(set(int(c) for c in g.integers(1, kbt, size=3))) if kbt > 1 else []
            bounds = [0] + cuts + [kbt]
            seen = []
            for a, b in zip(bounds[:-1], bounds[1:]):
                walk = _kwalk(kbt, early, a, b)
                n_early = sum(1 for kb in walk if kb < early)
                assert all(kb < early for kb in walk[:n_early]) and all(kb >= early for kb in walk[n_early:])
                seen += walk
            assert sorted(seen) == list(range(kbt)), (kbt, early, bounds)
