"""Host-side tests of the C ABI (no GPU needed): the library loads and
exports every declared symbol, argument validation, path selection, and the
shared-memory layouts' swizzle properties."""
import ctypes
import os
import re

import numpy as np

import pytest

import __graft_entry__
import dense_gemm_major_gb300 as dg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()
    return dg.load()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(gemm_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol(built):
    declared = _declared_functions()
    assert {"gemm_f32", "gemm_f16", "gemm_bf16", "gemm_status_string"} <= declared
    for name in declared:
        assert hasattr(built, name), name
    assert declared == set(dg.EXPORTED)


def test_status_strings():
    for code in range(7):
        s = dg.status_string(code)
        assert s and s != "unknown status"
    assert dg.status_string(99) == "unknown status"


FAKE = 1 << 40   # a 16-byte aligned fake device address, never dereferenced


@pytest.mark.parametrize("entry", ["f32", "f16", "bf16"])
def test_invalid_arguments_rejected_before_any_device_work(entry):
    bad = [
        (-1, 4, 4, FAKE, 4, FAKE + 4096, 4, FAKE + 8192, 4),          # negative M
        (4, -1, 4, FAKE, 4, FAKE + 4096, 4, FAKE + 8192, 4),          # negative N
        (4, 4, -1, FAKE, 4, FAKE + 4096, 4, FAKE + 8192, 4),          # negative K
        (4, 4, 8, FAKE, 4, FAKE + 4096, 4, FAKE + 8192, 4),           # lda < K
        (4, 8, 4, FAKE, 4, FAKE + 4096, 4, FAKE + 8192, 8),           # ldb < N
        (4, 8, 4, FAKE, 4, FAKE + 4096, 8, FAKE + 8192, 4),           # ldc < N
        (4, 4, 4, 0, 4, FAKE + 4096, 4, FAKE + 8192, 4),              # null A
        (4, 4, 4, FAKE, 4, 0, 4, FAKE + 8192, 4),                     # null B
        (4, 4, 4, FAKE, 4, FAKE + 4096, 4, 0, 4),                     # null C
        (4, 4, 4, FAKE, 4, FAKE + 4096, 4, FAKE + 16, 4),             # C overlaps A
        (4, 4, 4, FAKE + 4096, 4, FAKE, 4, FAKE + 16, 4),             # C overlaps B
    ]
    for args in bad:
        assert dg.gemm(entry, *args, 0) == dg.GEMM_ERR_INVALID_ARG, args


@pytest.mark.parametrize("entry", ["f32", "f16", "bf16"])
def test_empty_output_is_a_noop_without_a_device(entry):
    assert dg.gemm(entry, 0, 5, 7, 0, 7, 0, 5, 0, 5, 0) == dg.GEMM_OK
    assert dg.gemm(entry, 5, 0, 7, 0, 7, 0, 1, 0, 1, 0) == dg.GEMM_OK


def test_valid_call_without_a_gpu_fails_loudly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = dg.gemm("f32", 4, 4, 4, FAKE, 4, FAKE + 4096, 4, FAKE + 8192, 4, 0)
    assert st == dg.GEMM_ERR_UNSUPPORTED_DEVICE


def _dp_tiles(tiles, grid):
    """Whole tiles of the full waves before the stream-K share."""
    return (tiles // grid - 1) * grid if tiles // grid >= 2 else 0


def _streamk_cuts(tiles, nk, grid):
    """Tiles that a boundary c * total // grid (0 < c < grid) cuts, total the
    k-tiles of the tiles left after the full waves."""
    total = (tiles - _dp_tiles(tiles, grid)) * nk
    return sum(1 for c in range(1, grid) if (c * total // grid) % nk)


def _streamk_units(tiles, nk, grid):
    """The SGEMM kernel's unit loop, per CTA: (tile, k_begin, k_end) -- its
    whole tiles of the waves, then of its stream-K range the whole tiles,
    the head of the last tile (k from 0) and the tail of the first (to nk)."""
    dp = _dp_tiles(tiles, grid)
    total = (tiles - dp) * nk
    out = []
    for b in range(grid):
        units = [(t, 0, nk) for t in range(b, dp, grid)]
        it0, it1 = b * total // grid, (b + 1) * total // grid
        if it1 > it0:
            t0, kb0 = divmod(it0, nk)
            t1, ke1 = (it1 - 1) // nk, (it1 - 1) % nk + 1
            if t0 == t1:
                units.append((dp + t0, kb0, ke1))
            else:
                head = ke1 < nk
                w0 = t0 + (1 if kb0 > 0 else 0)
                w1 = t1 - (1 if head else 0)
                units += [(dp + t, 0, nk) for t in range(w0, w1 + 1)]
                if head:
                    units.append((dp + t1, 0, ke1))
                if kb0 > 0:
                    units.append((dp + t0, kb0, nk))
        out.append(units)
    return out


@pytest.mark.parametrize("tiles,nk,slots", [(512, 128, 152), (2048, 256, 152), (252, 8, 152),
                                            (153, 3, 152), (60, 5, 152), (1000, 1, 304),
                                            (305, 17, 304), (7, 2, 152)])
def test_streamk_schedule_covers_every_k_tile_once(tiles, nk, slots):
    # The plan's grid rule, then the kernel's unit loop: every (tile, k-tile)
    # is computed exactly once, no tile has more than two pieces, the cut
    # count is what the plan reports, and the two pieces of a cut tile meet
    # at one boundary (its flag words and workspace tile), a different one
    # for every cut tile.
    grid = slots if tiles > slots else (2 * tiles if (2 * tiles <= slots and nk >= 2) else tiles)
    units = _streamk_units(tiles, nk, grid)
    seen = {}
    slots_used = {}
    for b, us in enumerate(units):
        for (t, kb, ke) in us:
            for k in range(kb, ke):
                assert (t, k) not in seen
                seen[(t, k)] = b
            if (kb, ke) != (0, nk):
                piece = 0 if kb == 0 else 1
                cb = b + 1 if piece == 0 else b
                assert 1 <= cb < grid
                slots_used.setdefault((t, cb), set()).add(piece)
    assert len(seen) == tiles * nk
    pieces = {}
    for (t, k), b in seen.items():
        pieces.setdefault(t, set()).add(b)
    assert max(len(v) for v in pieces.values()) <= 2
    assert all(v == {0, 1} for v in slots_used.values())
    assert len(slots_used) == _streamk_cuts(tiles, nk, grid)
    assert len({cb for (_, cb) in slots_used}) == len(slots_used)   # one tile per boundary


def test_plan_paths():
    ok, p = dg.gemm_plan("f32", 4096, 4096, 4096, FAKE, 4096, FAKE + (1 << 30), 4096,
                         FAKE + (2 << 30), 4096)
    assert ok == dg.GEMM_OK and p.path == dg.PATH_SIMT_TMA
    # many tiles: the wide 128 x 256 configuration, one CTA per SM; of the
    # 512 tiles, two full waves (304) run whole and the other 208 are shared
    # out stream-K over 152 CTAs (1.37 tiles each); the range boundaries that
    # fall inside a tile cut it in two
    assert (p.block_m, p.block_n, p.block_k, p.stages) == (128, 256, 32, 4)
    assert p.tiles == 32 * 16 and p.ctas == 152
    assert _dp_tiles(512, 152) == 304
    assert p.split_tiles == _streamk_cuts(512, 128, 152) == 144
    ok, p = dg.gemm_plan("f32", 8192, 8192, 8192, FAKE, 8192, FAKE + (1 << 30), 8192,
                         FAKE + (2 << 30), 8192, num_sms=152)
    assert p.ctas == 152 and p.split_tiles == _streamk_cuts(2048, 256, 152)
    # 252 = 152 + 100 tiles: balanced the same way
    ok, p = dg.gemm_plan("f32", 128 * 21, 256 * 12, 256, FAKE, 256, FAKE + (1 << 30), 3072,
                         FAKE + (2 << 30), 3072, num_sms=152)
    assert p.tiles == 252 and p.ctas == 152 and p.split_tiles == _streamk_cuts(252, 8, 152)
    # a single k-tile cannot be split
    ok, p = dg.gemm_plan("f32", 1000, 1030, 32, FAKE, 32, FAKE + (1 << 30), 1030,
                         FAKE + (2 << 30), 1030, num_sms=152)
    assert p.split_tiles == 0 and p.splitk_slices == 1 and p.workspace_bytes == 0
    # skinny: 4 tiles, K = 65536 -> 32 slices (the cap)
    ok, p = dg.gemm_plan("f32", 256, 256, 65536, FAKE, 65536, FAKE + (1 << 34), 256,
                         FAKE + (2 << 34), 256, num_sms=152)
    assert (p.tiles, p.splitk_slices, p.ctas) == (4, 32, 128)
    assert p.workspace_bytes == 32 * 256 * 256 * 4
    # 2048^3: 128 wide tiles would leave 24 SMs idle; 256 narrow tiles with
    # one CTA per SM are balanced by stream-K over all 152 (speed 0.93 x 1
    # beats 1.00 x 128/152)
    ok, p = dg.gemm_plan("f32", 2048, 2048, 2048, FAKE, 2048, FAKE + (1 << 30), 2048,
                         FAKE + (2 << 30), 2048, num_sms=152)
    assert ok == dg.GEMM_OK and (p.block_n, p.stages, p.tiles, p.ctas) == (128, 6, 256, 152)
    assert p.split_tiles == _streamk_cuts(256, 64, 152)
    # at most one narrow tile per SM: the narrow 128 x 128 configuration
    # with one CTA per SM (six stages)
    ok, p = dg.gemm_plan("f32", 1024, 1024, 512, FAKE, 512, FAKE + (1 << 30), 1024,
                         FAKE + (2 << 30), 1024, num_sms=152)
    assert ok == dg.GEMM_OK and (p.block_n, p.stages, p.tiles) == (128, 6, 64)
    # lda = 777 and ldb = 1030 floats are not 16-byte pitches: with
    # 8.0e8 >= 2^29 multiply-adds both operands are first re-pitched into
    # scratch (A's copy, 1000 x 780 floats, rounded up to 256 bytes, then
    # B's, 777 x 1032) and the product runs with TMA staging
    ok, p = dg.gemm_plan("f32", 1000, 1030, 777, FAKE, 777, FAKE + (1 << 30), 1030,
                         FAKE + (2 << 30), 1030)
    assert ok == dg.GEMM_OK and p.path == dg.PATH_SIMT_TMA
    assert p.pack == 3 and p.pack_bytes == (1000 * 780 * 4 + 255) // 256 * 256 + 777 * 1032 * 4
    # 72 narrow tiles as two k-halves each keep 144 of the 152 SMs busy
    # (score 0.91): the halves of a tile run as a 2-CTA cluster and add in
    # distributed shared memory (two k-slices, no workspace, no cut tiles)
    assert p.tiles == 8 * 9 and p.block_n == 128 and p.split_tiles == 0
    assert (p.splitk_slices, p.cluster_ctas, p.ctas, p.workspace_bytes) == (2, 2, 144, 0)
    # a smaller product with an unaligned pitch: staged in place by cp.async
    ok, p = dg.gemm_plan("f32", 700, 300, 333, FAKE, 333, FAKE + (1 << 30), 300,
                         FAKE + (2 << 30), 300)
    assert ok == dg.GEMM_OK and p.path == dg.PATH_SIMT_CPASYNC and p.pack == 0
    # 36 narrow tiles over K = 4096 (best whole-K score 0.45): split-K, 4
    # slices of 32 k-tiles (one CTA per SM; 8 slices would put two on each
    # SM for the same k-tiles per SM) into a 4 x 768 x 768 FP32 workspace
    ok, p = dg.gemm_plan("f32", 768, 768, 4096, FAKE, 4096, FAKE + (1 << 30), 768,
                         FAKE + (2 << 30), 768)
    assert (p.tiles, p.splitk_slices, p.cluster_ctas, p.ctas) == (36, 4, 0, 144)
    assert p.workspace_bytes == 4 * 768 * 768 * 4
    # tiny products: one k-tile per slice when the SMs allow (256^3: 4 tiles
    # x 8 slices), the split that minimises the busiest SM's k-tiles plus a
    # fixed cost per slice (512^3: 16 tiles x 9 slices)
    for (m, n, k), want in [((256, 256, 256), (4, 8)), ((512, 512, 512), (16, 9)),
                            ((384, 384, 384), (9, 12)), ((256, 256, 1024), (4, 32))]:
        ok, p = dg.gemm_plan("f32", m, n, k, FAKE, k, FAKE + (1 << 30), n, FAKE + (2 << 30), n)
        assert (p.tiles, p.splitk_slices, p.cluster_ctas) == want + (0,)
    # misaligned base pointer (4-byte aligned only)
    ok, p = dg.gemm_plan("f32", 64, 64, 64, FAKE + 4, 64, FAKE + (1 << 30), 64,
                         FAKE + (2 << 30), 64)
    assert ok == dg.GEMM_OK and p.path == dg.PATH_SIMT_CPASYNC
    # K == 0 -> zero fill, A and B may be null
    ok, p = dg.gemm_plan("f32", 64, 64, 0, 0, 0, 0, 64, FAKE, 64)
    assert ok == dg.GEMM_OK and p.path == dg.PATH_ZERO_FILL
    # FP16 / BF16: tensor-core path with a persistent grid
    for dt in ("f16", "bf16"):
        ok, p = dg.gemm_plan(dt, 4096, 4096, 4096, FAKE, 4096, FAKE + (1 << 30), 4096,
                             FAKE + (2 << 30), 4096, num_sms=152)
        assert ok == dg.GEMM_OK and p.path == dg.PATH_TC_TMA
        # CTA pairs: 256 tiles of 256 x 256 = 3 x 76 + 28; the last 104
        # tiles are a stream-K share (72 of them cut into a head and a tail)
        assert (p.cluster_ctas, p.block_m, p.block_n, p.block_k, p.stages) == (2, 256, 256, 128, 3)
        assert p.tiles == 16 * 16 and p.ctas == 152
        assert (p.split_in_k, p.streamk_first_tile, p.split_tiles, p.split_pieces) == \
            (1, 152, 72, 2)
        ok, p = dg.gemm_plan(dt, 4097, 3000, 1536, FAKE, 1536, FAKE + (1 << 30), 3000,
                             FAKE + (2 << 30), 3000, num_sms=152)
        assert ok == dg.GEMM_OK and p.path == dg.PATH_TC_TMA and p.tiles == 17 * 12
        assert p.cluster_ctas == 2
        # one tile: a CTA pair with two 128-column parts (4 SMs), the same
        # number of busy SMs as four single-CTA parts, and the pair kernel
        # is the faster one per SM
        ok, p = dg.gemm_plan(dt, 2, 3, 4, FAKE, 8, FAKE + 4096, 8, FAKE + 8192, 8, num_sms=152)
        assert ok == dg.GEMM_OK and (p.tiles, p.split_tiles, p.split_pieces, p.ctas) == (1, 1, 2, 4)
        assert p.cluster_ctas == 2 and (p.block_m, p.block_n) == (256, 256) and p.splitk_slices == 1
        # a 129 x 264 grid: four single-CTA tiles in four column parts (16
        # SMs) beat two pair tiles in two parts (8 SMs)
        ok, p = dg.gemm_plan(dt, 129, 264, 72, FAKE, 72, FAKE + 4096, 264, FAKE + (1 << 20), 264,
                             num_sms=152)
        assert (p.cluster_ctas, p.tiles, p.split_tiles, p.split_pieces, p.ctas) == (1, 4, 4, 4, 16)
        # 4 tiles, 16 k-tiles: split-K, 4 slices of 4 k-tiles on 16 CTAs
        ok, p = dg.gemm_plan(dt, 256, 512, 1024, FAKE, 1024, FAKE + (1 << 30), 512,
                             FAKE + (2 << 30), 512, num_sms=152)
        assert (p.tiles, p.split_tiles, p.splitk_slices, p.ctas) == (4, 0, 4, 16)
        assert p.workspace_bytes == 4 * 256 * 512 * 4
        # K of 2 k-tiles is too short for split-K: 4 column parts instead
        ok, p = dg.gemm_plan(dt, 256, 512, 128, FAKE, 128, FAKE + (1 << 30), 512,
                             FAKE + (2 << 30), 512, num_sms=152)
        assert (p.tiles, p.split_tiles, p.split_pieces, p.splitk_slices, p.ctas) == (4, 4, 4, 1, 16)
        # skinny: 2 tiles, K = 65536 -> 32 slices
        ok, p = dg.gemm_plan(dt, 256, 256, 65536, FAKE, 65536, FAKE + (1 << 34), 256,
                             FAKE + (2 << 34), 256, num_sms=152)
        assert (p.tiles, p.splitk_slices, p.ctas) == (2, 32, 64)
        # 8192^3: 1024 pair tiles = 13 x 76 + 36 -> stream-K share of the
        # last 112; the edge shape: 204 pair tiles = 2 x 76 + 52, but only 12
        # k-tiles -> a partial last round (52 tiles do not fit it twice)
        ok, p = dg.gemm_plan(dt, 8192, 8192, 8192, FAKE, 8192, FAKE + (1 << 30), 8192,
                             FAKE + (2 << 30), 8192, num_sms=152)
        assert (p.cluster_ctas, p.split_in_k, p.streamk_first_tile) == (2, 1, 912)
        ok, p = dg.gemm_plan(dt, 4097, 3000, 1536, FAKE, 1536, FAKE + (1 << 30), 3000,
                             FAKE + (2 << 30), 3000, num_sms=152)
        assert (p.split_in_k, p.split_tiles, p.split_pieces) == (0, 0, 1)
        # fewer pair tiles than SM pairs (2048 x 1024: 32 tiles): still pairs,
        # as two column parts each, 128 SMs busy like 64 single-CTA tiles in
        # two parts would keep
        ok, p = dg.gemm_plan(dt, 2048, 1024, 512, FAKE, 512, FAKE + (1 << 30), 1024,
                             FAKE + (2 << 30), 1024, num_sms=152)
        assert (p.cluster_ctas, p.tiles, p.split_tiles, p.split_pieces, p.ctas) == (2, 32, 32, 2, 128)
        # long K on a small grid: single-CTA split-K (2 x 1 tiles, 32 slices)
        ok, p = dg.gemm_plan(dt, 256, 256, 65536, FAKE, 65536, FAKE + (1 << 30), 256,
                             FAKE + (2 << 30), 256, num_sms=152)
        assert (p.cluster_ctas, p.tiles, p.splitk_slices) == (1, 2, 32)
        # lda not a multiple of 8 elements, or a 2-byte aligned base: refused
        ok, _ = dg.gemm_plan(dt, 64, 64, 60, FAKE, 60, FAKE + 4096, 64, FAKE + 65536, 64)
        assert ok == dg.GEMM_ERR_MISALIGNED
        ok, _ = dg.gemm_plan(dt, 64, 64, 64, FAKE + 2, 64, FAKE + 65536, 64, FAKE + (1 << 20), 64)
        assert ok == dg.GEMM_ERR_MISALIGNED


# ------------------------------------------------ shared-memory layouts

def _tma_swizzle_128b(byte_offset):
    """TMA's 128-byte swizzle on a 1024-byte aligned tile: bits [4,7) of the
    byte address are XOR-ed with bits [7,10)."""
    return byte_offset ^ (((byte_offset >> 7) & 7) << 4)


def test_a_tile_layout_is_the_tma_128b_swizzle_and_a_bijection():
    seen = set()
    for m in range(128):
        for k in range(32):
            off = dg.gemm_smem_layout_offset(0, m, k)
            assert 0 <= off < 128 * 32
            logical = (m * 32 + k) * 4
            assert off * 4 == _tma_swizzle_128b(logical), (m, k)
            seen.add(off)
    assert len(seen) == 128 * 32
    assert dg.gemm_smem_layout_offset(0, 128, 0) == -1
    assert dg.gemm_smem_layout_offset(5, 0, 0) == -1


def _wavefronts(byte_addrs, width):
    """Shared-memory wavefronts of one warp-wide load, by the rule measured on
    sm_103a with a shared-load probe under ncu: requests to one address are
    merged (broadcast); a wavefront delivers at most 16 bytes of distinct data
    to each group of 4 consecutive lanes; a 16-byte load takes at least 2
    wavefronts; and distinct words that fall in one bank serialise."""
    lanes = list(byte_addrs)
    per_group = max(len(set(lanes[4 * g:4 * g + 4])) * width for g in range(8))
    need = max(2 if width == 16 else 1, -(-per_group // 16))
    load = [0] * 32
    for a in sorted(set(lanes)):
        for b in range(width // 4):
            load[(a // 4 + b) % 32] += 1
    return max(need, max(load))


def _lane_rc(l):
    """The SGEMM kernel's lane -> (tr, tc) map: each 4-lane group is a 2 x 2
    block of the 4 x 8 lane grid."""
    return ((l >> 4) << 1) | ((l >> 1) & 1), (((l >> 2) & 3) << 1) | (l & 1)


def test_lane_map_is_a_bijection():
    assert sorted(_lane_rc(l) for l in range(32)) == [(r, c) for r in range(4) for c in range(8)]


def test_wavefront_rule_reproduces_the_probe():
    # Values measured on GB300 for 32 lanes reading 16-byte chunk f(l)
    # (or 8-byte word f(l) for the 8-byte loads).
    cases16 = {lambda l: 0: 2, lambda l: l >> 3: 2, lambda l: l >> 4: 2, lambda l: l & 1: 2,
               lambda l: (l >> 2) & 1: 2, lambda l: l >> 2: 2, lambda l: (l >> 1) & 3: 2,
               lambda l: l & 7: 4, lambda l: (l & 1) + 2 * (l >> 4): 2,
               lambda l: (l >> 1) & 7: 2, lambda l: l >> 1: 2,
               lambda l: ((l >> 3) & 1) + 2 * (l & 1): 2}
    for f, wf in cases16.items():
        assert _wavefronts([16 * f(l) for l in range(32)], 16) == wf
    cases8 = {lambda l: 0: 1, lambda l: l >> 3: 1, lambda l: l & 7: 2,
              lambda l: (l >> 1) & 3: 1, lambda l: (l >> 1) & 7: 1, lambda l: l >> 1: 1}
    for f, wf in cases8.items():
        assert _wavefronts([8 * f(l) for l in range(32)], 8) == wf
    assert _wavefronts([128 * (l >> 3) for l in range(32)], 16) == 4   # bank conflict


def test_fragment_reads_take_the_minimum_wavefronts():
    # Warp (wm, wn) of a 4 x 2 grid; lane (tr, tc) owns rows 32 wm + tr + 4 i
    # and columns (BN/2) wn + 4 tc + 32 h.  A reads: 16 bytes (four k-steps)
    # of one row; B reads: 16 bytes of one k row.  Both must deliver 8 bytes
    # per lane per wavefront: 2 wavefronts each.
    for wm in range(4):
        for i in range(8):
            for kq in range(8):
                addrs = [4 * dg.gemm_smem_layout_offset(0, 32 * wm + _lane_rc(l)[0] + 4 * i, 4 * kq)
                         for l in range(32)]
                assert _wavefronts(addrs, 16) == 2, (wm, i, kq)
    for layout, bn in ((1, 128), (2, 256)):
        for wn in range(2):
            for k in range(32):
                for h in range(bn // 64):
                    addrs = [4 * dg.gemm_smem_layout_offset(
                        layout, k, (bn // 2) * wn + 4 * _lane_rc(l)[1] + 32 * h) for l in range(32)]
                    assert _wavefronts(addrs, 16) == 2
    assert dg.gemm_smem_layout_offset(2, 0, 255) == 255
    assert dg.gemm_smem_layout_offset(1, 0, 128) == -1


def test_row_major_lane_map_would_cost_more():
    # With lanes laid out row-major (tc = l % 8) a 4-lane group reads 4 B
    # chunks and the B reads cost 4 wavefronts: the check above can tell the
    # two lane maps apart.
    addrs = [4 * dg.gemm_smem_layout_offset(1, 0, 4 * (l % 8)) for l in range(32)]
    assert _wavefronts(addrs, 16) == 4


def test_cp_async_tile_writes_are_conflict_free():
    # Unaligned path: warp w writes A row (w + 8 j), k = lane; B row k, 32
    # consecutive columns.
    for w in range(8):
        for j in range(16):
            addrs = [4 * dg.gemm_smem_layout_offset(0, w + 8 * j, l) for l in range(32)]
            assert _wavefronts(addrs, 4) == 1
    for layout, bn in ((1, 128), (2, 256)):
        for k in range(32):
            for c0 in range(0, bn, 32):
                addrs = [4 * dg.gemm_smem_layout_offset(layout, k, c0 + l) for l in range(32)]
                assert _wavefronts(addrs, 4) == 1


def test_naive_row_major_a_tile_would_conflict():
    # The A read pattern on an unswizzled tile (rows 128 bytes apart) is a
    # bank conflict: the check above is able to see one.
    addrs = [4 * (_lane_rc(l)[0] * 32 + 0) for l in range(32)]
    assert _wavefronts(addrs, 16) == 4


def test_scaled_plans():
    # alpha == 0 or K == 0: C := beta * C, A and B may be null
    ok, p = dg.gemm_plan_ex("f32", 64, 64, 32, 0.0, 0, 32, 0, 64, 2.0, FAKE, 64, 152)
    assert ok == dg.GEMM_OK and p.path == dg.PATH_ZERO_FILL
    ok, p = dg.gemm_plan_ex("bf16", 64, 64, 0, 1.0, 0, 0, 0, 64, 0.5, FAKE, 64, 152)
    assert ok == dg.GEMM_OK and p.path == dg.PATH_ZERO_FILL
    # The SGEMM's stream-K pieces either way; with beta != 0 the first of a
    # cut tile's pieces leaves its sums in a workspace of one FP32 tile per
    # range boundary (151 x 128 x 256 x 4 bytes), with beta == 0 it stores
    # them to C and the second piece adds into C.
    args = (4096, 4096, 4096, 1.0, FAKE, 4096, FAKE + (1 << 30), 4096)
    ok, p0 = dg.gemm_plan_ex("f32", *args, 0.0, FAKE + (2 << 30), 4096, 152)
    ok, p1 = dg.gemm_plan_ex("f32", *args, 0.5, FAKE + (2 << 30), 4096, 152)
    assert p0.split_tiles == 144 and p1.split_tiles == 144 and p1.ctas == 152
    assert p0.workspace_bytes == 0 and p1.workspace_bytes == 151 * 128 * 256 * 4
    # FP16/BF16 plans do not depend on alpha and beta
    for dt in ("f16", "bf16"):
        ok, q0 = dg.gemm_plan(dt, 4096, 4096, 4096, FAKE, 4096, FAKE + (1 << 30), 4096,
                              FAKE + (2 << 30), 4096, 152)
        ok, q1 = dg.gemm_plan_ex(dt, *args, -1.0, FAKE + (2 << 30), 4096, 152)
        assert (q0.split_tiles, q0.ctas, q0.cluster_ctas) == (q1.split_tiles, q1.ctas, q1.cluster_ctas)
    # the scaled entry points validate like the plain ones
    for dt in ("f32", "f16", "bf16"):
        assert dg.gemm_ex(dt, -1, 4, 4, 1.0, FAKE, 4, FAKE + 4096, 4, 0.0, FAKE + 8192, 4, 0) \
            == dg.GEMM_ERR_INVALID_ARG
        assert dg.gemm_ex(dt, 4, 4, 4, 1.0, FAKE, 4, FAKE + 4096, 4, 1.0, FAKE + 16, 4, 0) \
            == dg.GEMM_ERR_INVALID_ARG


# ------------------------------------------------ operands stored transposed

def test_transposed_b_tiles_permute_chunks_within_rows():
    for layout, bn in ((3, 128), (4, 256)):
        for k in range(32):
            offs = [dg.gemm_smem_layout_offset(layout, k, n) for n in range(bn)]
            assert sorted(offs) == list(range(k * bn, (k + 1) * bn))
            for n in range(0, bn, 4):     # 16-byte chunks stay whole and aligned
                assert offs[n] % 4 == 0 and offs[n + 1:n + 4] == [offs[n] + 1, offs[n] + 2, offs[n] + 3]
                assert (offs[n] - k * bn) // 32 == n // 32   # within its 128-byte segment
        assert dg.gemm_smem_layout_offset(layout, 32, 0) == -1
        assert dg.gemm_smem_layout_offset(layout, 0, bn) == -1


def test_transposed_b_fragment_reads():
    # The kernel reads B element (k, n = (BN/2) wn + 4 tc + 32 h) of a
    # transposed-B tile at k BN + (BN/2) wn + 4 (tc ^ (k / 4)) + 32 h: that
    # formula must agree with the layout, and the reads take 2 wavefronts.
    for layout, bn in ((3, 128), (4, 256)):
        for wn in range(2):
            for k in range(32):
                for h in range(bn // 64):
                    addrs = []
                    for l in range(32):
                        tc = _lane_rc(l)[1]
                        n = (bn // 2) * wn + 4 * tc + 32 * h
                        kernel = k * bn + (bn // 2) * wn + 4 * (tc ^ (k >> 2)) + 32 * h
                        assert dg.gemm_smem_layout_offset(layout, k, n) == kernel
                        addrs.append(4 * kernel)
                    assert _wavefronts(addrs, 16) == 2


def _bt_copy(j, w, l, bn):
    """(k, n) that lane l of warp w writes in copy j of a transposed B."""
    return 4 * (l & 7) + (j & 3), 4 * ((bn // 32) * w + (j >> 2)) + (l >> 3)


def _at_copy(j, w, l):
    """(m, k) that lane l of warp w writes in copy j of a transposed A."""
    idx = 16 * w + j
    return 8 * (idx >> 3) + (l & 7), 4 * (idx & 7) + (l >> 3)


def test_transposing_copies_cover_the_tiles_and_are_conflict_free():
    seen = set()
    for w in range(8):
        for j in range(16):
            mk = [_at_copy(j, w, l) for l in range(32)]
            seen.update(mk)
            assert _wavefronts([4 * dg.gemm_smem_layout_offset(0, m, k) for m, k in mk], 4) == 1
    assert seen == {(m, k) for m in range(128) for k in range(32)}
    for layout, bn in ((3, 128), (4, 256)):
        seen = set()
        for w in range(8):
            for j in range(bn // 8):
                kn = [_bt_copy(j, w, l, bn) for l in range(32)]
                seen.update(kn)
                assert _wavefronts([4 * dg.gemm_smem_layout_offset(layout, k, n) for k, n in kn],
                                   4) == 1
        assert seen == {(k, n) for k in range(32) for n in range(bn)}


def test_transposing_b_copy_into_plain_rows_would_conflict():
    # The same copy pattern into the unswizzled B tile puts 8 lanes on each
    # bank: the swizzle of the transposed-B tile is what removes that.
    kn = [_bt_copy(0, 0, l, 256) for l in range(32)]
    assert _wavefronts([4 * dg.gemm_smem_layout_offset(2, k, n) for k, n in kn], 4) == 8


def test_op_plans_and_validation():
    M, N, K = 300, 200, 100
    args = (FAKE, 0, FAKE + (1 << 24), 0)
    def plan(dt, oa, ob, lda, ldb, alpha=1.0, beta=0.0):
        return dg.gemm_plan_op(dt, oa, ob, M, N, K, alpha, FAKE, lda, FAKE + (1 << 24), ldb,
                               beta, FAKE + (1 << 26), N, 152)
    # leading dimensions: op N A needs lda >= K, op T A needs lda >= M;
    # op N B needs ldb >= N, op T B needs ldb >= K
    assert plan("f32", "N", "N", K, N)[0] == dg.GEMM_OK
    assert plan("f32", "T", "N", M, N)[0] == dg.GEMM_OK
    assert plan("f32", "T", "N", M - 1, N)[0] == dg.GEMM_ERR_INVALID_ARG
    assert plan("f32", "N", "T", K, K)[0] == dg.GEMM_OK
    assert plan("f32", "N", "T", K, K - 1)[0] == dg.GEMM_ERR_INVALID_ARG
    assert plan("f32", "T", "T", M, K)[0] == dg.GEMM_OK
    # an unknown op is an argument error
    assert dg.load().gemm_plan_op(0, 2, 0, M, N, K, 1.0, FAKE, K, FAKE + (1 << 24), N, 0.0,
                                  FAKE + (1 << 26), N, 152, ctypes.byref(dg.Plan())) \
        == dg.GEMM_ERR_INVALID_ARG
    # FP32: a transposed operand that is not packed (too small a product
    # here) is staged by cp.async; the other one by TMA when it is 16-byte
    # aligned (mixed), else by cp.async too
    assert plan("f32", "N", "N", 104, 200)[1].path == dg.PATH_SIMT_TMA
    assert plan("f32", "T", "N", 304, 200)[1].path == dg.PATH_SIMT_MIXED
    assert plan("f32", "N", "T", 104, 104)[1].path == dg.PATH_SIMT_MIXED
    assert plan("f32", "T", "N", 304, 201)[1].path == dg.PATH_SIMT_CPASYNC
    assert plan("f32", "N", "T", 101, 104)[1].path == dg.PATH_SIMT_CPASYNC
    assert plan("f32", "T", "N", 304, 200)[1].pack == 0
    # both transposed: computed as C^T = B_st . A_st, two row-major arrays
    # (TMA when aligned), stored transposed; the plan describes that product
    st, p = plan("f32", "T", "T", 304, 104)
    assert p.path == dg.PATH_SIMT_TMA
    assert p.tiles == ((N + 127) // 128) * ((M + 127) // 128)     # N x M output, narrow tiles
    assert plan("f32", "T", "T", 301, 104)[1].path == dg.PATH_SIMT_CPASYNC
    # FP16/BF16: TMA either way; the stored row must be 16-byte aligned
    for dt in ("f16", "bf16"):
        st, p = plan(dt, "T", "T", 304, 104)
        assert st == dg.GEMM_OK and p.path == dg.PATH_TC_TMA
        assert plan(dt, "T", "N", 301, 200)[0] == dg.GEMM_ERR_MISALIGNED
        assert plan(dt, "N", "T", 104, 100)[0] == dg.GEMM_ERR_MISALIGNED
    # the same tiles and split as the row-major call
    st0, p0 = dg.gemm_plan("bf16", 4096, 4096, 4096, FAKE, 4096, FAKE + (1 << 30), 4096,
                           FAKE + (2 << 30), 4096, 152)
    st1, p1 = dg.gemm_plan_op("bf16", "T", "T", 4096, 4096, 4096, 1.0, FAKE, 4096,
                              FAKE + (1 << 30), 4096, 0.0, FAKE + (2 << 30), 4096, 152)
    assert (p0.tiles, p0.ctas, p0.split_tiles, p0.cluster_ctas) == \
        (p1.tiles, p1.ctas, p1.split_tiles, p1.cluster_ctas)
    # nothing is packed for FP16/BF16 (the tensor cores read either major
    # order) or with both operands transposed (C^T = B_st . A_st)
    assert plan("bf16", "N", "T", 104, 104)[1].pack == 0
    assert plan("f32", "T", "T", 304, 104)[1].pack == 0
    # overlap uses the stored extent: A stored K x M spans (K-1) lda + M
    A = FAKE
    C = FAKE + 4 * ((K - 1) * M + M)          # just past A's last element
    assert dg.gemm_plan_op("f32", "T", "N", M, N, K, 1.0, A, M, FAKE + (1 << 24), N, 0.0, C, N,
                           152)[0] == dg.GEMM_OK
    assert dg.gemm_plan_op("f32", "T", "N", M, N, K, 1.0, A, M, FAKE + (1 << 24), N, 0.0, C - 4,
                           N, 152)[0] == dg.GEMM_ERR_INVALID_ARG


def test_sgemm_pack_decisions():
    # One FP32 operand stored transposed is packed (copied transposed into
    # row-major scratch) when the other output dimension reuses each of its
    # elements at least 256 times, M * N * K >= 2^30 and the copy fits
    # 1 GiB; the plan is then the row-major product's.
    def plan(oa, ob, M, N, K):
        lda = M if oa == "T" else K
        ldb = K if ob == "T" else N
        return dg.gemm_plan_op("f32", oa, ob, M, N, K, 1.0, FAKE, lda, FAKE + (1 << 36), ldb,
                               0.0, FAKE + (1 << 38), N, 152)
    def nn(M, N, K):
        return dg.gemm_plan("f32", M, N, K, FAKE, K, FAKE + (1 << 36), N, FAKE + (1 << 38), N,
                            152)[1]
    for oa, ob, M, N, K in (("T", "N", 4096, 4096, 4096), ("N", "T", 4096, 4096, 4096),
                            ("T", "N", 2048, 2048, 1000), ("N", "T", 256, 8192, 1024),
                            ("N", "T", 4096, 128, 4096), ("T", "N", 128, 4096, 4096)):
        st, p = plan(oa, ob, M, N, K)
        q = nn(M, N, K)
        packed = (M, (K + 3) // 4 * 4) if oa == "T" else (K, (N + 3) // 4 * 4)
        assert st == dg.GEMM_OK and p.pack == (1 if oa == "T" else 2)
        assert p.pack_bytes == packed[0] * packed[1] * 4
        assert (p.path, p.tiles, p.ctas, p.block_n, p.split_tiles, p.splitk_slices) == \
            (q.path, q.tiles, q.ctas, q.block_n, q.split_tiles, q.splitk_slices)
    # too little reuse, or too small a product: staged transposed by cp.async
    assert plan("T", "N", 4096, 255, 4096)[1].pack == 0
    assert plan("N", "T", 255, 4096, 4096)[1].pack == 0
    assert plan("T", "N", 4096, 256, 4096)[1].pack == 1
    assert plan("T", "N", 1000, 1030, 777)[1].pack == 0
    assert plan("N", "T", 1024, 1024, 1023)[1].pack == 0
    assert plan("N", "T", 1024, 1024, 1024)[1].pack == 2
    # over the 1 GiB cap: A stored 65536 x 8192 would need 2 GiB of scratch
    st, p = plan("T", "N", 8192, 4096, 65536)
    assert st == dg.GEMM_OK and p.pack == 0 and p.path == dg.PATH_SIMT_MIXED


def test_sgemm_repitch_decisions():
    # Row-major FP32 operands whose base or leading dimension is not 16-byte
    # aligned are copied into 16-byte-pitched scratch (plan.pack bit 0 for
    # A, bit 1 for B; A's copy first, rounded up to 256 bytes) when
    # M * N * K >= 2^29, and the product then runs with TMA staging; below
    # that they are staged in place by cp.async.
    def plan(M, N, K, lda, ldb, a_off=0, b_off=0):
        return dg.gemm_plan("f32", M, N, K, FAKE + a_off, lda, FAKE + (1 << 36) + b_off, ldb,
                            FAKE + (1 << 38), N, 152)[1]
    r256 = lambda x: (x + 255) // 256 * 256
    p = plan(1024, 1024, 1024, 1025, 1024)
    assert (p.pack, p.path, p.pack_bytes) == (1, dg.PATH_SIMT_TMA, 1024 * 1024 * 4)   # M x K
    p = plan(1024, 1030, 600, 600, 1030)
    assert (p.pack, p.path, p.pack_bytes) == (2, dg.PATH_SIMT_TMA, 600 * 1032 * 4)
    p = plan(1100, 900, 555, 555, 903)
    assert (p.pack, p.path) == (3, dg.PATH_SIMT_TMA)
    assert p.pack_bytes == r256(1100 * 556 * 4) + 555 * 900 * 4
    # a base 4 bytes past a 16-byte boundary counts as unaligned as well
    p = plan(1024, 1024, 1024, 1024, 1024, a_off=4, b_off=4)
    assert (p.pack, p.pack_bytes) == (3, r256(1024 * 1024 * 4) + 1024 * 1024 * 4)
    # 2^29 is the threshold: 512 x 1024 x 1024 copies, 512 x 1024 x 1020 does not
    assert plan(512, 1024, 1024, 1025, 1024).pack == 1
    p = plan(512, 1024, 1020, 1021, 1024)
    assert (p.pack, p.path) == (0, dg.PATH_SIMT_CPASYNC)
    # aligned operands are never copied
    assert plan(4096, 4096, 4096, 4096, 4096).pack == 0
    # a transposed operand that is packed takes its unaligned row-major
    # partner along: A stored K x M transposed, B (ldb 2061) re-pitched
    st, p = dg.gemm_plan_op("f32", "T", "N", 1024, 2048, 1025, 1.0, FAKE, 1024,
                            FAKE + (1 << 36), 2061, 0.0, FAKE + (1 << 38), 2048, 152)
    assert st == dg.GEMM_OK and (p.pack, p.path) == (3, dg.PATH_SIMT_TMA)
    assert p.pack_bytes == r256(1024 * 1028 * 4) + r256(1025 * 2048 * 4)


def test_sgemm_cluster_query_without_a_device():
    # The device's cluster capacities are only known on a device: -1 here,
    # and -1 for sizes or configurations that do not exist.
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert dg.gemm_sgemm_clusters(0, 2) == -1
    assert dg.gemm_sgemm_clusters(3, 2) == -1 and dg.gemm_sgemm_clusters(0, 3) == -1


def test_host_entry_blocks_and_validation():
    # Row blocks: FP32 two while each block keeps a full grid of 128 x 256
    # tiles, else one; FP16 / BF16 up to four blocks of whole 256-row units.
    assert dg.gemm_host_blocks("f32", 4096, 4096, 152) == 2
    assert dg.gemm_host_blocks("f32", 2048, 2048, 152) == 1
    assert dg.gemm_host_blocks("f32", 8192, 1024, 152) == 1
    assert dg.gemm_host_blocks("f16", 4096, 4096, 152) == 4
    assert dg.gemm_host_blocks("bf16", 4097, 3000, 152) == 4
    assert dg.gemm_host_blocks("f16", 300, 4096, 152) == 2
    assert dg.gemm_host_blocks("f16", 256, 4096, 152) == 1
    assert dg.gemm_host_blocks("bf16", 0, 4096, 152) == 1
    # FP32 products of >= 2^36 FLOPs with K >= 2048 also run as three
    # ranges of K (never FP16 / BF16, whose partial C would be rounded)
    assert dg.gemm_host_k_blocks("f32", 4096, 4096, 4096) == 3
    assert dg.gemm_host_k_blocks("f32", 4096, 4096, 2048) == 3
    assert dg.gemm_host_k_blocks("f32", 4096, 4096, 1024) == 1
    assert dg.gemm_host_k_blocks("f32", 2048, 2048, 2048) == 1
    assert dg.gemm_host_k_blocks("f16", 8192, 8192, 8192) == 1
    # Argument errors are found before any CUDA call (no device needed)
    H = 1 << 32
    call = dg.gemm_host
    assert call("f32", "N", "N", 0, 8, 8, 1.0, 0, 8, 0, 8, 0.0, 0, 8) == dg.GEMM_OK
    assert call("f32", "N", "N", 8, 8, 8, 1.0, H, 8, H + 4096, 8, 0.0, H + 8192, 7) == \
        dg.GEMM_ERR_INVALID_ARG                                     # ldc < N
    assert call("f32", "N", "N", 8, 8, 8, 1.0, 0, 8, H + 4096, 8, 0.0, H + 8192, 8) == \
        dg.GEMM_ERR_INVALID_ARG                                     # A null
    assert call("f32", "T", "N", 8, 8, 4, 1.0, H, 7, H + 4096, 8, 0.0, H + 8192, 8) == \
        dg.GEMM_ERR_INVALID_ARG                                     # A stored K x M, lda < M
    assert call("f16", "N", "N", 8, 8, 8, 1.0, H + 1, 8, H + 4096, 8, 0.0, H + 8192, 8) == \
        dg.GEMM_ERR_INVALID_ARG                                     # not element-aligned
    assert call("f32", "N", "N", 8, 8, 8, 1.0, H, 8, H + 4096, 8, 0.0, H + 128, 8) == \
        dg.GEMM_ERR_INVALID_ARG                                     # C overlaps A
    assert dg.load().gemm_host(3, 0, 0, 8, 8, 8, 1.0, H, 8, H + 4096, 8, 0.0, H + 8192, 8,
                               None) == dg.GEMM_ERR_INVALID_ARG     # unknown dtype


def test_pair_streamk_plans():
    # The CTA-pair kernel's tiles beyond whole rounds: with at least 24
    # k-tiles of 128 the last partial round and the round before it (or the
    # two before it, when one leaves a range less than 8 k-tiles beyond a
    # tile) are shared out as equal ranges of (tile, k-tile) work (one head
    # partial per range boundary in the workspace); with fewer, the last
    # round's tiles run as column parts when they fit it twice.
    def plan(dt, M, N, K):
        return dg.gemm_plan(dt, M, N, K, FAKE, K, FAKE + (1 << 34), N, FAKE + (1 << 36), N, 152)[1]
    ws = 76 * 256 * 256 * 4
    p = plan("f16", 4096, 4096, 4096)              # 256 tiles = 3 x 76 + 28
    assert (p.cluster_ctas, p.ctas, p.split_in_k, p.streamk_first_tile) == (2, 152, 1, 152)
    assert (p.split_tiles, p.split_pieces, p.workspace_bytes) == (72, 2, ws)
    p = plan("bf16", 8192, 8192, 8192)             # 1024 tiles = 13 x 76 + 36
    assert (p.split_in_k, p.streamk_first_tile, p.ctas) == (1, 912, 152)
    p = plan("bf16", 4096, 4096, 3072)             # 24 k-tiles: 28 x 24 / 76 = 8.8 beyond
    assert (p.split_in_k, p.streamk_first_tile) == (1, 152)
    p = plan("f16", 4096, 4608, 2816)              # 288 tiles, 22 k-tiles: too short
    assert p.split_in_k == 0
    p = plan("f16", 4096, 4096, 2944)              # 23 k-tiles: column parts
    assert (p.split_in_k, p.split_tiles, p.split_pieces, p.workspace_bytes) == (0, 28, 2, 0)
    p = plan("f16", 1280, 4864, 3328)              # 95 tiles, 26 k-tiles: 19 x 26 / 76 < 8,
    assert (p.split_in_k, p.ctas) == (0, 152)      # no second round to widen into
    p = plan("f16", 4096, 4608, 4096)              # 16 x 18 = 288 tiles = 3 x 76 + 60
    assert (p.split_in_k, p.streamk_first_tile) == (1, 152)
    p = plan("f16", 4864, 4096, 4096)              # 19 x 16 = 304 = 4 x 76: whole rounds
    assert (p.split_in_k, p.split_tiles, p.ctas) == (0, 0, 152)
    p = plan("f16", 2048, 2048, 2048)              # 64 tiles: one partial round
    assert (p.split_in_k, p.ctas) == (0, 128)


@pytest.mark.parametrize("dt,M,N,K", [("f16", 4096, 4096, 4096), ("bf16", 8192, 8192, 8192),
                                      ("bf16", 4097, 3000, 1536), ("f16", 4000, 4000, 6200),
                                      ("bf16", 4096, 4096, 3072), ("f16", 4864, 2560, 4096),
                                      ("f16", 2304, 4096, 1024), ("bf16", 4096, 4096, 896),
                                      ("f16", 1280, 4864, 6144), ("bf16", 2048, 2048, 2048)])
def test_pair_schedule_covers_every_k_tile_once(dt, M, N, K):
    # The units every pair runs (the kernel's own schedule code, run on the
    # host): each (tile, column, k-tile) exactly once; a cut tile is one head
    # (on pair q - 1 right after its whole tiles of the rounds, k-tiles
    # [0, h)) and one tail (last unit of pair q, k-tiles [h, nk)) for
    # boundary q; whole units have every k-tile; pairs get equal work within
    # one k-tile of a full-width tile; the rounds before the share are in
    # step (unit i of every pair is a tile of round i).
    st, p = dg.gemm_plan(dt, M, N, K, FAKE, K, FAKE + (1 << 34), N, FAKE + (1 << 36), N, 152)
    assert st == dg.GEMM_OK and p.cluster_ctas == 2
    pairs = p.ctas // 2
    tm_n, tn_n, nk = -(-M // 256), -(-N // 256), -(-K // p.block_k)
    cover = np.zeros((tm_n, tn_n, 256, nk), dtype=np.int32)
    heads, tails, work = {}, {}, []
    for q in range(pairs):
        units = dg.gemm_pair_units(p, M, N, K, q)
        w_q = 0
        for j, (tm, tn, n_off, n_w, kb, ke, kind, slot) in enumerate(units):
            assert 0 <= tm < tm_n and 0 <= tn < tn_n and 0 <= kb < ke <= nk
            cover[tm, tn, n_off:n_off + n_w, kb:ke] += 1
            w_q += (ke - kb) * n_w
            if kind == 1:
                assert j == p.streamk_first_tile // pairs and kb == 0 and ke < nk
                assert slot == q + 1 and n_w == 256
                heads[slot] = (tm, tn, ke)
            elif kind == 2:
                assert j == len(units) - 1 and kb > 0 and ke == nk and slot == q and n_w == 256
                tails[slot] = (tm, tn, kb)
            else:
                assert kind == 0 and (kb, ke) == (0, nk)
        work.append(w_q)
    assert np.all(cover == 1)
    assert heads == tails
    assert len(heads) == (p.split_tiles if p.split_in_k else 0)
    if p.split_in_k:
        assert max(work) - min(work) <= 256
        assert p.workspace_bytes >= (max(heads, default=0) + 1) * 256 * 256 * 4


def test_pair_plan_with_fewer_resident_clusters():
    # A device that holds fewer CTA pairs at once than num_sms / 2 (shared
    # or partitioned): the persistent pair grid shrinks to what fits, and no
    # pair is left polling for a partial from another pair.
    def plan(dt, M, N, K, clusters):
        st, p = dg.gemm_plan_resident(dt, "N", "N", M, N, K, 1.0, FAKE, K, FAKE + (1 << 34), N,
                                      0.0, FAKE + (1 << 36), N, 152, clusters)
        assert st == dg.GEMM_OK
        return p
    full = plan("f16", 4096, 4096, 8192, 0)
    assert (full.cluster_ctas, full.split_in_k, full.ctas) == (2, 1, 152)
    same = plan("f16", 4096, 4096, 8192, 76)       # every pair fits: as planned
    assert (same.split_in_k, same.ctas, same.workspace_bytes) == \
        (1, 152, full.workspace_bytes)
    more = plan("f16", 4096, 4096, 8192, 80)       # more than the SMs allow: as planned
    assert (more.split_in_k, more.ctas) == (1, 152)
    few = plan("f16", 4096, 4096, 8192, 72)        # 144 of 152 SMs
    assert (few.cluster_ctas, few.split_in_k, few.ctas, few.workspace_bytes) == (2, 0, 144, 0)
    few = plan("bf16", 8192, 8192, 8192, 60)        # 120 of 152: single CTAs keep more busy
    assert (few.cluster_ctas, few.split_in_k, few.ctas) == (1, 0, 152)
    assert dg.gemm_plan_resident("f16", "N", "N", 64, 64, 64, 1.0, FAKE, 64, FAKE + 8192, 64,
                                 0.0, FAKE + 16384, 64, 152, -1)[0] == dg.GEMM_ERR_INVALID_ARG
