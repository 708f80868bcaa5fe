"""Host-side tests of the C ABI (no GPU needed): the library loads and
exports every declared symbol, argument validation, path selection, and the
shared-memory layouts' swizzle properties."""
import os
import re

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
    for code in range(6):
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


def test_plan_paths():
    ok, p = dg.gemm_plan("f32", 4096, 4096, 4096, FAKE, 4096, FAKE + (1 << 30), 4096,
                         FAKE + (2 << 30), 4096)
    assert ok == dg.GEMM_OK and p.path == dg.PATH_SIMT_TMA
    assert (p.block_m, p.block_n, p.block_k) == (128, 128, 32)
    assert p.tiles == 32 * 32 and p.ctas == 1024
    # lda = 777 floats is not a 16-byte pitch: cp.async staging
    ok, p = dg.gemm_plan("f32", 1000, 1030, 777, FAKE, 777, FAKE + (1 << 30), 1030,
                         FAKE + (2 << 30), 1030)
    assert ok == dg.GEMM_OK and p.path == dg.PATH_SIMT_CPASYNC
    assert p.tiles == 8 * 9
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
        assert p.tiles == 32 * 16 and p.ctas == 152
        ok, p = dg.gemm_plan(dt, 4097, 3000, 1536, FAKE, 1536, FAKE + (1 << 30), 3000,
                             FAKE + (2 << 30), 3000, num_sms=152)
        assert ok == dg.GEMM_OK and p.path == dg.PATH_TC_TMA and p.tiles == 33 * 12
        ok, p = dg.gemm_plan(dt, 2, 3, 4, FAKE, 8, FAKE + 4096, 8, FAKE + 8192, 8, num_sms=152)
        assert ok == dg.GEMM_OK and p.ctas == 1
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
    assert dg.gemm_smem_layout_offset(2, 0, 0) == -1


def _wavefronts(byte_addrs, width):
    """Shared-memory wavefronts one warp-wide access needs: requests to the
    same address are merged (broadcast); each distinct `width`-byte word
    occupies width/4 consecutive banks; the access takes as many wavefronts as
    the most-loaded bank has distinct words, and at least total/128 bytes."""
    distinct = sorted(set(byte_addrs))
    load = [0] * 32
    for a in distinct:
        for b in range(width // 4):
            load[(a // 4 + b) % 32] += 1
    return max(max(load), -(-len(distinct) * width // 128))


def test_fragment_reads_are_conflict_free():
    # The SGEMM thread mapping: warp (wm, wn) of a 4 x 2 grid, lane (tr, tc)
    # = (lane // 8, lane % 8) owns rows 32 wm + tr + 4 i and columns
    # 64 wn + 4 tc + {0..3} (+32).  A reads: one 16-byte k-quad of one row.
    for wm in range(4):
        for i in range(8):
            for kq in range(8):
                addrs = [4 * dg.gemm_smem_layout_offset(0, 32 * wm + (l // 8) + 4 * i, 4 * kq)
                         for l in range(32)]
                assert _wavefronts(addrs, 16) == 1, (wm, i, kq)
    # B reads: 16 bytes at column 64 wn + 4 tc (+32) of one k row.
    for wn in range(2):
        for k in range(32):
            for h in range(2):
                addrs = [4 * dg.gemm_smem_layout_offset(1, k, 64 * wn + 4 * (l % 8) + 32 * h)
                         for l in range(32)]
                assert _wavefronts(addrs, 16) == 1


def test_cp_async_tile_writes_are_conflict_free():
    # Unaligned path: warp w writes A row (w + 8 j), k = lane; B row k, 32
    # consecutive columns.
    for w in range(8):
        for j in range(16):
            addrs = [4 * dg.gemm_smem_layout_offset(0, w + 8 * j, l) for l in range(32)]
            assert _wavefronts(addrs, 4) == 1
    for k in range(32):
        for c0 in range(0, 128, 32):
            addrs = [4 * dg.gemm_smem_layout_offset(1, k, c0 + l) for l in range(32)]
            assert _wavefronts(addrs, 4) == 1


def test_naive_row_major_a_tile_would_conflict():
    # The same A read pattern on an unswizzled tile is a 4-way conflict: the
    # check above is able to see one.
    addrs = [4 * ((l // 8) * 32 + 0) for l in range(32)]
    assert _wavefronts(addrs, 16) == 4
