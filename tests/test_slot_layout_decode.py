"""CPU pins of the slot-layout decoders used by the per-step GPU test: every (row, column) of each
tile maps to its own element-aligned offset and together they fill the tile's bytes exactly, as
the layouts in include/kda.h state (a wrong XOR, stride or block size breaks one of these)."""
import numpy as np

from tests.test_gpu_slot_steps import SLOT_LAYOUT, _cm16, _cm32, _sw128


def _tiles_once(off, elem, size):
    flat = np.sort(off.ravel())
    assert np.all(flat % elem == 0)
    assert np.array_equal(flat, np.arange(0, size, elem))


def test_swizzled_tiles_are_bijections():
    _tiles_once(_sw128(32), 2, 32 * 256)   # Z': 32 rows x 128 bf16
    _tiles_once(_sw128(16), 2, 16 * 256)   # V, Kbar: 16 rows x 128 f16
    # within a 128-byte row, the 16-byte chunks of eight consecutive rows are all different (the
    # swizzle spreads a column block over the eight chunk positions)
    off = _sw128(16)
    for c in range(0, 64, 8):
        assert len({int(off[r, c]) % 128 // 16 for r in range(8)}) == 8


def test_core_matrix_tiles_are_bijections():
    _tiles_once(_cm16(32), 2, 32 * 32)     # TM, (H Phi^T)^T, H''^T: 32 x 16 f16
    _tiles_once(_cm32(), 4, 32 * 128)      # Phi: 32 x 32 fp32
    # an 8x8 (f16) / 8x4 (fp32) core matrix is 128 contiguous bytes
    assert _cm16(32)[7, 7] - _cm16(32)[0, 0] == 126 and _cm32()[7, 3] - _cm32()[0, 0] == 124


def test_slot_regions_do_not_overlap():
    size = {"Z": 8192, "V": 4096, "KB": 4096, "PHI": 4096, "TM": 1024, "CC": 1024, "HP": 1024, "GAM": 512}
    spans = sorted((SLOT_LAYOUT[k], SLOT_LAYOUT[k] + size[k]) for k in size)
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0
    assert spans[-1][1] <= 24576
