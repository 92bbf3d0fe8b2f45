"""Pins for the oracle's scale-factor layout and group lookup.

The swizzled layout is defined on the pages as a logical 6-D shape
(32, 4, ceil(rows/128), 4, ceil(kblocks/4), L) ("Grouped GEMM + Quant
(SM100)", Shapes) stored in the physical C-contiguous order
(L, ceil(rows/128), ceil(kblocks/4), 32, 4, 4) ("Grouped GEMM + SwiGLU
(SM100)", Canonical layouts).  numpy's transpose of that logical array is the
independent check of the oracle's closed-form offset.
"""
import numpy as np
import pytest

import oracle as orc


@pytest.mark.parametrize("rows,kblocks,L", [(128, 4, 1), (300, 10, 2), (384, 8, 1), (33, 1, 3)])
def test_sf_offset_equals_physical_permutation(rows, kblocks, L):
    R, KQ = -(-rows // 128), -(-kblocks // 4)
    # logical index tensor: element (i0,i1,i2,i3,i4,l) carries its own (row, kblk, l)
    i0, i1, i2, i3, i4, l = np.meshgrid(np.arange(32), np.arange(4), np.arange(R), np.arange(4),
                                        np.arange(KQ), np.arange(L), indexing="ij")
    row = 128 * i2 + 32 * i1 + i0
    kb = 4 * i4 + i3
    # physical order (L, R, KQ, 32, 4, 4) = axes (l, i2, i4, i0, i1, i3)
    perm = (5, 2, 4, 0, 1, 3)
    phys_row = np.transpose(row, perm).reshape(-1)
    phys_kb = np.transpose(kb, perm).reshape(-1)
    phys_l = np.transpose(l, perm).reshape(-1)
    assert orc.sf_bytes(rows, kblocks, L) == phys_row.size
    for flat in range(0, phys_row.size, 7):
        assert orc.sf_offset(int(phys_row[flat]), int(phys_kb[flat]), int(phys_l[flat]),
                             rows, kblocks) == flat


def test_sf_offset_is_a_bijection_on_the_padded_domain():
    rows, kblocks, L = 260, 9, 2
    R, KQ = -(-rows // 128), -(-kblocks // 4)
    seen = set()
    for l in range(L):
        for r in range(R * 128):
            for kb in range(KQ * 4):
                seen.add(orc.sf_offset(r, kb, l, rows, kblocks))
    assert seen == set(range(orc.sf_bytes(rows, kblocks, L)))


def test_atom_inner_offset():
    # Inside each 512-byte atom the byte of (row, kblk) is
    # 16*(row%32) + 4*((row/32)%4) + kblk%4.
    for row in (0, 1, 31, 32, 63, 64, 127):
        for kb in range(4):
            assert orc.sf_offset(row, kb, 0, 128, 4) == 16 * (row % 32) + 4 * ((row // 32) % 4) + kb


def test_pack_sf_roundtrip_and_zero_padding():
    rng = np.random.default_rng(3)
    L, rows, kb = 2, 200, 7
    logical = rng.integers(1, 255, size=(L, rows, kb), dtype=np.uint8)
    swz = orc.pack_sf(logical)
    R, KQ = -(-rows // 128), -(-kb // 4)
    phys = swz.reshape(L, R, KQ, 32, 4, 4)
    # back to logical (32,4,R,4,KQ,L) then to (L, R*128, KQ*4)
    lg = np.transpose(phys, (3, 4, 1, 5, 2, 0))           # (i0,i1,i2,i3,i4,l)
    full = np.transpose(lg, (5, 2, 1, 0, 4, 3)).reshape(L, R * 128, KQ * 4)
    assert np.array_equal(full[:, :rows, :kb], logical)
    assert (full[:, rows:, :] == 0).all() and (full[:, :, kb:] == 0).all()


def test_group_of_row():
    off = np.array([128, 128, 384, 512], dtype=np.int32)   # group 1 is empty
    assert orc.group_of_row(off, 0) == 0
    assert orc.group_of_row(off, 127) == 0
    assert orc.group_of_row(off, 128) == 2
    assert orc.group_of_row(off, 383) == 2
    assert orc.group_of_row(off, 384) == 3
    assert orc.group_of_row(off, 511) == 3
    assert orc.group_of_row(off, 512) == -1
