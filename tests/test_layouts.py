"""The host-side packers of the input module (scales: bench.py's
--scale-layout packed; sub-byte elements: --element-layout packed) against
the packed layouts that mxgemm.h defines, worked out per element.  CPU
only."""
import numpy as np
import torch

import mx_inputs as mi


def test_pack_scales_places_every_scale_once():
    # the bench's host packer (a layout change only): every row-major scale
    # lands at the chunk byte the layout of mxgemm.h gives it, worked here
    # per element from the definition, and the rest of the area is 127
    g = torch.Generator().manual_seed(61)
    for n, kbn, cols in [(300, 13, False), (130, 9, True), (1, 1, False), (257, 8, True)]:
        s = torch.randint(0, 255, (n, kbn), generator=g, dtype=torch.int64).to(torch.uint8)
        packed = mi.pack_scales(s, along_cols=cols).numpy()
        steps = -(-kbn // 4)
        size = (-(-n // 256) * steps * 1024) if cols else (-(-n // 128) * steps * 512)
        assert packed.size == size
        seen = np.zeros(size, dtype=bool)
        for r in range(n):
            for kb in range(kbn):
                chunk = (((r // 256) * steps + kb // 4) * 2 + (r // 128) % 2) if cols else \
                    ((r // 128) * steps + kb // 4)
                at = chunk * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4
                assert packed[at] == int(s[r, kb])
                seen[at] = True
        assert np.all(packed[~seen] == 127)


def test_pack_elements_places_each_code_at_its_bits():
    # element i of a 16-element group at bits [b*i, b*i + b) of the group's
    # little-endian 128-bit number; the high bits of each input byte dropped
    g = torch.Generator().manual_seed(5)
    for nbits in (4, 6):
        codes = torch.randint(0, 256, (3, 48), generator=g, dtype=torch.int32).to(torch.uint8)
        packed = mi.pack_elements(codes, nbits).numpy()
        c = codes.numpy()
        for r in range(3):
            for grp in range(3):
                value = int.from_bytes(packed[r, 16 * grp:16 * grp + 16].tobytes(), "little")
                for i in range(16):
                    assert (value >> (nbits * i)) & ((1 << nbits) - 1) == c[r, 16 * grp + i] & ((1 << nbits) - 1)
                assert value >> (16 * nbits) == 0


def test_pattern_matrix_rows_and_exactness():
    # the large-index tests rebuild sampled rows of this matrix on the CPU:
    # a row subset must equal the same rows of the whole matrix, every value
    # must be exact in BF16 (so the BF16 input holds the same numbers), and
    # the blocks' magnitudes must vary (different scales)
    x = mi.pattern_matrix(96, 160)
    rows = [0, 31, 32, 95]
    assert torch.equal(mi.pattern_matrix(96, 160, rows=rows), x[rows])
    assert torch.equal(x.to(torch.bfloat16).float(), x)
    r, c = 37, 70
    k = ((7919 * r + 104729 * c) % 255) - 127
    e = ((r + c // 32) % 16) - 8
    assert x[r, c].item() == k / 8 * 2.0 ** e
    amax = x.reshape(96, 5, 32).abs().amax(-1)
    assert torch.unique(amax).numel() > 8
