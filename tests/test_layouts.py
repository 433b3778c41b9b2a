"""The host-side scale packer of the input module (used by bench.py's
--scale-layout packed) against the packed scale layout that mxgemm.h
defines, worked out per element.  CPU only."""
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
