"""The storage layout against sizes the pages print (tests/golden/page_sizes.txt).

The oracle's decoder accepts a projection only as (in/16)(out/16) tiles of
16*K uint16 words; these tests build code arrays of exactly the printed
sizes and require the oracle to decode them, so a layout with any per-tile
or per-expert overhead (or a different tile shape) fails."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_sizes.txt")


def _rows():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, *kv, nbytes = line.split()
        out.append((name, {k: int(v) for k, v in (x.split("=") for x in kv)}, int(nbytes)))
    return out


@pytest.mark.parametrize("row", [r for r in _rows() if r[0] == "half"], ids=lambda r: f"K{r[1]['K']}")
def test_half_projection_bytes(row):
    _, a, nbytes = row
    words = np.zeros(nbytes // 2, np.uint16)
    dense = oracle.decode_dense(words, a["rows"], a["cols"], a["K"])
    assert dense.shape == (a["rows"], a["cols"])
    assert (dense == 0x3F60).all()   # zero codes: every weight 1.84375 (fp16 0x3F60)


def test_layer_file_bytes():
    """The codes of a K4 layer of 289 experts in this layout take all but
    65,536 bytes of the printed file size.  Those 64 KiB are less than one
    byte per 400 tiles, so the file leaves no room for per-tile overhead
    (a trellis that was not tail-biting, with even 16 spare bits a tile, would
    need 57 MB more), and 65,536 is no multiple of the 867 expert
    projections, so no fixed per-projection header either."""
    (_, a, nbytes), = [r for r in _rows() if r[0] == "layer_file"]
    H, I, K, n = a["hidden"], a["inter"], a["K"], a["experts"]
    # one expert's projection: gate/up are H x I, down I x H; the oracle takes
    # exactly (in/16)(out/16)*16*K words for each
    per_proj_words = (H // 16) * (I // 16) * 16 * K
    code_bytes = n * 3 * per_proj_words * 2
    tiles = n * 3 * (H // 16) * (I // 16)
    assert code_bytes == n * 3 * H * I * K // 8
    assert nbytes - code_bytes == 65536
    assert (nbytes - code_bytes) * 400 < tiles and (nbytes - code_bytes) % (3 * n) != 0
    # and decodes a block of tiles of that layout (a 256 x 256 corner)
    words = np.zeros((256 // 16) * (256 // 16) * 16 * K, np.uint16)
    assert oracle.decode_dense(words, 256, 256, K).shape == (256, 256)
