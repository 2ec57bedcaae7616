"""afx_tile_order on the host: the element order the fused prefill product
reads -- 128 x 64 tiles, row-major inside a tile, the tiles of a 128-row
band in column order, the bands in row order."""
import numpy as np
import pytest

from weight_streaming_canonical_gb300 import afx


@pytest.mark.parametrize("rows,cols", [(128, 64), (256, 192), (384, 5120)])
def test_tile_order_places_every_element(rows, cols):
    W = (np.arange(rows * cols, dtype=np.uint64) % 65521).astype(np.uint16).reshape(rows, cols)
    out = afx.afx_tile_order(W, rows, cols)
    # element (r, c) at ((r // 128) * (cols // 64) + c // 64) * 8192 + (r % 128) * 64 + c % 64
    r, c = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    pos = ((r // 128) * (cols // 64) + c // 64) * 8192 + (r % 128) * 64 + c % 64
    expect = np.empty(rows * cols, dtype=np.uint16)
    expect[pos.reshape(-1)] = W.reshape(-1)
    assert np.array_equal(out, expect)
    # the first tile is the top-left 128 x 64 block, row by row
    assert np.array_equal(out[:8192].reshape(128, 64), W[:128, :64])


def test_tile_order_refuses_ragged_shapes():
    with pytest.raises(afx.AfxError):
        afx.afx_tile_order(np.zeros(100 * 64, dtype=np.uint16), 100, 64)
    with pytest.raises(afx.AfxError):
        afx.afx_tile_order(np.zeros(128 * 40, dtype=np.uint16), 128, 40)
    with pytest.raises(afx.AfxError):
        afx.afx_tile_order(np.zeros(128 * 48, dtype=np.uint16), 128, 48)
