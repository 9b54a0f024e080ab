"""Host-side shape checks of the Python binding (no GPU): a decode call whose tensors
disagree in shape is refused before anything reaches the library."""

import pytest

from paged_kv_cache_264_gb300.api import check_decode_shapes


def test_agreeing_shapes_pass():
    assert check_decode_shapes(128, (4, 32, 128), (4, 10), (4,)) == (4, 1, 32)
    assert check_decode_shapes(64, (3, 2, 8, 64), (3, 7), (3,), (3, 2, 8, 64)) == (3, 2, 8)
    assert check_decode_shapes(64, (0, 8, 64), (0, 1), (0,)) == (0, 1, 8)


@pytest.mark.parametrize("q, tables, lens, out", [
    ((4, 32, 64), (4, 10), (4,), None),              # head_dim of another pool
    ((4, 32, 128), (3, 10), (4,), None),             # fewer table rows than sequences
    ((4, 32, 128), (4, 10), (5,), None),             # more lengths than sequences
    ((4, 32, 128), (4,), (4,), None),                # table not 2-D
    ((4, 32, 128), (4, 10), (4, 1), None),           # lengths not 1-D
    ((4, 32, 128), (4, 10), (4,), (4, 16, 128)),     # out not q's shape
    ((2, 3, 32, 128), (2, 10), (2,), (2, 32, 128)),  # 4-D q with a 3-D out
    ((32, 128), (4, 10), (4,), None),                # q neither 3-D nor 4-D
])
def test_disagreeing_shapes_raise(q, tables, lens, out):
    with pytest.raises(ValueError):
        check_decode_shapes(128, q, tables, lens, out)
