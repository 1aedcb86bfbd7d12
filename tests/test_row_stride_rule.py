"""Page 1's padded-row-stride rule, pinned on the CPU.

A model of a tiled store: each output row of OW columns is written by
ceil(OW / BLOCK_OW) tiles of BLOCK_OW columns into a buffer whose rows are
`stride` elements apart; the store is clipped only at the end of the whole
buffer (the 2-D descriptor shape), not at the end of the row.  With the
wrong stride rule the last tile of a row spills into the next row; the page
prints how many columns (tests/golden/tma_row_stride.json).  The fixed rule
spills nothing.
"""
import json
import os

import pytest

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tma_row_stride.json")))
BLOCK_OW = GOLDEN["block_ow"]


def wrong_stride(ow):
    return -(-max(ow, BLOCK_OW) // 4) * 4


def fixed_stride(ow):
    return -(-ow // BLOCK_OW) * BLOCK_OW


def columns_past_row_end(ow, stride, rows=3):
    """Count elements of row r+1 (or padding) a row-r tile store writes."""
    written_into_next_row = 0
    for r in range(rows - 1):
        for t0 in range(0, ow, BLOCK_OW):
            for c in range(t0, t0 + BLOCK_OW):
                addr = r * stride + c
                if addr >= (r + 1) * stride:
                    written_into_next_row += 1
    return written_into_next_row // (rows - 1)


@pytest.mark.parametrize("case", GOLDEN["cases"])
def test_wrong_rule_reproduces_page_counts(case):
    ow = case["ow"]
    assert columns_past_row_end(ow, wrong_stride(ow)) == case["columns_written_past_row_end"]
    assert BLOCK_OW - ow % BLOCK_OW == case["columns_written_past_row_end"]


@pytest.mark.parametrize("ow", [1, 15, 16, 17, 20, 40, 80, 160, 320])
def test_fixed_rule_never_spills(ow):
    assert columns_past_row_end(ow, fixed_stride(ow)) == 0
