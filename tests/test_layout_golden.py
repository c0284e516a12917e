"""CPU pins of the pair-interleaved value-code plane (include/tq.h, storage format):
a hand-worked 16-token block (tests/golden/v_pair_block_b3.txt) read back by the
binding's plane converter, and the same codes packed by the oracle into per-token
records. No GPU is used."""

import numpy as np
import torch

from conftest import read_golden
from oracle import turboquant as otq
from quantised_kv_cache_gb300 import tq

VB = 3
PLANE_BYTES = 16 * 16 * VB  # eight pair rows of d * VB / 4 bytes
RECORD_BYTES = 16 * VB


def _golden():
    codes = np.zeros((16, 128), dtype=np.int64)
    plane = np.zeros(PLANE_BYTES, dtype=np.uint8)
    records = np.zeros((16, RECORD_BYTES), dtype=np.uint8)
    for row in read_golden("v_pair_block_b3.txt"):
        kind, vals = row[0], [int(x, 0) for x in row[1:]]
        if kind == "code":
            codes[vals[0], vals[1]] = vals[2]
        elif kind == "plane":
            plane[vals[0]] = vals[1]
        elif kind == "record":
            records[vals[0], vals[1]] = vals[2]
    return codes, plane, records


def test_golden_block_records_match_the_oracle_packing():
    codes, _, records = _golden()
    np.testing.assert_array_equal(otq.pack_codes(codes, VB), records)


def test_plane_converter_reads_the_hand_worked_block():
    _, plane, records = _golden()
    planes = torch.from_numpy(plane).view(1, 1, PLANE_BYTES)  # one sequence-head, one block
    got = tq._pair_rows_to_records(planes, VB).numpy().reshape(16, RECORD_BYTES)
    np.testing.assert_array_equal(got, records)


def test_plane_converter_keeps_blocks_and_heads_apart():
    # the same block placed at (head 1, block 2) of a 2 x 3 grid of blocks: its tokens
    # come out at slots 32..47 of head 1 and nothing else is set
    _, plane, records = _golden()
    planes = torch.zeros((2, 3, PLANE_BYTES), dtype=torch.uint8)
    planes[1, 2] = torch.from_numpy(plane)
    got = tq._pair_rows_to_records(planes, VB).numpy()
    assert got.shape == (2, 48, RECORD_BYTES)
    np.testing.assert_array_equal(got[1, 32:48], records)
    got[1, 32:48] = 0
    assert not got.any()
