"""Pins of the oracle's batching arithmetic against the values the pages print."""
import pytest

from oracle import batching
from oracle.paged_attention import OracleError, slot_of
from conftest import read_golden


def test_padding_waste_printed_values():
    for row in read_golden("padding_waste.txt"):
        if row[0] == "ratio":
            continue
        if row[0] == "mixed_second_difference":
            mixed = (batching.padding_waste(9, 101) - batching.padding_waste(9, 100)
                     - batching.padding_waste(8, 101) + batching.padding_waste(8, 100))
            assert mixed == int(row[1])
            continue
        B, n, waste, padded, real = map(int, row)
        batch = [n] + [1] * (B - 1)
        assert batching.padding_waste(B, n) == waste
        assert batching.padded_slots(batch) == padded
        assert batching.useful_slots(batch) == real


def test_padding_ratios_printed_values():
    w = batching.padding_waste
    got = {
        "double_B": w(16, 100) / w(8, 100),
        "double_n": w(8, 200) / w(8, 100),
        "double_both": w(16, 200) / w(8, 100),
    }
    for row in read_golden("padding_waste.txt"):
        if row[0] == "ratio":
            assert f"{got[row[1]]:.3f}" == row[2]


def test_padding_waste_closed_form_and_linearity():
    # (n-1)(B-1) for every B, n < 40, against the brute-force rectangle.
    for B in range(1, 40):
        for n in range(1, 40):
            assert batching.padding_waste(B, n) == (n - 1) * (B - 1)
    # Linear in each variable: second differences vanish; the growth is not quadratic.
    for B in range(1, 20):
        assert (batching.padding_waste(B + 2, 100) - 2 * batching.padding_waste(B + 1, 100)
                + batching.padding_waste(B, 100)) == 0
    for n in range(1, 20):
        assert (batching.padding_waste(8, n + 2) - 2 * batching.padding_waste(8, n + 1)
                + batching.padding_waste(8, n)) == 0


def test_zero_length_row_is_rejected():
    with pytest.raises(OracleError):
        batching.padded_slots([100, 0, 1])
    with pytest.raises(OracleError):
        batching.useful_slots([])


def test_static_utilisation_printed_values():
    for row in read_golden("utilisation.txt"):
        bar = row.index("|")
        useful, total, pct = int(row[0]), int(row[1]), float(row[2])
        lengths = [int(x) for x in row[bar + 1:]]
        assert batching.useful_slots(lengths) == useful
        assert batching.padded_slots(lengths) == total
        assert round(100 * batching.static_utilisation(lengths), 1) == pct


def test_block_arithmetic_printed_values():
    for tokens, bs, blocks, waste in (map(int, r) for r in read_golden("block_arithmetic.txt")):
        assert batching.blocks_for(tokens, bs) == blocks
        assert batching.tail_waste(tokens, bs) == waste


def test_tail_waste_bound_is_tight():
    for bs in (4, 16, 64, 256, 1024):
        worst = max(batching.tail_waste(L, bs) for L in range(1, 2 * bs + 1))
        assert worst == bs - 1
        assert all(batching.tail_waste(L, bs) < bs for L in range(0, 3 * bs))


def test_block_size_below_four_is_rejected():
    for bad in (0, 1, 2, 3):
        with pytest.raises(OracleError):
            batching.blocks_for(10, bad)
        with pytest.raises(OracleError):
            slot_of([0], 0, bad)
    assert batching.blocks_for(10, 4) == 3


def test_block_table_worked_example():
    for row in read_golden("block_table_example.txt"):
        bar = row.index("|")
        table = [int(x) for x in row[2].split(",")]
        pos, blk, off, flat = map(int, row[bar + 1:])
        assert slot_of(table, pos, 4) == flat
        assert divmod(slot_of(table, pos, 4), 4) == (blk, off)
    # tail waste of the example: 2 slots in A's last block, 2 in B's
    assert batching.tail_waste(10, 4) == 2 and batching.tail_waste(6, 4) == 2


def test_slot_of_rejects_undefined_positions():
    with pytest.raises(OracleError):
        slot_of([7, 2, 5], 12, 4)          # logical block 3 is not in the table
    with pytest.raises(OracleError):
        slot_of([7, -1, 5], 5, 4)          # unused entry
    with pytest.raises(OracleError):
        slot_of([7, 2, 5], 1, 4, num_pages=6)  # block 7 outside a 6-block pool
