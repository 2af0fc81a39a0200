"""The m16n8k16 fragment formulas as the mma.sync page prints them
("hgemm_mma_m16n8k16_naive_kernel详解", section 4.3 for A and B, section 6.2
for C/D), restated as functions of the lane and the element index:

    groupID = lane >> 2,  threadID_in_group = lane % 4
    A (a0..a7):  row = groupID for i in {0, 1, 4, 5}, else groupID + 8
                 col = 2 * threadID_in_group + (i & 1), + 8 for i >= 4
    B (b0..b3):  row = 2 * threadID_in_group + (i & 1), + 8 for i >= 2
                 col = groupID
    C (c0..c3):  row = groupID for i < 2, else groupID + 8
                 col = 2 * threadID_in_group + (i & 1)
"""


def a_coord(lane: int, i: int) -> tuple[int, int]:
    g, t = lane >> 2, lane % 4
    row = g if (i < 2 or 4 <= i < 6) else g + 8
    col = 2 * t + (i & 1) + (8 if i >= 4 else 0)
    return row, col


def b_coord(lane: int, i: int) -> tuple[int, int]:
    g, t = lane >> 2, lane % 4
    row = 2 * t + (i & 1) + (8 if i >= 2 else 0)
    return row, g


def c_coord(lane: int, i: int) -> tuple[int, int]:
    g, t = lane >> 2, lane % 4
    return (g if i < 2 else g + 8), 2 * t + (i & 1)
