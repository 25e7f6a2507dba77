"""Philox4x32-10 counter-based generator (oracle side).

Written from the published definition in Salmon, Moraes, Dror, Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11): a 4x32-bit counter
and a 2x32-bit key; each of the 10 rounds multiplies words 0 and 2 by the
two round multipliers, takes the high and low halves of the 64-bit products
and mixes them with words 1 and 3 and the key; the key is bumped by the two
Weyl constants (golden ratio, sqrt(3)-1) before every round after the first.

The pages prescribe no generator; they only require a uniform r for the
accept test and draws from the draft and residual distributions
(Page A §6.2, Page B "随机采样验证").  This stream is our fixed choice.

Stream layout (shared specification with the CUDA library, implemented
independently on each side):
    key     = (seed, 0x000EA61E)
    counter = (draw_index, node_slot, (purpose << 16) | request, round_id)
    u32     = word 0 of the output
    purpose: 0 = child draw in the draft step, 1 = accept test, 2 = final draw
"""

MASK32 = 0xFFFFFFFF
ROUND_MUL = (0xD2511F53, 0xCD9E8D57)
KEY_BUMP = (0x9E3779B9, 0xBB67AE85)
KEY_TAG = 0x000EA61E

PURPOSE_DRAW = 0
PURPOSE_ACCEPT = 1
PURPOSE_FINAL = 2


def philox4x32_10(ctr, key):
    c0, c1, c2, c3 = (int(x) & MASK32 for x in ctr)
    k0, k1 = (int(x) & MASK32 for x in key)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + KEY_BUMP[0]) & MASK32
            k1 = (k1 + KEY_BUMP[1]) & MASK32
        prod0 = ROUND_MUL[0] * c0
        prod1 = ROUND_MUL[1] * c2
        hi0, lo0 = prod0 >> 32, prod0 & MASK32
        hi1, lo1 = prod1 >> 32, prod1 & MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & MASK32, lo1, (hi0 ^ c3 ^ k1) & MASK32, lo0
    return c0, c1, c2, c3


def uniform_u32(seed: int, draw_index: int, node_slot: int, purpose: int,
                request: int, round_id: int) -> int:
    """One 32-bit uniform of the round's stream (word 0 of Philox4x32-10)."""
    assert 0 <= request < (1 << 16) and 0 <= purpose < (1 << 16)
    ctr = (draw_index, node_slot, (purpose << 16) | request, round_id)
    return philox4x32_10(ctr, (seed, KEY_TAG))[0]
