"""The row-parallel projection kernel's schedule (k_gemv.cu), replayed on the
CPU: the stage ring (STAGES slots of ROWS rows, STAGES - 1 in flight), the x
groups (256 rows per load of warp 0, double-buffered in shared memory, one
group ahead in registers) and the copies issued before and after the wait for
the kernel before.  For ragged k and every prefetch depth it checks that every
row is folded exactly once and in order, from the slot its copy went to, with
the x of that row; that a slot is refilled only after its stage was folded;
and that an x buffer is rewritten only after the last stage that read it.  No
kernel code runs here; the constants are the kernel's."""
import re
from pathlib import Path

import pytest

HDR = Path(__file__).resolve().parents[1] / "barrier_free_message_gb300" / "csrc" / "sfar_gemv.h"


def constant(name):
    m = re.search(r"#define %s (\d+)" % name, HDR.read_text())
    assert m, name
    return int(m.group(1))


ROWS, STAGES = constant("SFAR_GEMV_ROWS"), constant("SFAR_GEMV_STAGES")
GROUP = 32 * 8


def replay(k, pre):
    nst = (k + ROWS - 1) // ROWS
    group_stages = GROUP // ROWS
    slot_stage = {}                      # slot -> stage whose copy is in it
    folded = {}                          # slot -> folded since its last copy
    issued = []
    waited = None
    # prologue: stages 0 .. STAGES - 2 into slots 0 .. STAGES - 2, the wait after `pre` of them
    for q in range(STAGES - 1):
        if q == pre:
            waited = len(issued)
        if q < nst:
            slot_stage[q] = q
            folded[q] = False
            issued.append(q)
    if pre >= STAGES - 1:
        waited = len(issued)
    assert waited == min(pre, STAGES - 1, nst), "the wait comes after the copies issued before it"
    xbuf = {0: 0, 1: 1}                  # buffer -> x group it holds
    xreg = 2                              # group in warp 0's registers
    last_read = {0: -1, 1: -1}            # buffer -> last stage that read it
    rows = []
    rd = 0
    for q in range(nst):
        assert slot_stage.get(rd) == q, (q, rd)          # the stage waited for is in its slot
        G, j = divmod(q, group_stages)
        wr = STAGES - 1 if rd == 0 else rd - 1
        if q + STAGES - 1 < nst:
            assert wr not in slot_stage or folded[wr], "slot refilled before its stage was folded"
            slot_stage[wr] = q + STAGES - 1
            folded[wr] = False
            issued.append(q + STAGES - 1)
        if j == 0 and G > 0:
            b = (G + 1) & 1
            assert last_read[b] < q, "x buffer rewritten while a later stage still reads it"
            xbuf[b] = xreg
            xreg = G + 2
        b = G & 1
        assert xbuf[b] == G, "stage folded with the x of another group"
        last_read[b] = q
        n = min(ROWS, k - q * ROWS)
        rows.extend(range(q * ROWS, q * ROWS + n))
        folded[rd] = True
        rd = 0 if rd == STAGES - 1 else rd + 1
    assert issued == list(range(nst)), "every stage copied once, in order"
    assert rows == list(range(k)), "every row folded once, in row order"


@pytest.mark.parametrize("k", [1, 7, 63, 64, 65, 255, 256, 257, 1000, 1024, 3584, 4097])
@pytest.mark.parametrize("pre", [0, 1, 2, 5])
def test_schedule_folds_every_row_once_in_order(k, pre):
    replay(k, min(pre, STAGES - 1))
