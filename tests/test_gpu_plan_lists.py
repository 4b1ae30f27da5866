"""The planner's work lists checked bit for bit against the planning rules.

The lists are index work: they decide which CTA walks which blocks, never a
result, so the parity tests only see them indirectly.  Here a plan's lists
are read back (bsr_plan_work_list) and compared with the lists the rules
give, computed on the host from the block structure alone:

* the per-CTA share Lmax = max(8, ceil(nnzb * H' / G)) (capped at the grid
  size) with H' and G as the plan reports them;
* a line longer than Lmax cut into ceil(len / Lmax) chunks whose lengths
  differ by at most one, the longer ones first, offsets consecutive;
* lines with no stored block left out;
* the items ordered by length, longest first, then line, then chunk;
* -1 as the slot of a whole line, and consecutive slots, distinct between
  lines, for the chunks of a split line.

Above 2048 lines the planner places the items of one length with atomics
instead of in line order; there the lists must agree as sets and still be
ordered by length.
"""

import math

import numpy as np
import pytest
import torch

import block_sparse_attention_bsr_gb300 as bsr
from block_sparse_attention_bsr_gb300 import inputs

pytestmark = pytest.mark.gpu


def expected_items(ptr, n, nnzb, heads, G):
    """(line, first, n, chunk, chunks) of every item, in the rules' order."""
    lmax = min(max(8, math.ceil(nnzb * heads / G)), n)
    items = []
    for line in range(n):
        length = int(ptr[line + 1] - ptr[line])
        if length == 0:
            continue
        nc = math.ceil(length / lmax) if length > lmax else 1
        b, r = divmod(length, nc)
        off = int(ptr[line])
        for c in range(nc):
            clen = b + (1 if c < r else 0)
            items.append((line, off, clen, c, nc))
            off += clen
    items.sort(key=lambda t: (-t[2], t[0], t[3]))
    return items


def check_list(got, info, ptr, n, nnzb):
    want = expected_items(ptr, n, nnzb, info["heads"], info["G"])
    assert info["items"] == len(want) == len(got)
    assert info["buckets"] == len({w[2] for w in want})
    assert all(got[i, 2] >= got[i + 1, 2] for i in range(len(got) - 1)), "not longest first"
    if n <= 2048:
        assert [tuple(g[:3]) for g in got] == [w[:3] for w in want]
    else:
        assert sorted(tuple(g[:3]) for g in got) == sorted(w[:3] for w in want)
    # slots: -1 for whole lines; a split line's chunks get consecutive slots
    by_line = {}
    for line, first, _, slot in got.tolist():
        by_line.setdefault(line, []).append((first, slot))
    chunks = {w[0]: w[4] for w in want}
    used = set()
    for line, parts in by_line.items():
        slots = [s for _, s in sorted(parts)]
        if chunks[line] == 1:
            assert slots == [-1], (line, slots)
        else:
            assert slots == list(range(slots[0], slots[0] + len(slots))), (line, slots)
            assert not used & set(slots), (line, slots)
            used |= set(slots)


CASES = [
    # (name, block mask, batch, heads, head_dim, dtype)
    ("global 20, split row 0 and column 0", inputs.block_mask("global", 20, radius=1), 1, 3, 128, torch.bfloat16),
    ("random 40, p 0.3", inputs.block_mask("random", 40, p=0.3, seed=3), 2, 2, 128, torch.bfloat16),
    ("two rows of 32 stored", None, 1, 8, 128, torch.bfloat16),
    ("global 20 at head_dim 512 (two output slices)", inputs.block_mask("global", 20, radius=1), 1, 2, 512,
     torch.bfloat16),
    ("global 16, fp32", inputs.block_mask("global", 16, radius=2), 1, 2, 64, torch.float32),
    ("band over 2100 block rows", inputs.block_mask("local", 2100, radius=1), 1, 1, 64, torch.bfloat16),
]


@pytest.mark.parametrize("name,bm,B,H,D,dtype", CASES, ids=[c[0] for c in CASES])
def test_work_lists_follow_the_planning_rules(name, bm, B, H, D, dtype):
    if bm is None:
        bm = np.zeros((32, 32), bool)
        bm[0:2, 0:4] = True
    n = bm.shape[0]
    dev = torch.device("cuda")
    rp, ci = inputs.bsr_from_block_mask(bm)
    st = bsr.Structure(rp, ci, n, dev)
    q = torch.empty(B, H, n * 128, D, device=dev, dtype=dtype)
    plan = st.plan(q)
    cp = np.concatenate([[0], np.cumsum(bm.sum(0))])
    nnzb = int(bm.sum())
    for which, ptr in ((0, rp), (1, cp), (2, cp)):
        got, info = plan.work_list(which)
        check_list(got, info, ptr, n, nnzb)
