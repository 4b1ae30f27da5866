"""CPU fp64 oracles for block-sparse attention and BSR SpMM (test infrastructure only).

Imported by ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg; never by the library.  See ``oracle/attention.py`` and
``oracle/spmm.py``.
"""

from .attention import (  # noqa: F401
    attn_bwd,
    attn_bwd_blockwalk,
    attn_fwd,
    attn_fwd_bwd_head,
    block_mask_from_bsr,
    bsc_from_block_mask,
    element_mask,
)
from .spmm import bsr_to_dense, spmm  # noqa: F401
