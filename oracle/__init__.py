"""CPU fp64 oracles for block-sparse attention, BSR SpMM and screened SpMM (test infrastructure only).

Imported by ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg; never by the library.  See ``oracle/attention.py``,
``oracle/spmm.py`` and ``oracle/screened.py``.
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
from .screened import schwarz_mask, screened_spmm  # noqa: F401
