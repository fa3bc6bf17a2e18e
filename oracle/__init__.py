"""fp64 CPU oracle for packed variable-length (TND) attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
link this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library, and the CUDA library never feeds it inputs or
expected values.

Source of the definitions: the web page "CANN/ops-transformer
FlashAttention梯度V2", which documents the Ascend operator
aclnnFlashAttentionUnpaddingScoreGradV2 (called "the FAG-V2 page" in this
package's docstrings).  Every function cites the section of that page it
restates.

Parity status: every public function here is pinned by the CPU tests in
``tests/test_oracle.py`` (finite differences, closed forms, invariants, torch
fp64 autograd and the page's own call example).  No function is "parity
unpinned".
"""

from .attention import (  # noqa: F401
    mode_window,
    window_allowed,
    keep_bits_unit,
    unit_logits,
    unit_forward,
    unit_backward,
    unit_backward_rows,
    unit_backward_cols,
    varlen_forward,
    varlen_backward,
    mask_bit_offsets,
    cu_seqlens,
)
