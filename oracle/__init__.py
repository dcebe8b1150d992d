"""CPU oracle of the sliding-window GQA token path (and of the full-sequence
attention beside it): test infrastructure only.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
leg may import this package; the product path never does.
"""
from .swa_oracle import (  # noqa: F401
    WIN_LEN, WIN_HEAD, FAR_LEN, WINDOW,
    ring_modulus, rope_table, rotate_head, unit_head, prep, prep_ring_slot,
    prep_ring_write, row_window, row_key_list, sigmoid_gate, attend_row, attend,
    commit_slot, commit_meta, commit, rollback_meta, rollback,
    far_evict, far_evictions, far_part, far_row_state, attend_far_row, attend_far, far_commit,
    flash_row, flash_attention,
)
