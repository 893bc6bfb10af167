"""fp64 CPU oracle of the Vegas hot path.  TEST INFRASTRUCTURE ONLY.

Imported by the tests, by ``__graft_entry__.smoke()`` and by ``bench.py``'s CPU
baseline leg, never by the product path.
"""
from .vegas_oracle import (  # noqa: F401
    PAGE_SIZE, gather_rows, logits_row, softmax, attention_row, verify_attention,
    capture_scores, raw_capture_logits, select_topk, select_topk_batch, summed_head_scores,
    summed_head_scores_f32, select_topk_shared_batch, select_topk_shared_batch_f32, window_select,
    window_select_batch, sparse_positions, sparse_decode, iteration,
)
