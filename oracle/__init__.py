"""fp64 CPU oracle for the attention forward: test infrastructure only.

Imported by tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
reference legs; the CUDA library never uses it.
"""
from .attention import (NEG_INF, attention, attention_head, attention_rows, attention_state_head,  # noqa: F401
                        attention_states, bf16_to_f64, finish_state, merge_states, online_softmax_attention,
                        softmax_naive, softmax_safe, softmax_stats, visible, visible_row, visible_rows)
