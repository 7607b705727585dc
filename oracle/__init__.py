"""CPU oracle for the dynamic-vocabulary draft LM head — TEST INFRASTRUCTURE.

Plain, slow, obviously correct numpy restatement of what the method computes
(the NanoSpec / MicroSpec candidate stream, sliding-window active vocabulary,
sub-head gather, projection and top-k).  It shares no code with the CUDA path
and imports nothing from it.  Only the test suite, the package-level smoke
check and the benchmark's CPU-baseline leg may import it; the product path
never routes through it.

Every function is pinned by ``tests/test_oracle_pins.py`` against hand-worked
values, brute force on tiny inputs, exact-arithmetic cases and invariants.
No function here is "parity unpinned".
"""

from .nanospec_oracle import (  # noqa: F401
    OracleSlots,
    OracleStream,
    active_vocab,
    bf16_to_f64,
    bitmap_words,
    dense_logits,
    draft_candidates,
    gather_rows,
    project,
    slot_gather,
    slot_high_water,
    slot_project_topk,
    slot_update,
    stream_append,
    stream_init,
    sub_head_step,
    top_k,
    top_k_rows,
    topk_remap,
    union_sub_head_step,
    union_vocab,
)
