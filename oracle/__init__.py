"""fp64 CPU oracle for exact softmax attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this package:
only the test suite, the smoke check in ``__graft_entry__`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it. It
shares no code, tables or helpers with the CUDA library.

Parity status: every public function here is pinned by tests in
``tests/test_oracle.py`` (closed forms, invariants, brute force and the
worked tables the pages print). Element values of O on random inputs are not
printed by any page, so they are pinned only through those properties.
"""

from .exact import (  # noqa: F401
    attention,
    attention_rows,
    attention_brute,
    attention_online,
    merge_partials,
    probabilities,
    kv_head_of,
    visibility,
)
