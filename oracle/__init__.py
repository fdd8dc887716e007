"""fp64 CPU oracle of the language-model loss head (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  It shares no code with ``lm_head_linear_fwd_gb300``.
"""
from .lm_head_ce import (  # noqa: F401
    BlockwiseError, ce_backward, ce_forward, divisor, flce_backward, flce_forward, flce_logits,
    logsumexp_rows, max_rel_err, normwise_err, packed_document_labels, scale, valid_rows,
)
