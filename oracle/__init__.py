"""CPU fp64 oracle of the dual-mode attention forward pass.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` use it; the CUDA library and its
Python binding never import it.
"""

from .attention import (MODE_BIDIRECTIONAL, MODE_CAUSAL, attention,  # noqa: F401
                        kv_head_of, log_sum_exp, masked_softmax, scores,
                        visible_mask, weighted_values)
