"""CPU oracle of one batched DMTP speculative-decoding round.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The CUDA library never
calls it and shares no code with it.

Plain, slow float64 NumPy. Weights arrive as the same bf16- (or fp32-) valued
tensors the GPU receives and are upcast to float64. Every function cites the page
passage it follows. Pins live in ``tests/test_oracle_*.py``.

Parity unpinned: no page prints a worked numeric example of the round, so no value
of the round is pinned to a printed number. The steps are pinned instead by
library special cases (torch fp64 routines), closed forms, invariants (losslessness,
causality, window, swap == recompute) and reductions (W = 0, identity MTP block).
"""
from .dmtp_oracle import (OracleModel, SeqState, attend_rows, gdn_step,
                          mean_accept_len, first_candidate_acceptance,
                          rms_norm, rope, silu)

__all__ = ["OracleModel", "SeqState", "attend_rows", "gdn_step", "mean_accept_len",
           "first_candidate_acceptance", "rms_norm", "rope", "silu"]
