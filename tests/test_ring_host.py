"""Host logic of the ring-attention steps (CPU): the kind of each (query chunk, key chunk)
step equals what the oracle's mask on global positions leaves of that block."""
import numpy as np
import pytest

from oracle import ring as oring
from ulysses_sequence_seq_gb300.ring import step_kind


def oracle_block_kind(q_rank, k_rank, L, causal):
    q = np.zeros((1, L, 1), dtype=np.uint16)
    seen = np.zeros((L, L), dtype=bool)
    # which (i, j) pairs the oracle's chunk attention lets through, read from its lse:
    # a one-key chunk at global position k_rank * L + j is visible to row i iff lse_i > -inf
    for j in range(L):
        _, lse = oring.chunk_attn_fwd(q, q[:, j:j + 1], q[:, j:j + 1], q_rank * L, k_rank * L + j, causal)
        seen[:, j] = np.isfinite(lse[0])
    if seen.all():
        return "full"
    if not seen.any():
        return "none"
    assert np.array_equal(seen, np.tril(np.ones((L, L), dtype=bool)))
    return "causal"


@pytest.mark.parametrize("causal", [True, False])
def test_step_kind_matches_the_mask_on_global_positions(causal):
    for q_rank in range(4):
        for k_rank in range(4):
            assert step_kind(q_rank, k_rank, causal) == oracle_block_kind(q_rank, k_rank, 5, causal)
