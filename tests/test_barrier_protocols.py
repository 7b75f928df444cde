"""The barrier protocols of the tcgen05 kernels (the paired-head forward, the
dK/dV and dQ kernels), checked in a discrete-event model (protocol_model.py)
over randomised interleavings: the committed issue orders pass every hazard
and parity check, and the planted mistakes (protocol variants that are not in
the library) are caught."""
import pytest

from protocol_model import dkdv_cta, dq_rings

SEEDS = range(60)


@pytest.mark.parametrize("steps", [1, 2, 3, 5, 8, 13])
def test_dkdv_head64_scores_a_step_ahead(steps):
    for seed in SEEDS:
        dkdv_cta(seed, steps, double_scores=True, n_stages=4)


@pytest.mark.parametrize("steps", [1, 2, 3, 5, 8, 13])
def test_dkdv_head128_order(steps):
    for seed in SEEDS:
        dkdv_cta(seed, steps, double_scores=False, n_stages=2)


@pytest.mark.parametrize("steps", [1, 2, 3, 4, 7, 16])
def test_dq_rings_with_v_released_on_dp(steps):
    for seed in SEEDS:
        dq_rings(seed, steps)


def _fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_planted_one_p_barrier_pair_for_two_score_buffers():
    """With one P^T barrier pair the elementwise groups can finish P^T(n+1)
    before the issuer has waited for P^T(n)."""
    assert any(_fails(lambda s=s: dkdv_cta(s, 8, True, 4, p_barrier_per_buffer=False)) for s in range(200))


def test_planted_ring_release_on_dp_full():
    """Reloading the two-stage Q/dO ring on dp_full: the first reload waits for
    dp_full's second completion before its first can be seen (the order that
    faulted the GPU)."""
    assert all(_fails(lambda s=s: dkdv_cta(s, 6, False, 2, release_by_dp=True)) for s in range(20))


def test_paired_forward_protocol():
    import random

    from protocol_model import fwd_pair_cta
    for seed in range(150):
        rng = random.Random(seed)
        items = [rng.randint(1, 5) for _ in range(rng.randint(1, 4))]
        fwd_pair_cta(seed, items)


def test_planted_forward_staging_without_release_wait():
    """The two heads share one staging tile: without the wait for the previous
    store to have read it, a head overwrites the tile under the copy."""
    from protocol_model import fwd_pair_cta
    assert any(_fails(lambda s=s: fwd_pair_cta(s, [2, 2, 3, 1], wait_stage_free=False)) for s in range(100))
