"""The barrier protocols of the tcgen05 kernels (the paired-head and one-head
forwards, the dK/dV kernel, the whole dQ CTA, the QKV projection on CTA
pairs, the three kernels of the float32 split path), checked in
a discrete-event model (protocol_model.py) over randomised interleavings: the
committed issue orders pass every hazard and parity check, and the planted
mistakes (protocol variants that are not in the library) are caught."""
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
    """The paired-head forward's protocol (the bf16 and the FP8 kernels issue
    and wait in the same order), random item lengths."""
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


@pytest.mark.parametrize("n_tiles,n_kb,n_stages", [(1, 1, 2), (2, 3, 2), (3, 4, 3), (5, 2, 6), (6, 1, 6), (4, 7, 6)])
def test_projection_pair_protocol(n_tiles, n_kb, n_stages):
    from protocol_model import proj_pair
    for seed in SEEDS:
        proj_pair(seed, n_tiles, n_kb, n_stages)


def test_planted_projection_expects_one_half():
    """A stage barrier that expects one CTA's bytes completes on the first
    half to land: the pair's MMA then reads the other CTA's stale half."""
    from protocol_model import proj_pair
    assert any(_fails(lambda s=s: proj_pair(s, 4, 3, 2, expect_both=False)) for s in range(100))


def test_planted_projection_accumulator_not_released():
    """Without the wait for both CTAs' epilogues, the MMAs of tile n+2 write
    the accumulator that tile n is still being read from."""
    from protocol_model import proj_pair
    assert any(_fails(lambda s=s: proj_pair(s, 6, 1, 6, acc_empty_wait=False)) for s in range(100))


def test_planted_projection_peer_ignores_stage_release():
    """The second CTA's copies must wait for the multicast stage release too:
    its half is read by MMAs that the first CTA issues."""
    from protocol_model import proj_pair
    assert any(_fails(lambda s=s: proj_pair(s, 4, 3, 2, peer_empty_wait=False)) for s in range(100))


@pytest.mark.parametrize("k_stages,v_stages", [(3, 1), (4, 4)])
def test_dq_cta_protocol(k_stages, v_stages):
    """The dQ kernel's whole CTA (item queue, two Q buffers, deferred
    epilogues and their tile stores) at both head sizes' ring depths."""
    import random

    from protocol_model import dq_cta
    for seed in range(150):
        rng = random.Random(seed)
        items = [rng.randint(1, 5) for _ in range(rng.randint(1, 7))]
        dq_cta(seed, items, k_stages=k_stages, v_stages=v_stages)


def test_dq_accumulator_release_is_implied():
    """Dropping the wait for the epilogue two items back still passes: every
    elementwise warp reads the accumulator before its first dS arrival of the
    item that overwrites it."""
    import random

    from protocol_model import dq_cta
    for seed in range(100):
        rng = random.Random(seed)
        dq_cta(seed, [rng.randint(1, 3) for _ in range(rng.randint(3, 6))], wait_dq_free=False)


def test_planted_dq_q_reload_before_store_read():
    """The Q producer reloading a buffer before the dQ tile staged in it has
    been read by its store."""
    from protocol_model import dq_cta
    assert any(_fails(lambda s=s: dq_cta(s, [2, 1, 3, 1, 2], wait_stage_free=False)) for s in range(100))


def test_planted_dq_k_released_after_score():
    """Releasing a K stage after its score MMA (its dQ MMA still reads it):
    caught with the head-64 rings; with the head-128 rings (three K stages,
    one V stage) the V reload's wait for the previous dP already orders the
    K reload after that dQ MMA."""
    from protocol_model import dq_cta
    assert any(_fails(lambda s=s: dq_cta(s, [3, 2, 4], 4, 4, k_release_on_s=True)) for s in range(100))
    for s in range(100):
        dq_cta(s, [3, 2, 4], 3, 1, k_release_on_s=True)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 12])
def test_split_kernels_protocols(n):
    """The float32 split path's forward, dK/dV and dQ kernels."""
    from protocol_model import split_dkdv_cta, split_dq_cta, split_fwd_cta
    for seed in range(60):
        split_fwd_cta(seed, n)
        split_dkdv_cta(seed, n)
        split_dq_cta(seed, n)


def test_planted_split_variants():
    """Each dropped or moved step of the split kernels' protocols is caught:
    the softmax writing P over the previous PV's operand, a V stage reloaded
    before its PV, S^T(n+1) issued before dV(n) read P^T(n), the Q/dO stage
    released before dK read it, K stages released after their score product,
    and one score buffer for all key tiles of the dQ kernel."""
    from protocol_model import split_dkdv_cta, split_dq_cta, split_fwd_cta
    cases = [(split_fwd_cta, dict(pv_wait=False)), (split_fwd_cta, dict(v_release=False)),
             (split_dkdv_cta, dict(s_before_p=True)), (split_dkdv_cta, dict(release_after_dp=True)),
             (split_dq_cta, dict(k_release_after_s=True)), (split_dq_cta, dict(one_s_buffer=True))]
    for fn, kw in cases:
        assert any(_fails(lambda s=s: fn(s, 6, **kw)) for s in range(100)), (fn.__name__, kw)


@pytest.mark.parametrize("hd", [128, 64])
@pytest.mark.parametrize("rope", [False, True])
def test_one_head_forward_protocol(hd, rope):
    """The one-head forward at both head sizes' ring depths (K 3 / V 2 / one
    O buffer at 128; 4 / 4 / two at 64), with and without the rotating
    warps."""
    import random

    from protocol_model import fwd_one_cta
    nk, nv, no = (3, 2, 1) if hd == 128 else (4, 4, 2)
    for seed in range(100):
        rng = random.Random(seed)
        items = [rng.randint(1, 5) for _ in range(rng.randint(1, 5))]
        fwd_one_cta(seed, items, nk=nk, nv=nv, no=no, rope=rope)


def test_planted_one_head_forward_variants():
    """The Q buffer released by the score MMAs alone (the output tile staged in
    it could be overwritten under its store), the O rescale without the wait
    for the previous PV, and the score MMA waiting for a K tile to land rather
    than to be rotated."""
    from protocol_model import fwd_one_cta
    for kw in (dict(store_release=False), dict(rescale_wait=False), dict(wait_rotated_k=False, rope=True)):
        assert any(_fails(lambda s=s: fwd_one_cta(s, [3, 2, 4, 1], **kw)) for s in range(100)), kw
