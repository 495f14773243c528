"""The tensor-core kernels' mbarrier protocols, checked on the CPU with a
randomized model (tests/barrier_model.py): random interleavings and random
per-warp speeds, asserting that no barrier phase completes with arrivals for
two different blocks, that no tensor-memory buffer is overwritten before it is
read (where a protocol names its buffers) and that no run deadlocks.  The model also has to find
the lapping race of the dq kernel's earlier single dS-ready barrier, which
shows that it can see this class of bug."""
import random

import barrier_model as bm


def test_dq_protocol_alternating_ds_barriers():
    assert bm.explore(bm.dq_protocol, trials=500, seed=11) is None


def test_the_model_finds_the_single_ds_barrier_race():
    found = bm.explore(bm.dq_protocol, trials=500, seed=12, split_ds=False)
    assert found is not None
    assert any(v.startswith("ds_ready phase") for v in found["violations"])


def test_the_model_finds_tmem_buffers_overwritten_before_they_are_read():
    """Planted in the model: S_{j+1} issued without waiting for every warp's
    read of S_j, and one dS buffer where dQ_j runs after dS_{j+1} is written."""
    found = bm.explore(bm.dq_protocol, trials=500, seed=16, test_s_free=False)
    assert found is not None and any(" read S holding " in v for v in found["violations"])
    found = bm.explore(bm.dq_protocol, trials=500, seed=17, ds_buffers=1)
    assert found is not None and any("mma read ('dS', 0) holding" in v for v in found["violations"])


def test_forward_protocol():
    assert bm.explore(bm.fwd_protocol, trials=500, seed=13) is None


def test_dkdv_protocol():
    assert bm.explore(bm.dkdv_protocol, trials=500, seed=14) is None


def test_the_model_finds_p_overwritten_before_dv_reads_it():
    """Planted in the model: S^T of the next block issued ahead of dV, which
    still has to read P^T from the same TMEM columns."""
    found = bm.explore(bm.dkdv_protocol, trials=300, seed=18, s_before_dv=True)
    assert found is not None and any(v.startswith("mma read ('S', ") for v in found["violations"])


def test_the_model_reports_a_deadlock():
    never = bm.Barrier("never", 1)

    def waiter():
        yield ("wait", never, 0)

    violations, deadlocked = bm.run({"waiter": waiter()}, bm.TensorCore(), random.Random(0))
    assert deadlocked and not violations


def _explore_fwd(trials, seed, **kw):
    rng = random.Random(seed)
    for _ in range(trials):
        items = []
        for _ in range(rng.randint(1, 4)):
            n0 = rng.choice([0, 1, 1, 2, 3, 5])
            n1 = n0 + rng.choice([0, 1]) if n0 else rng.choice([0, 1, 2])
            items.append((n0, n1))  # causal: the second query tile sees one more key tile
        roles, tc = bm.fwd_loads_protocol(items, rng, **kw)
        violations, deadlocked = bm.run(roles, tc, rng)
        if violations or deadlocked:
            return items, violations, deadlocked
    return None


def test_forward_with_its_producer_shared_kv_barrier():
    assert _explore_fwd(400, 21) is None                          # bf16: K ring 2, V ring 3
    assert _explore_fwd(300, 22, kstages=4, vstages=3) is None    # fp8 Q / K: K ring 4


def test_the_model_finds_forward_tmem_overwrites():
    """Planted: S_{j+1} issued ahead of the PV_j that reads P_j from the same
    columns."""
    found = _explore_fwd(300, 34, s_before_pv=True)
    assert found is not None and any(v.startswith("mma read ('S', ") for v in found[1])


def test_dkdv_with_both_producers_shared_q_do_barrier():
    assert bm.explore(bm.dkdv_loads_protocol, trials=400, seed=23) is None
    assert bm.explore(bm.dkdv_loads_protocol, trials=300, seed=24, stages=4) is None  # D = 64


def test_the_model_notices_a_missing_producer_arrival():
    assert bm.explore(bm.dkdv_loads_protocol, trials=200, seed=25, q_full_arrivals=1) is not None


def test_dq_with_its_producer_shared_kv_barrier():
    assert bm.explore(bm.dq_loads_protocol, trials=400, seed=26) is None
    assert bm.explore(bm.dq_loads_protocol, trials=300, seed=27, kstages=5, vstages=3) is None  # D = 64


def test_fused_dq_dkdv_protocol():
    assert bm.explore(bm.dkdv_fused_protocol, trials=400, seed=31) is None
    assert bm.explore(bm.dkdv_fused_protocol, trials=300, seed=32, stages=4, ds_in_do_slot=False) is None


def _ring_runs(trials, seed, **kw):
    rng = random.Random(seed)
    for _ in range(trials):
        n = rng.randint(1, 6)
        seen = {}
        roles, tc = bm.sched_ring_protocol(n, rng, record=seen, **kw)
        violations, deadlocked = bm.run(roles, tc, rng)
        wrong = any(v != list(range(n + 1)) for v in seen.values())
        if violations or deadlocked or wrong:
            return n, seen, violations, deadlocked
    return None


def test_work_item_ring_hands_every_item_to_every_consumer():
    assert _ring_runs(400, 41, n_consumers=10) is None  # dK/dV: issuer, 8 warps, dO producer


def test_the_model_notices_an_uncounted_ring_consumer():
    assert _ring_runs(400, 42, n_consumers=10, counted_consumers=9) is not None
