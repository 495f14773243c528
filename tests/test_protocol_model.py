"""The tensor-core kernels' mbarrier protocols, checked on the CPU with a
randomized model (tests/barrier_model.py): random interleavings and random
per-warp speeds, asserting that no barrier phase completes with arrivals for
two different blocks and that no run deadlocks.  The model also has to find
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


def test_forward_protocol():
    assert bm.explore(bm.fwd_protocol, trials=500, seed=13) is None


def test_dkdv_protocol():
    assert bm.explore(bm.dkdv_protocol, trials=500, seed=14) is None


def test_the_model_reports_a_deadlock():
    never = bm.Barrier("never", 1)

    def waiter():
        yield ("wait", never, 0)

    violations, deadlocked = bm.run({"waiter": waiter()}, bm.TensorCore(), random.Random(0))
    assert deadlocked and not violations
