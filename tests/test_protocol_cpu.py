"""The mbarrier protocols of the persistent dQ kernel (split algorithm) and of the forward
kernel, run through the discrete-event model in protocol_model.py under random
interleavings of their roles, copies and products: no wait passes early or aliases a
later phase, no arrival lands in the wrong phase, no buffer is read with other data than
the code relies on, and nothing deadlocks.  Each model is also shown to catch the race it
guards against.  CPU only."""

import random

import pytest

import protocol_model as pm

SEEDS = range(250)


def _tiles(seed, lo):
    r = random.Random(seed)
    return [r.randint(lo, 5) for _ in range(r.randint(1, 7))], r.choice([2, 3])


@pytest.mark.parametrize("kst", [3])
def test_dq_kernel_protocol(kst):
    for seed in SEEDS:
        totals, warps = _tiles(seed, 0)
        sim = pm.Sim(seed)
        pm.dq_kernel(sim, totals, warps=warps, kst=kst)
        try:
            sim.run()
        except pm.ProtocolError as e:
            raise AssertionError(f"seed {seed}, tiles {totals}, warps {warps}: {e}") from None


def test_dq_model_catches_single_ds_barrier():
    """One dS-full barrier for every step (the kernel's earlier form): a warp that has
    finished step j can arrive for step j+1 before a slower warp arrives for step j."""
    caught = 0
    for seed in SEEDS:
        totals, _ = _tiles(seed, 1)
        sim = pm.Sim(seed)
        pm.dq_kernel(sim, totals, warps=2, dsfull_per_parity=False)
        try:
            sim.run()
        except pm.ProtocolError:
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("two_issuers", [True, False])
def test_forward_protocol(two_issuers):
    for seed in SEEDS:
        nvis, warps = _tiles(seed, 0)
        sim = pm.Sim(seed)
        pm.forward_kernel(sim, nvis, warps=warps, two_issuers=two_issuers)
        try:
            sim.run()
        except pm.ProtocolError as e:
            raise AssertionError(f"seed {seed}, items {nvis}, warps {warps}: {e}") from None


def test_forward_score_products_need_the_pd_wait_with_two_issuers():
    """With one issuing thread a score product may follow the P V product whose P it
    overwrites without waiting (the products run in issue order); with two issuers that
    wait is what keeps P intact."""
    caught = {True: 0, False: 0}
    for two in (True, False):
        for seed in SEEDS:
            nvis, _ = _tiles(seed, 1)
            sim = pm.Sim(seed)
            pm.forward_kernel(sim, nvis, warps=2, two_issuers=two, s_waits_pd=False)
            try:
                sim.run()
            except pm.ProtocolError:
                caught[two] += 1
    assert caught[True] > 0
    assert caught[False] == 0


def test_model_flags_premature_and_aliased_waits():
    sim = pm.Sim(0)
    sim.barrier("B")

    def early():
        yield ("wait", "B", 1)  # phase 0 incomplete: parity 0 != 1 lets it through at once

    sim.add("early", early())
    with pytest.raises(pm.ProtocolError, match="passes with only 0"):
        sim.run()

    sim = pm.Sim(0)
    sim.barrier("B")

    def late():
        yield ("arrive", "B", 0)
        yield ("arrive", "B", 1)
        yield ("wait", "B", 0)  # two phases done: the parity names phase 2

    sim.add("late", late())
    with pytest.raises(pm.ProtocolError, match="parity aliases"):
        sim.run()


@pytest.mark.parametrize("kst", [1, 2])
@pytest.mark.parametrize("issuers", [1, 2])
def test_main_kernel_protocol(kst, issuers):
    """The fused main kernel as built (one MMA issuer) and the split of its MMA issue over
    two threads (S / dP and dV / dK / dQ) with the extra completion wait that split needs."""
    for seed in SEEDS:
        tiles, warps = _tiles(seed, 0)
        sim = pm.Sim(seed)
        pm.main_kernel(sim, tiles, warps=warps, drains=2, kst=kst, issuers=issuers)
        try:
            sim.run()
        except pm.ProtocolError as e:
            raise AssertionError(f"seed {seed}, tiles {tiles}, warps {warps}: {e}") from None


def test_main_model_catches_do_reuse_with_two_issuers():
    caught = 0
    for seed in SEEDS:
        tiles, _ = _tiles(seed, 1)
        sim = pm.Sim(seed)
        pm.main_kernel(sim, tiles, warps=2, drains=2, issuers=2, do_waits_dp=False)
        try:
            sim.run()
        except pm.ProtocolError:
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("s_behind", [True, False])
def test_dkdv_kernel_protocol(s_behind):
    """The split algorithm's dK/dV kernel, with S_i+1 / dP_i+1 queued right behind dK_i
    (as built) and after dV_i / dK_i have completed (its earlier form)."""
    for seed in SEEDS:
        r = random.Random(seed)
        total, warps = r.randint(0, 9), r.choice([2, 3])
        sim = pm.Sim(seed)
        pm.dkdv_kernel(sim, total, warps=warps, s_behind=s_behind)
        try:
            sim.run()
        except pm.ProtocolError as e:
            raise AssertionError(f"seed {seed}, steps {total}, warps {warps}: {e}") from None


@pytest.mark.parametrize("kst", [1, 2])
def test_main_kernel_ordered_mode_protocol(kst):
    for seed in SEEDS:
        tiles, warps = _tiles(seed, 0)
        sim = pm.Sim(seed)
        pm.main_kernel(sim, tiles, warps=warps, drains=2, kst=kst, ordered=True)
        try:
            sim.run()
        except pm.ProtocolError as e:
            raise AssertionError(f"seed {seed}, tiles {tiles}, warps {warps}: {e}") from None


@pytest.mark.parametrize("nst", [1, 2])
def test_wide_backward_protocol(nst):
    """The wide backward (head dims above 128) with one and two Q / dO stages."""
    for seed in SEEDS:
        r = random.Random(seed)
        total, warps = r.randint(0, 9), r.choice([2, 3])
        sim = pm.Sim(seed)
        pm.wide_bwd_kernel(sim, total, nst=nst, warps=warps)
        try:
            sim.run()
        except pm.ProtocolError as e:
            raise AssertionError(f"seed {seed}, steps {total}, warps {warps}: {e}") from None
