"""Host scheduler simulator ("Prefix caching on Gated DeltaNet hybrids",
sections "Correctness" and "The prefix cache changed the answer"): on seeded
agent traffic every state check passes with the real mechanisms, and switching
off any one of them (checkpoint saves, restores, slot hand-back on preemption,
zeroing of handed-out blocks) makes a check fail."""
import pytest

from gated_deltanet_state_gb300 import sched_sim as ss

SEEDS = range(12)


def test_fingerprint_is_split_invariant():
    toks = list(range(17))
    whole = ss.fingerprint(toks)
    assert ss._chain(ss.fingerprint(toks[:5]), toks[5:]) == whole
    assert ss._chain(ss._chain(ss.ZERO, toks[:8]), toks[8:]) == whole
    assert ss.fingerprint(toks[:-1]) != whole
    assert ss.fingerprint([]) == ss.ZERO


def test_clean_scheduler_passes_every_check():
    checks = preemptions = hits = 0
    for seed in SEEDS:
        eng = ss.simulate(seed)
        assert eng.idle()
        assert sorted(eng.free_slots) == list(range(len(eng.slot_state)))
        assert all(r == 0 for r in eng.refs)
        checks += eng.checks
        preemptions += eng.preemptions
        hits += eng.hits
    # the workload has to exercise what the mutants switch off
    assert checks > 1000
    assert preemptions >= 20
    assert hits >= 200


@pytest.mark.parametrize("mutation", [ss.Mutation.NO_SAVE, ss.Mutation.NO_RESTORE, ss.Mutation.NO_ZEROING])
def test_mutant_fails_on_every_seed(mutation):
    for seed in SEEDS:
        with pytest.raises(ss.SimFailure):
            ss.simulate(seed, mutation)


def test_kept_slot_is_caught_wherever_a_preemption_happens():
    preempting = [s for s in SEEDS if ss.simulate(s).preemptions]
    assert len(preempting) >= len(SEEDS) // 2
    for seed in preempting:
        with pytest.raises(ss.SimFailure, match="slot leaked"):
            ss.simulate(seed, ss.Mutation.NO_HANDBACK)


def test_larger_blocks_and_tighter_pool():
    # a different block size and pool pressure keep the same guarantees
    for seed in range(4):
        eng = ss.simulate(seed, block=16, num_blocks=16, num_slots=2, budget=48)
        assert eng.checks > 0
        with pytest.raises(ss.SimFailure):
            ss.simulate(seed, ss.Mutation.NO_RESTORE, block=16, num_blocks=16, num_slots=2, budget=48)


def test_save_off_a_block_boundary_fails_closed():
    eng = ss.Engine(block=8, num_blocks=4, num_slots=1, budget=8)
    req = ss.Request(0, list(range(12)), 12)
    eng._take_slot(req)
    eng._ensure_blocks(req, 12)
    with pytest.raises(ss.SimFailure, match="off a block boundary"):
        eng._save(req, 12)


REPLAY = dict(replay=True, gen_len=40, num_blocks=48)


def test_replay_mode_passes_every_check():
    """Speculative decoding on checkpoint + log with prefix caching: flushes
    write the block-boundary checkpoints that later hits resume from."""
    checks = hits = flushes = saves = preemptions = 0
    for seed in SEEDS:
        eng = ss.simulate(seed, **REPLAY)
        assert eng.idle()
        assert sorted(eng.free_slots) == list(range(len(eng.slot_state)))
        checks += eng.checks
        hits += eng.hits
        flushes += eng.flushes
        saves += eng.boundary_saves
        preemptions += eng.preemptions
    assert checks > 2000 and hits > 300 and flushes > 200 and saves > 200 and preemptions > 50


@pytest.mark.parametrize("mutation", [ss.Mutation.NO_BOUNDARY, ss.Mutation.NO_SAVE, ss.Mutation.NO_RESTORE,
                                      ss.Mutation.NO_HANDBACK, ss.Mutation.NO_ZEROING])
def test_replay_mutant_fails_on_every_seed(mutation):
    for seed in SEEDS:
        with pytest.raises(ss.SimFailure):
            ss.simulate(seed, mutation, **REPLAY)


def test_boundary_mutant_is_harmless_without_replay():
    # plain decoding writes its checkpoints step by step; the replay-only
    # mechanism switched off changes nothing there
    for seed in range(4):
        ss.simulate(seed, ss.Mutation.NO_BOUNDARY)
