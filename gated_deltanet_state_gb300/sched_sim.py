"""Host simulator of the serving scheduler around the GDN state engine.

"Prefix caching on Gated DeltaNet hybrids", sections "The in-page layout" and
"Correctness" (the CPU simulator with a patched scheduler, its state checks,
preemptions and mutants), and "The prefix cache changed the answer" (every
crossed boundary must be checkpointed): requests keep their recurrent state
in a compact slot; checkpoints live in KV blocks; a prefix-cache hit or a
request resumed after preemption restores its slot from a block; preemption
hands the slot back; newly handed-out blocks are zeroed; a copy off a block
boundary fails closed.

The state is symbolic: a slot or a block holds the fingerprint of the token
prefix it summarises (a chained hash), so the simulator can check, before
every step, that a request's slot holds exactly the state of the tokens it
has computed.  It drives the library's own cache arithmetic (``gdn_chunk_end``,
``gdn_resume_block``), so a wrong block boundary or resume rule shows up as a
failed check.  ``Mutation`` switches off one mechanism at a time (saves,
restores, slot hand-back, zeroing, boundary checkpoints of replay flushes):
each must make the checks fail.

Replay mode ("Caching less to serve more requests", "What we changed" and
"Other models": speculative decoding on one checkpoint plus an input log,
served with prefix caching): a decoding request keeps its checkpoint in the
slot and the kept rows in a log of REPLAY_LOG_SLOTS; each cycle appends a
draft, keeps an accepted prefix (at least the row the previous cycle's
verification produced), and flushes when the log would overflow or its rows
would cross a second block boundary.  A flush whose kept rows cross a block
boundary writes that block's checkpoint (``gdn_replay_boundary_rows``), so a
later prefix hit can resume inside the decoded tokens.
"""
from __future__ import annotations

import dataclasses
import enum
import hashlib
import random
from collections import OrderedDict

from . import REPLAY_LOG_SLOTS, gdn_chunk_end, gdn_replay_boundary_rows, gdn_resume_block

ZERO = b"zero"                  # a zeroed block or a fresh slot
POISON = b"stale-checkpoint"    # what a reused block holds if it is not zeroed


def _extend(fp: bytes, tokens) -> bytes:
    h = hashlib.blake2b(fp, digest_size=16)
    h.update(bytes(str(list(tokens)), "ascii"))
    return h.digest()


def fingerprint(tokens) -> bytes:
    """The state after `tokens` from a cold start (chained per token, so any
    split of the same tokens into steps gives the same value)."""
    fp = ZERO
    for t in tokens:
        fp = _extend(fp, [t])
    return fp


class Mutation(enum.Enum):
    NONE = "none"
    NO_SAVE = "no_save"            # boundaries are not checkpointed into their blocks
    NO_RESTORE = "no_restore"      # a hit or a resume keeps the slot's previous contents
    NO_HANDBACK = "no_handback"    # preemption keeps the slot
    NO_ZEROING = "no_zeroing"      # blocks are handed out with their old contents
    NO_BOUNDARY = "no_boundary"    # replay flushes skip the block-boundary checkpoint


class SimFailure(AssertionError):
    """A state check, a fail-closed rule or a resource invariant broke."""


@dataclasses.dataclass
class Request:
    rid: int
    tokens: list                   # prompt followed by the tokens it will generate
    prompt_len: int
    computed: int = 0
    slot: int | None = None
    blocks: list = dataclasses.field(default_factory=list)
    started: bool = False
    log_len: int = 0               # replay mode: kept rows past the slot's checkpoint


class Engine:
    """One replica: `num_blocks` KV blocks of `block` tokens, `num_slots`
    compact state slots, a token budget per step."""

    def __init__(self, block: int, num_blocks: int, num_slots: int, budget: int,
                 mutation: Mutation = Mutation.NONE, replay: bool = False, seed: int = 0):
        self.block, self.budget, self.mutation = block, budget, mutation
        self.replay = replay
        self.rng = random.Random(seed)
        self.flushes = 0
        self.boundary_saves = 0
        self.block_ckpt = [ZERO] * num_blocks        # checkpoint content of each block
        self.block_key = [None] * num_blocks         # prefix-cache key of a sealed block
        self.free_blocks = OrderedDict((b, None) for b in range(num_blocks))   # LRU of free blocks
        self.refs = [0] * num_blocks
        self.cache = {}                              # prefix key -> block id
        self.slot_state = [ZERO] * num_slots
        self.free_slots = list(range(num_slots))
        self.running: list[Request] = []
        self.waiting: list[Request] = []
        self.checks = 0
        self.preemptions = 0
        self.hits = 0

    # ---- blocks
    def _key(self, req: Request, j: int):
        return tuple(req.tokens[:(j + 1) * self.block])

    def _take_block(self) -> int:
        if not self.free_blocks:
            raise MemoryError
        b, _ = self.free_blocks.popitem(last=False)
        if self.block_key[b] is not None:          # evict its cached checkpoint
            self.cache.pop(self.block_key[b], None)
            self.block_key[b] = None
        if self.mutation != Mutation.NO_ZEROING:
            self.block_ckpt[b] = ZERO
        elif self.block_ckpt[b] != ZERO:
            self.block_ckpt[b] = POISON
        self.refs[b] = 1
        return b

    def _release(self, req: Request):
        for b in req.blocks:
            self.refs[b] -= 1
            if self.refs[b] == 0:
                self.free_blocks[b] = None           # still in the prefix cache until reused
        req.blocks = []

    def _ensure_blocks(self, req: Request, upto: int):
        need = (upto + self.block - 1) // self.block
        while len(req.blocks) < need:
            req.blocks.append(self._take_block())

    # ---- slots
    def _take_slot(self, req: Request):
        if not self.free_slots:
            raise SimFailure(f"request {req.rid}: no free state slot")
        req.slot = self.free_slots.pop()

    def _preempt(self, req: Request):
        self.preemptions += 1
        self.running.remove(req)
        self._release(req)
        if self.mutation != Mutation.NO_HANDBACK:
            self.free_slots.append(req.slot)
        req.slot = None
        # the tokens it generated join the prompt it re-prefills on resume
        req.prompt_len = max(req.prompt_len, req.computed)
        req.computed = 0
        req.log_len = 0
        req.started = False
        self.waiting.insert(0, req)

    # ---- state checks and copies
    def _check(self, req: Request):
        self.checks += 1
        absorbed = req.computed - req.log_len
        want = fingerprint(req.tokens[:absorbed])
        if self.slot_state[req.slot] != want:
            raise SimFailure(f"request {req.rid}: slot state is not the state after {absorbed} tokens")

    def _save(self, req: Request, pos: int):
        """slot -> block at a boundary (every crossed one, in-kernel)."""
        if pos % self.block:
            raise SimFailure("checkpoint save off a block boundary")
        j = pos // self.block - 1
        # the block manager caches every full block by its prefix; the state
        # copy into it is what a missing save drops
        if self.mutation != Mutation.NO_SAVE:
            self.block_ckpt[req.blocks[j]] = fingerprint(req.tokens[:pos])
        key = self._key(req, j)
        old = self.cache.get(key)
        if old is None:
            self.cache[key] = req.blocks[j]
            self.block_key[req.blocks[j]] = key

    def _start(self, req: Request):
        """Schedule a waiting request: longest cached prefix of full blocks,
        resume from the block before the hit (or cold), restore the slot."""
        self._take_slot(req)
        k = 0
        while (k + 1) * self.block <= req.prompt_len and self._key(req, k) in self.cache:
            k += 1
        hit = k * self.block
        resume = gdn_resume_block(hit, self.block) if hit else -1
        if resume >= 0:
            self.hits += 1
            # share the cached blocks up to the resume block
            for j in range(resume + 1):
                b = self.cache[self._key(req, j)]
                if self.refs[b] == 0:
                    self.free_blocks.pop(b, None)
                self.refs[b] += 1
                req.blocks.append(b)
            req.computed = (resume + 1) * self.block
            if req.computed % self.block:
                raise SimFailure("restore off a block boundary")
            if self.mutation != Mutation.NO_RESTORE:
                self.slot_state[req.slot] = self.block_ckpt[req.blocks[resume]]
        else:
            req.computed = 0
            if self.mutation != Mutation.NO_RESTORE:
                self.slot_state[req.slot] = ZERO   # a cold start never reads the pool
        req.started = True

    # ---- replay (speculative) decoding
    def _replay_flush(self, req: Request):
        """Fold the kept rows into the slot; a block boundary inside them gets
        its checkpoint (the state after the rows up to it)."""
        absorbed = req.computed - req.log_len
        j = gdn_replay_boundary_rows(absorbed, req.log_len, self.block)
        if j < 0:
            raise SimFailure("a flush crossing two block boundaries")
        if j > 0:
            pos = absorbed + j
            blk = pos // self.block - 1
            if self.mutation != Mutation.NO_BOUNDARY:
                self.block_ckpt[req.blocks[blk]] = fingerprint(req.tokens[:pos])
                self.boundary_saves += 1
            key = self._key(req, blk)
            if key not in self.cache:
                self.cache[key] = req.blocks[blk]
                self.block_key[req.blocks[blk]] = key
        self.slot_state[req.slot] = _chain(self.slot_state[req.slot], req.tokens[absorbed:req.computed])
        req.log_len = 0
        self.flushes += 1

    def _replay_cycle(self, req: Request) -> int:
        """One draft / verify cycle; returns the rows it keeps."""
        m = min(self.rng.randint(1, 8), len(req.tokens) - req.computed)
        absorbed = req.computed - req.log_len
        if req.log_len + m > REPLAY_LOG_SLOTS or gdn_replay_boundary_rows(absorbed, req.log_len + m,
                                                                          self.block) < 0:
            self._replay_flush(req)
        keep = self.rng.randint(1, m)      # the first row is the previous verification's token
        req.computed += keep
        req.log_len += keep
        return keep

    # ---- one scheduler step
    def step(self):
        budget = self.budget
        # slot accounting: every slot is free or held by a running request
        held = sum(1 for r in self.running if r.slot is not None)
        if held + len(self.free_slots) != len(self.slot_state):
            raise SimFailure("a state slot leaked: a preempted request kept it")
        if self.waiting and not self.running and not self.free_slots:
            raise SimFailure("the state slots ran dry")
        while self.waiting and self.free_slots:
            req = self.waiting.pop(0)
            self._start(req)
            self.running.append(req)
        for req in list(self.running):
            if budget <= 0 or req not in self.running:
                continue
            total = len(req.tokens)
            if req.computed < req.prompt_len:                 # prefill: block-floored chunk
                end = gdn_chunk_end(req.computed, req.prompt_len, budget, self.block)
                if end <= req.computed:
                    continue
            elif self.replay:                                 # replay: a draft of up to 8 rows
                end = min(req.computed + 8, len(req.tokens))
            else:                                             # decode: one token
                end = req.computed + 1
            try:
                self._ensure_blocks(req, end)
            except MemoryError:
                victim = self.running[-1]
                self._preempt(victim)
                if victim is req:
                    continue
                try:
                    self._ensure_blocks(req, end)
                except MemoryError:
                    self._preempt(req)
                    continue
            # attention reads every block of the request: a stale checkpoint
            # left in a reused block poisons it (NaN times zero is NaN)
            if any(self.block_ckpt[b] == POISON for b in req.blocks):
                raise SimFailure(f"request {req.rid}: reads a block that was handed out unzeroed")
            self._check(req)
            start = req.computed
            if self.replay and start >= req.prompt_len:
                budget -= self._replay_cycle(req)
            else:
                if req.log_len:
                    self._replay_flush(req)        # a prefill chunk continues from a folded log
                self.slot_state[req.slot] = _chain(self.slot_state[req.slot], req.tokens[start:end])
                req.computed = end
                for pos in range((start // self.block + 1) * self.block, end + 1, self.block):
                    self._save(req, pos)
                budget -= end - start
            if req.computed >= total:
                self.running.remove(req)
                self._release(req)
                self.free_slots.append(req.slot)
                req.slot = None

    def idle(self) -> bool:
        return not self.running and not self.waiting


def _chain(fp: bytes, tokens) -> bytes:
    for t in tokens:
        fp = _extend(fp, [t])
    return fp


def agent_workload(seed: int, sessions: int = 4, turns: int = 6, sys_len: int = 40, new_len: int = 24,
                   gen_len: int = 6, vocab: int = 50):
    """Synthetic agent traffic: every turn re-sends the whole conversation
    (shared system prompt, earlier turns and answers) plus new tokens."""
    rng = random.Random(seed)
    system = [rng.randrange(vocab) for _ in range(sys_len)]
    reqs = []
    rid = 0
    for s in range(sessions):
        history = list(system)
        for _ in range(turns):
            history = history + [rng.randrange(vocab) for _ in range(rng.randint(1, new_len))]
            answer = [rng.randrange(vocab) for _ in range(rng.randint(1, gen_len))]
            reqs.append((s, Request(rid, history + answer, len(history))))
            history = history + answer
            rid += 1
    return reqs


def simulate(seed: int, mutation: Mutation = Mutation.NONE, block: int = 8, num_blocks: int = 32,
             num_slots: int = 3, budget: int = 32, max_steps: int = 100000, replay: bool = False,
             gen_len: int = 6) -> Engine:
    """Run one seeded workload to completion; raises SimFailure on the first
    broken check.  Turns of a session arrive after the previous turn ends."""
    eng = Engine(block, num_blocks, num_slots, budget, mutation, replay=replay, seed=seed + 7)
    reqs = agent_workload(seed, gen_len=gen_len)
    rng = random.Random(seed + 1)
    pending = {}
    for s, r in reqs:
        pending.setdefault(s, []).append(r)
    active = {}
    for _ in range(max_steps):
        for s in list(pending):
            if s not in active or active[s].computed >= len(active[s].tokens) and active[s] not in eng.running:
                if pending[s]:
                    r = pending[s].pop(0)
                    active[s] = r
                    eng.waiting.insert(rng.randrange(len(eng.waiting) + 1), r)
                else:
                    del pending[s]
        if not pending and eng.idle():
            return eng
        eng.step()
    raise SimFailure("simulation did not finish")
