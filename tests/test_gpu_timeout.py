"""Bounded device waits of the tensor-core prefill ("Prefix caching on Gated
DeltaNet hybrids", "The in-page layout": a restore that cannot be trusted
fails closed).  Every mbarrier wait of the kernel is bounded; a wait that
runs out reports GDN_ERR_TIMEOUT, drains the work already issued (with the
default bound) and releases tensor memory.  These tests make the waits run
out without any fault: `wait_cycles < 0` makes every wait of the chunk loop
report a timeout at once.  They check that the call returns, that nothing
is written, that later pieces of a call do not continue from a state an
earlier launch failed to write, and that the next call on the same stream
gives the oracle's results."""
import numpy as np
import pytest
import torch

import oracle
import gated_deltanet_state_gb300 as gdn
from gated_deltanet_state_gb300 import inputs

from harness import assert_out_close, assert_state_close, dev, dims, oracle_head, run_prefill

pytestmark = pytest.mark.gpu

TIMEOUT = gdn.STATUS_CODE["GDN_ERR_TIMEOUT"]


def _call(sh, pool, ti, w, cu, bt, slots, err, wait_cycles, max_seq_len=0, path=gdn.PREFILL_AUTO):
    T = int(cu[-1])
    n = len(cu) - 1
    o = torch.full((T, sh.num_v_heads, sh.head_dim_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_prefill_chunked(sh, pool, cu_seqlens=dev(cu, torch.int32), start_pos=dev([0] * n, torch.int64),
                            init_page=dev([-1] * n, torch.int32), block_table=dev(bt, torch.int32),
                            out_slot=dev(slots, torch.int32), x=dev(ti["x"]), g=dev(ti["g"]),
                            beta=dev(ti["beta"]), conv_w=dev(w), o=o, dev_error=err,
                            start_pos_host=[0] * n, init_page_host=[-1] * n, max_seq_len=max_seq_len,
                            wait_cycles=wait_cycles, path=path)
    torch.cuda.synchronize()
    return o


def test_every_wait_running_out_writes_nothing_and_the_next_call_is_exact():
    sh = inputs.LayerShape(2, 6, 128, 128, block_size=128, chunk_size=64)
    lens = [300, 200]
    cu = np.concatenate([[0], np.cumsum(lens)])
    ti = inputs.token_inputs(sh, int(cu[-1]), seed=71)
    w = inputs.conv_weights(sh, 71)
    bt = [[2, 3], [4, -1]]
    pool = gdn.StatePool(sh, 5, fill=0x5A)
    before = pool.buf.cpu().clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = _call(sh, pool, ti, w, cu, bt, [0, 1], err, wait_cycles=-1)
    assert err.item() == TIMEOUT
    assert torch.equal(pool.buf.cpu(), before)               # no state, checkpoint or window
    assert torch.isnan(o.float()).all()                      # no output
    # the context is intact: the same call with the default bound, on the
    # same stream, gives the oracle's results
    o2, err2, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, cu, [0, 0], [-1, -1], bt, [0, 1])
    assert err2 == 0
    ref = oracle.prefill(dims(sh), cu, [0, 0], sh.block_size, ti["x"], ti["g"], ti["beta"], w)
    assert_out_close(o2, ref["o"], cu)
    assert_state_close(torch.stack([pool.state(0), pool.state(1)]).cpu(), ref["S"])
    assert_state_close(torch.stack([pool.state(p) for p in (2, 3, 4)]).cpu(), ref["ck_S"])


@pytest.mark.parametrize("case", ["levels", "one_level"])
def test_the_chain_kernel_does_not_start_after_a_run_out(case):
    """On the two-kernel path a chain launch that finds GDN_ERR_TIMEOUT in the
    error word stands down: the word stands for a wait that ran out in an
    earlier launch of the call (the chunk kernel, or the level before), whose
    images or state cannot be trusted.  Nothing is written, neither by any
    level (the overlapped levels of a 4,133-token sequence of the 27B-shaped
    layer, or the single launch of two short ones) nor by the window pass; the
    next call with a clear word is exact."""
    if case == "levels":
        sh, lens, heads = inputs.QWEN27B, [4133], (0, 47)
        plan = gdn.gdn_prefill_plan_for(sh, 1, 4133, 0, gdn.PREFILL_TWO_KERNELS)
        if plan["chunk_launches"] < 2:
            pytest.skip(f"this GPU runs the two kernels one after the other: {plan}")
    else:
        sh, lens, heads = inputs.LayerShape(2, 6, 128, 128, block_size=128, chunk_size=64), [300, 200], None
    N, B = len(lens), sh.block_size
    cu = np.concatenate([[0], np.cumsum(lens)])
    ti = inputs.token_inputs(sh, int(cu[-1]), seed=74)
    w = inputs.conv_weights(sh, 74)
    nb = max(lens) // B
    bt = [[N + s * nb + j if (j + 1) * B <= lens[s] else -1 for j in range(nb)] for s in range(N)]
    pool = gdn.StatePool(sh, N + N * nb, fill=0x5A)
    before = pool.buf.cpu().clone()
    err = torch.full((1,), TIMEOUT, dtype=torch.int32, device="cuda")
    o = _call(sh, pool, ti, w, cu, bt, list(range(N)), err, wait_cycles=0, max_seq_len=max(lens),
              path=gdn.PREFILL_TWO_KERNELS)
    assert err.item() == TIMEOUT
    assert torch.equal(pool.buf.cpu(), before)
    assert torch.isnan(o.float()).all()
    err.zero_()
    o = _call(sh, pool, ti, w, cu, bt, list(range(N)), err, wait_cycles=0, max_seq_len=max(lens),
              path=gdn.PREFILL_TWO_KERNELS)
    assert err.item() == 0
    if heads is None:
        ref = oracle.prefill(dims(sh), cu, [0] * N, B, ti["x"], ti["g"], ti["beta"], w)
        assert_out_close(o, ref["o"], cu)
        assert_state_close(torch.stack([pool.state(s) for s in range(N)]).cpu(), ref["S"])
    else:
        for h in heads:
            ref = oracle_head(sh, ti["x"], ti["g"], ti["beta"], w, h, cu, [0] * N, B)
            assert_out_close(o[:, h:h + 1], ref["o"], cu)
            assert_state_close(pool.state(0).cpu()[None, h:h + 1], ref["S"])


def _piece_case(seed):
    """27B-shaped heads with block 256: 4 x 1,024 tokens are 192 chains, more
    than the SMs, so the call runs as pieces of 8 chunks over two levels."""
    sh = inputs.with_(inputs.QWEN27B, block_size=256)
    N, L = 4, 1024
    plan = gdn.gdn_prefill_plan_for(sh, N, L, 0, gdn.PREFILL_FUSED)
    if plan["levels"] < 2:
        pytest.skip(f"this GPU runs the call in one level: {plan}")
    cu = np.arange(0, N * L + 1, L)
    ti = inputs.token_inputs(sh, N * L, seed=seed)
    w = inputs.conv_weights(sh, seed)
    nb = L // sh.block_size
    bt = [[N + s * nb + j for j in range(nb)] for s in range(N)]
    return sh, N, L, cu, ti, w, bt, plan


def test_a_run_out_on_the_piece_schedule_writes_nothing():
    sh, N, L, cu, ti, w, bt, plan = _piece_case(72)
    pool = gdn.StatePool(sh, N + N * len(bt[0]), fill=0x5A)
    before = pool.buf.cpu().clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = _call(sh, pool, ti, w, cu, bt, list(range(N)), err, wait_cycles=-1, max_seq_len=L)
    assert err.item() == TIMEOUT
    assert torch.equal(pool.buf.cpu(), before)
    assert torch.isnan(o.float()).all()


def test_later_pieces_do_not_continue_after_a_run_out():
    """An error word that already holds GDN_ERR_TIMEOUT when the call starts
    stands for a wait that ran out in an earlier launch of the call: the first
    pieces run (their waits do not run out), every later piece and the window
    pass write nothing, so no checkpoint past the first piece is written from
    a state that may be stale."""
    sh, N, L, cu, ti, w, bt, plan = _piece_case(73)
    P = plan["piece_chunks"] * 64                    # tokens of a first piece
    pool = gdn.StatePool(sh, N + N * len(bt[0]), fill=0x5A)
    before = pool.buf.cpu().clone()
    err = torch.full((1,), TIMEOUT, dtype=torch.int32, device="cuda")
    o = _call(sh, pool, ti, w, cu, bt, list(range(N)), err, wait_cycles=0, max_seq_len=L,
              path=gdn.PREFILL_FUSED).cpu()
    assert err.item() == TIMEOUT
    B = sh.block_size
    for s in range(N):
        for j, page in enumerate(bt[s]):
            written = (j + 1) * B <= P
            same = torch.equal(pool.payload(page).cpu(), before[page * sh.page:page * sh.page + sh.payload_bytes])
            # windows come from the window pass, which a run-out skips
            assert torch.equal(pool.window(page).cpu().view(-1).view(torch.uint8),
                               before[page * sh.page + sh.state_bytes:page * sh.page + sh.payload_bytes])
            assert same != written, (s, j)
        # the final slot holds the state after the first piece
        assert not torch.equal(pool.state(s).cpu().view(torch.int32).flatten()[:4],
                               before[s * sh.page:s * sh.page + 16].view(torch.int32))
        assert torch.isnan(o[cu[s] + P:cu[s + 1]].float()).all()
    for h in (0, 47):
        ref = oracle_head(sh, ti["x"], ti["g"], ti["beta"], w, h, cu, [0] * N, B)
        per = len(ref["ck_S"]) // N
        for s in range(N):
            a, b = int(cu[s]), int(cu[s]) + P
            assert_out_close(o[a:b, h:h + 1], ref["o"][a:b], [0, P])
            for j in range(P // B):
                assert_state_close(pool.state(bt[s][j]).cpu()[None, h:h + 1], ref["ck_S"][s * per + j][None])
            # after the first piece the final slot holds exactly the state of
            # the checkpoint at the piece's end (both come from one tensor-memory state)
            assert torch.equal(pool.state(s).cpu()[h].view(torch.int32),
                               pool.state(bt[s][P // B - 1]).cpu()[h].view(torch.int32))
