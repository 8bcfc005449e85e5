"""Prefill through the C ABI against the fp64 oracle, plus the bitwise
determinism contract (run to run, batch invariance, cold = resume)."""
import numpy as np
import pytest
import torch

import oracle
import gated_deltanet_state_gb300 as gdn
from gated_deltanet_state_gb300 import inputs

from harness import (assert_out_close, assert_state_close, dims, oracle_head, run_prefill)

pytestmark = pytest.mark.gpu


def _tiny():
    sh = inputs.TINY
    ti = inputs.token_inputs(sh, 256, seed=0)
    return sh, ti["x"], ti["g"], ti["beta"], inputs.conv_weights(sh, 0)


def test_tiny_cold_matches_oracle_and_checkpoints():
    sh, x, g, beta, w = _tiny()
    pool = gdn.StatePool(sh, 8, fill=0xFF)  # NaN-poisoned pages must not leak
    # checkpoints at 64, 128, 192; block 3 (the end of the prompt) has no page
    o, err, _ = run_prefill(sh, pool, x, g, beta, w, [0, 256], [0], [-1], [[5, 2, 7, -1]], [0])
    assert err == 0
    ref = oracle.prefill(dims(sh), [0, 256], [0], sh.block_size, x, g, beta, w)
    assert np.isfinite(o.numpy()).all()
    assert_out_close(o, ref["o"], [0, 256])
    assert_state_close(pool.state(0).cpu()[None], ref["S"])
    for jb, page in enumerate([5, 2, 7]):
        assert_state_close(pool.state(page).cpu()[None], ref["ck_S"][jb][None])
        assert torch.equal(pool.window(page).cpu(), torch.as_tensor(ref["ck_win"][jb], dtype=torch.float32))
    assert torch.equal(pool.window(0).cpu(), x[-3:])
    # the unused pages keep their poison
    assert (pool.payload(1).cpu() == 0xFF).all()


def test_tiny_resume_from_other_request_is_bitwise_cold():
    sh, x, g, beta, w = _tiny()
    pool = gdn.StatePool(sh, 8, fill=0)
    # request A: 200 tokens, writes blocks 0..2 (64, 128, 192) into pages 1..3
    run_prefill(sh, pool, x[:200], g[:200], beta[:200], w, [0, 200], [0], [-1], [[1, 2, 3, -1]], [4])
    # request B: 256 tokens sharing A's first 192, cold
    o_cold, err, _ = run_prefill(sh, pool, x, g, beta, w, [0, 256], [0], [-1], [[-1, -1, -1, -1]], [5])
    assert err == 0
    # B resumed from A's block 2 (hit at 3 blocks -> block 2)
    assert gdn.gdn_resume_block(192, 64) == 2
    o_res, err, _ = run_prefill(sh, pool, x[192:], g[192:], beta[192:], w, [0, 64], [192], [3],
                                [[-1, -1, -1, -1]], [6])
    assert err == 0
    assert torch.equal(o_res.view(torch.int32), o_cold[192:].view(torch.int32))
    assert torch.equal(pool.state(6).cpu().view(torch.int32), pool.state(5).cpu().view(torch.int32))
    assert torch.equal(pool.window(6).cpu(), pool.window(5).cpu())


@pytest.mark.parametrize("d", [32, 64, 128])
def test_ragged_batch_bf16_matches_oracle(d):
    sh = inputs.LayerShape(2, 4, d, d, block_size=64, chunk_size=16)
    lens = [100, 37, 0, 1, 70]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    ti = inputs.token_inputs(sh, T, seed=d)
    w = inputs.conv_weights(sh, d)
    N = len(lens)
    nb = 2
    bt = np.full((N, nb), -1)
    page = N
    for s in range(N):
        for jb in range(lens[s] // 64):
            bt[s, jb] = page
            page += 1
    pool = gdn.StatePool(sh, page, fill=0xFF)
    o, err, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, cu, [0] * N, [-1] * N, bt,
                            list(range(N)))
    assert err == 0
    ref = oracle.prefill(dims(sh), cu, [0] * N, 64, ti["x"], ti["g"], ti["beta"], w)
    assert_out_close(o, ref["o"], cu)
    for s in range(N):
        assert_state_close(pool.state(s).cpu()[None], ref["S"][s][None])
    k = 0
    for s in range(N):
        for jb in range(lens[s] // 64):
            assert_state_close(pool.state(int(bt[s, jb])).cpu()[None], ref["ck_S"][k][None])
            assert torch.equal(pool.window(int(bt[s, jb])).cpu().float(),
                               torch.as_tensor(ref["ck_win"][k], dtype=torch.float32))
            k += 1
    # empty sequence: final state is the (zero) cold state, window zeros
    assert (pool.state(2).cpu() == 0).all() and (pool.window(2).cpu() == 0).all()


def test_resume_with_start_state_matches_oracle():
    sh = inputs.LayerShape(2, 4, 64, 64, block_size=64, chunk_size=16)
    st = inputs.random_state(sh, 1, seed=11)
    ti = inputs.token_inputs(sh, 130, seed=12)
    w = inputs.conv_weights(sh, 12)
    pool = gdn.StatePool(sh, 4, fill=0)
    pool.state(1).copy_(st["S"][0].cuda())
    pool.window(1).copy_(st["win"][0].cuda())
    # resume at 128 (two full blocks) from page 1; boundaries 192 cross at token 64
    o, err, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, [0, 130], [128], [1],
                            [[-1, -1, 2, -1]], [1])   # in place: out_slot == init_page
    assert err == 0
    ref = oracle.prefill(dims(sh), [0, 130], [128], 64, ti["x"], ti["g"], ti["beta"], w,
                         st["S"].double().numpy(), st["win"].float().numpy())
    assert_out_close(o, ref["o"], [0, 130])
    assert_state_close(pool.state(1).cpu()[None], ref["S"])
    assert_state_close(pool.state(2).cpu()[None], ref["ck_S"][0][None])
    assert torch.equal(pool.window(1).cpu(), ti["x"][-3:])


def test_run_to_run_and_batch_invariance_bitwise():
    sh = inputs.LayerShape(4, 8, 128, 128, block_size=128, chunk_size=64)
    lens = [300, 129, 256]
    cu = np.concatenate([[0], np.cumsum(lens)])
    ti = inputs.token_inputs(sh, int(cu[-1]), seed=5)
    w = inputs.conv_weights(sh, 5)
    N = 3
    bt = [[3 + 3 * s + jb if jb < lens[s] // 128 else -1 for jb in range(3)] for s in range(N)]
    runs = []
    for _ in range(2):
        pool = gdn.StatePool(sh, 16, fill=0)
        o, err, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, cu, [0] * N, [-1] * N, bt, [0, 1, 2])
        assert err == 0
        runs.append((o, pool.buf.cpu()))
    assert torch.equal(runs[0][0].view(torch.int16), runs[1][0].view(torch.int16))
    assert torch.equal(runs[0][1], runs[1][1])
    # sequence 1 alone equals sequence 1 inside the batch
    pool = gdn.StatePool(sh, 16, fill=0)
    a, b = int(cu[1]), int(cu[2])
    o1, err, _ = run_prefill(sh, pool, ti["x"][a:b], ti["g"][a:b], ti["beta"][a:b], w, [0, b - a], [0], [-1],
                             [bt[1]], [1])
    assert torch.equal(o1.view(torch.int16), runs[0][0][a:b].view(torch.int16))
    assert torch.equal(pool.state(1).cpu(), runs[0][1][1 * sh.page:1 * sh.page + sh.state_bytes].view(torch.float32)
                       .view(sh.num_v_heads, sh.head_dim_v, sh.head_dim_k))


def test_27b_shape_multi_block_matches_oracle():
    sh = inputs.QWEN27B
    lens = [1000, 1800]
    cu = np.concatenate([[0], np.cumsum(lens)])
    ti = inputs.token_inputs(sh, int(cu[-1]), seed=2)
    w = inputs.conv_weights(sh, 2)
    perm = inputs.permutation(8, seed=2).tolist()
    bt = [[perm[0], -1, -1], [perm[1], perm[2], -1]]
    pool = gdn.StatePool(sh, 8, fill=0xFF)
    o, err, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, cu, [0, 0], [-1, -1], bt,
                            [perm[3], perm[4]])
    assert err == 0
    ref = oracle.prefill(dims(sh), cu, [0, 0], sh.block_size, ti["x"], ti["g"], ti["beta"], w)
    assert_out_close(o, ref["o"], cu)
    assert_state_close(torch.stack([pool.state(perm[3]), pool.state(perm[4])]).cpu(), ref["S"])
    for k, page in enumerate([perm[0], perm[1], perm[2]]):
        assert_state_close(pool.state(page).cpu()[None], ref["ck_S"][k][None])
        assert torch.equal(pool.window(page).cpu().float(), torch.as_tensor(ref["ck_win"][k], dtype=torch.float32))


def test_device_errors_skip_writes():
    sh = inputs.TINY
    ti = inputs.token_inputs(sh, 64, seed=3)
    w = inputs.conv_weights(sh, 3)
    pool = gdn.StatePool(sh, 4, fill=0x7F)
    before = pool.buf.cpu().clone()
    # out_slot outside the pool: the sequence is skipped, the error recorded
    o, err, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, [0, 64], [0], [-1], [[1]], [9])
    assert err == gdn.STATUS_CODE["GDN_ERR_PAGE_RANGE"]
    assert torch.equal(pool.buf.cpu(), before)
    assert torch.isnan(o.float()).all()
    # a checkpoint page outside the pool: error, the rest is still written
    o, err, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, [0, 64], [0], [-1], [[11]], [2])
    assert err == gdn.STATUS_CODE["GDN_ERR_PAGE_RANGE"]
    assert torch.isfinite(o.float()).all()
