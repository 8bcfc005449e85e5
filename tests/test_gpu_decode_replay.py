"""Decode step, checkpoint copies and replay (append / rollback / flush)
through the C ABI against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import gated_deltanet_state_gb300 as gdn
from gated_deltanet_state_gb300 import inputs

from harness import assert_out_close, assert_state_close, dev, dims, rel_fro, OUT_TOL, STATE_TOL

pytestmark = pytest.mark.gpu


def _seed_pages(pool, pages, st):
    for i, p in enumerate(pages):
        pool.state(p).copy_(st["S"][i].cuda())
        pool.window(p).copy_(st["win"][i].cuda())


def _decode(sh, pool, slots, ti, w):
    N = len(slots)
    o = torch.full((N, sh.num_v_heads, sh.head_dim_v), float("nan"), dtype=sh.torch_out(), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_decode_step(sh, pool, x=dev(ti["x"]), g=dev(ti["g"]), beta=dev(ti["beta"]), conv_w=dev(w),
                        slot=dev(slots, torch.int32), o=o, dev_error=err)
    torch.cuda.synchronize()
    return o.cpu(), int(err.item())


@pytest.mark.parametrize("shape", [inputs.TINY, inputs.LayerShape(2, 6, 64, 64, 64, 16), inputs.QWEN4B])
def test_decode_matches_oracle(shape):
    sh = shape
    N = 5 if sh is not inputs.QWEN4B else 9
    perm = inputs.permutation(2 * N, seed=1).tolist()
    slots = perm[:N]
    st = inputs.random_state(sh, N, seed=4)
    pool = gdn.StatePool(sh, 2 * N, fill=0xFF)
    _seed_pages(pool, slots, st)
    ti = inputs.token_inputs(sh, N, seed=6)
    w = inputs.conv_weights(sh, 6)
    o, err = _decode(sh, pool, slots, ti, w)
    assert err == 0
    o_ref, S_ref, win_ref = oracle.decode(dims(sh), ti["x"], ti["g"], ti["beta"], w,
                                          st["S"].double().numpy(), st["win"].float().numpy())
    assert_out_close(o, o_ref, list(range(N + 1)))
    assert_state_close(torch.stack([pool.state(p) for p in slots]).cpu(), S_ref)
    for i, p in enumerate(slots):
        assert torch.equal(pool.window(p).cpu().float(), torch.as_tensor(win_ref[i], dtype=torch.float32))


def test_decode_chain_matches_prefill_oracle_and_batch_invariance():
    sh = inputs.LayerShape(2, 4, 128, 128, 64, 16)
    N, steps = 4, 6
    pool = gdn.StatePool(sh, N, fill=0)
    ti = inputs.token_inputs(sh, N * steps, seed=8)
    w = inputs.conv_weights(sh, 8)
    xs = ti["x"].view(steps, N, -1)
    gs = ti["g"].view(steps, N, -1)
    bs = ti["beta"].view(steps, N, -1)
    outs = []
    for t in range(steps):
        o, err = _decode(sh, pool, list(range(N)), {"x": xs[t], "g": gs[t], "beta": bs[t]}, w)
        assert err == 0
        outs.append(o)
    o_gpu = torch.stack(outs, 1)  # [N, steps, Hv, dv]
    for s in range(N):
        ref = oracle.prefill(dims(sh), [0, steps], [0], 1 << 40, xs[:, s], gs[:, s], bs[:, s], w)
        assert_out_close(o_gpu[s], ref["o"], [0, steps])
        assert_state_close(pool.state(s).cpu()[None], ref["S"])
    # batch invariance: sequence 2 alone reproduces its batched bits
    pool1 = gdn.StatePool(sh, N, fill=0)
    for t in range(steps):
        o1, _ = _decode(sh, pool1, [2], {"x": xs[t, 2:3], "g": gs[t, 2:3], "beta": bs[t, 2:3]}, w)
        assert torch.equal(o1[0].view(torch.int16), outs[t][2].view(torch.int16))
    assert torch.equal(pool1.payload(2).cpu(), pool.payload(2).cpu())


def test_decode_bad_slot_sets_error_and_skips():
    sh = inputs.TINY
    pool = gdn.StatePool(sh, 3, fill=0x11)
    before = pool.buf.cpu().clone()
    ti = inputs.token_inputs(sh, 2, seed=1)
    o, err = _decode(sh, pool, [1, 7], ti, inputs.conv_weights(sh, 1))
    assert err == gdn.STATUS_CODE["GDN_ERR_PAGE_RANGE"]
    assert torch.isnan(o[1].float()).all() and torch.isfinite(o[0].float()).all()
    assert torch.equal(pool.payload(0).cpu(), before[:sh.payload_bytes])


@pytest.mark.parametrize("sh", [inputs.TINY, inputs.QWEN27B], ids=["tiny", "27b"])
def test_checkpoint_copy_is_bit_exact_with_nan_payloads(sh):
    # the tiny payload (656 words) is copied one word per thread; the 27B-shaped
    # one (200,448 words) mostly four words per thread, then the remainder
    B = sh.block_size
    pool = gdn.StatePool(sh, 6, fill=0)
    g = torch.Generator().manual_seed(3)
    raw = torch.randint(0, 256, (sh.payload_bytes,), dtype=torch.uint8, generator=g)
    raw[:64] = 0xFF       # NaN encodings with payload bits
    raw[64:128:4] = 0x01  # denormal-looking patterns
    pool.payload(1).copy_(raw.cuda())
    pool.payload(2).copy_(raw.flip(0).cuda())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_checkpoint_resume(sh, pool, dev([1, 2], torch.int32), dev([4, 5], torch.int32), [B, 2 * B], err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(pool.payload(4).cpu(), raw)
    assert torch.equal(pool.payload(5).cpu(), raw.flip(0))
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_checkpoint_save(sh, pool, dev([4], torch.int32), dev([3], torch.int32), [B + 1], err)
    assert ei.value.status == gdn.STATUS_CODE["GDN_ERR_NOT_BLOCK_ALIGNED"]
    assert (pool.payload(3).cpu() == 0).all()
    gdn.gdn_checkpoint_save(sh, pool, dev([4], torch.int32), dev([9], torch.int32), [B], err)
    torch.cuda.synchronize()
    assert err.item() == gdn.STATUS_CODE["GDN_ERR_PAGE_RANGE"]


class Replay:
    """Device-side replay state of N requests plus the host mirror the oracle uses."""

    def __init__(self, sh, N, seed):
        self.sh, self.N = sh, N
        self.pool = gdn.StatePool(sh, N + 2, fill=0xFF)
        self.slots = inputs.permutation(N + 2, seed).tolist()[:N]
        self.st = inputs.random_state(sh, N, seed)
        _seed_pages(self.pool, self.slots, self.st)
        L = gdn.REPLAY_LOG_SLOTS
        self.log_x = torch.zeros(N, L, sh.conv_dim, dtype=sh.torch_in(), device="cuda")
        self.log_g = torch.zeros(N, L, sh.num_v_heads, device="cuda")
        self.log_b = torch.zeros(N, L, sh.num_v_heads, device="cuda")
        self.log_len = torch.zeros(N, dtype=torch.int32, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.ckpt = dev(self.slots, torch.int32)
        self.w = inputs.conv_weights(sh, seed)

    def kw(self):
        return dict(ckpt_slot=self.ckpt, log_x=self.log_x, log_g=self.log_g, log_beta=self.log_b,
                    log_len=self.log_len, conv_w=dev(self.w), dev_error=self.err)

    def append(self, ti, m):
        o = torch.full((self.N, m, self.sh.num_v_heads, self.sh.head_dim_v), float("nan"),
                       dtype=self.sh.torch_out(), device="cuda")
        gdn.gdn_replay_append(self.sh, self.pool, x_new=dev(ti["x"]).view(self.N, m, -1),
                              g_new=dev(ti["g"]).view(self.N, m, -1), beta_new=dev(ti["beta"]).view(self.N, m, -1),
                              o=o, **self.kw())
        torch.cuda.synchronize()
        return o.cpu()


def test_replay_append_rollback_flush_matches_oracle():
    sh = inputs.QWEN4B
    N, m = 16, 16
    R = Replay(sh, N, seed=21)
    d = dims(sh)
    S0 = R.st["S"].double().numpy()
    win0 = R.st["win"].float().numpy()
    # step 1: append 16 rows to empty logs
    ti = inputs.token_inputs(sh, N * m, seed=22)
    o1 = R.append(ti, m)
    assert R.err.item() == 0 and R.log_len.cpu().tolist() == [m] * N
    xs, gs, bs = ti["x"].view(N, m, -1), ti["g"].view(N, m, -1), ti["beta"].view(N, m, -1)
    z = np.zeros((N, 32, sh.conv_dim)); zg = np.zeros((N, 32, sh.num_v_heads))
    o_ref = oracle.replay_append(d, R.w, S0, win0, z, zg, zg, [0] * N, xs, gs, bs)
    assert_out_close(o1, o_ref, list(range(N + 1)))
    # the log holds the appended rows bit for bit
    assert torch.equal(R.log_x[:, :m].cpu(), xs)
    # rollback to the accepted prefix, uniform in [0, 16]
    acc = inputs.accept_lengths(N, m, seed=23)
    gdn.gdn_replay_rollback(R.log_len, dev(acc), m, R.err)
    torch.cuda.synchronize()
    assert R.err.item() == 0 and R.log_len.cpu().tolist() == acc.tolist()
    # step 2: append again on top of the kept rows, outputs from checkpoint + log
    ti2 = inputs.token_inputs(sh, N * m, seed=24)
    o2 = R.append(ti2, m)
    assert R.err.item() == 0
    log_x = R.log_x.cpu().float().numpy(); log_g = R.log_g.cpu().numpy(); log_b = R.log_b.cpu().numpy()
    o_ref2 = oracle.replay_append(d, R.w, S0, win0, log_x, log_g, log_b, acc.numpy(),
                                  ti2["x"].view(N, m, -1), ti2["g"].view(N, m, -1), ti2["beta"].view(N, m, -1))
    assert_out_close(o2, o_ref2, list(range(N + 1)))
    # rollback then flush: the checkpoint absorbs exactly the accepted rows
    acc2 = inputs.accept_lengths(N, m, seed=25)
    gdn.gdn_replay_rollback(R.log_len, dev(acc2), m, R.err)
    keep = (acc + acc2).numpy()
    log_x = R.log_x.cpu().float().numpy(); log_g = R.log_g.cpu().numpy(); log_b = R.log_b.cpu().numpy()
    gdn.gdn_replay_flush(sh, R.pool, **R.kw())
    torch.cuda.synchronize()
    assert R.err.item() == 0 and R.log_len.cpu().tolist() == [0] * N
    S_ref, win_ref = oracle.replay_flush(d, R.w, S0, win0, log_x, log_g, log_b, keep)
    assert_state_close(torch.stack([R.pool.state(p) for p in R.slots]).cpu(), S_ref)
    for r, p in enumerate(R.slots):
        assert torch.equal(R.pool.window(p).cpu().float(), torch.as_tensor(win_ref[r], dtype=torch.float32))


@pytest.mark.parametrize("rows", [1, 2, 3, 15, 16, 17, 31, 32])
def test_flush_row_sweep(rows):
    sh = inputs.LayerShape(2, 4, 128, 128, 64, 16)
    N = 3
    R = Replay(sh, N, seed=rows)
    ti = inputs.token_inputs(sh, N * rows, seed=100 + rows)
    R.append(ti, rows)
    S0 = R.st["S"].double().numpy()
    win0 = R.st["win"].float().numpy()
    gdn.gdn_replay_flush(sh, R.pool, **R.kw())
    torch.cuda.synchronize()
    assert R.err.item() == 0
    S_ref, win_ref = oracle.replay_flush(dims(sh), R.w, S0, win0, ti["x"].view(N, rows, -1),
                                         ti["g"].view(N, rows, -1), ti["beta"].view(N, rows, -1), [rows] * N)
    assert_state_close(torch.stack([R.pool.state(p) for p in R.slots]).cpu(), S_ref)
    for r, p in enumerate(R.slots):
        assert torch.equal(R.pool.window(p).cpu().float(), torch.as_tensor(win_ref[r], dtype=torch.float32))


def test_replay_device_errors():
    sh = inputs.TINY
    N = 2
    R = Replay(sh, N, seed=7)
    ti = inputs.token_inputs(sh, N * 20, seed=8)
    R.append(ti, 20)
    assert R.err.item() == 0
    # 20 + 20 > 32: overflow recorded, log untouched
    o = R.append(inputs.token_inputs(sh, N * 20, seed=9), 20)
    assert R.err.item() == gdn.STATUS_CODE["GDN_ERR_LOG_OVERFLOW"]
    assert R.log_len.cpu().tolist() == [20, 20] and torch.isnan(o.float()).all()
    R.err.zero_()
    gdn.gdn_replay_rollback(R.log_len, dev([5, 21], torch.int32), 20, R.err)
    torch.cuda.synchronize()
    assert R.err.item() == gdn.STATUS_CODE["GDN_ERR_ROLLBACK_RANGE"]
    assert R.log_len.cpu().tolist() == [5, 20]


def test_decode_and_flush_replay_identically_inside_a_cuda_graph():
    # The entry points are stream-ordered and allocate nothing, so a captured
    # sequence of calls replays the eager arithmetic bit for bit.
    sh = inputs.LayerShape(2, 4, 128, 128, 64, 16)
    N = 3
    st = inputs.random_state(sh, N, seed=31)
    ti = inputs.token_inputs(sh, N, seed=32)
    w = dev(inputs.conv_weights(sh, 32))
    pools = []
    for _ in range(2):
        pool = gdn.StatePool(sh, N, fill=0)
        _seed_pages(pool, list(range(N)), st)
        pools.append(pool)
    args = dict(x=dev(ti["x"]), g=dev(ti["g"]), beta=dev(ti["beta"]), conv_w=w, slot=dev(list(range(N)), torch.int32))
    outs = [torch.empty(N, sh.num_v_heads, sh.head_dim_v, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_decode_step(sh, pools[0], o=outs[0], dev_error=err, **args)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn.gdn_decode_step(sh, pools[1], o=outs[1], dev_error=err, **args)
    graph.replay()
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(pools[0].buf, pools[1].buf)
