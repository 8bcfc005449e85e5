"""Tensor-core replay ("Caching less to serve more requests", "What we
changed"): the append's outputs of the new rows, computed from the checkpoint
and the log, and the flush, against the fp64 oracle at every log length and
draft length of the 32-slot log, on both sides of the 16-row switch, with
mixed log lengths in one launch, and bitwise determinism."""
import numpy as np
import pytest
import torch

import oracle
import gated_deltanet_state_gb300 as gdn
from gated_deltanet_state_gb300 import inputs

from harness import assert_out_close, assert_state_close, dev, dims

pytestmark = pytest.mark.gpu

SH = inputs.LayerShape(2, 4, 128, 128, 64, 16)          # d 128, bf16 in / out: the tensor-core path


class Log:
    def __init__(self, sh, N, seed, extra_pages=3):
        self.sh, self.N = sh, N
        self.pool = gdn.StatePool(sh, N + extra_pages, fill=0xFF)
        self.perm = inputs.permutation(N + extra_pages, seed).tolist()
        self.slots = self.perm[:N]
        self.st = inputs.random_state(sh, N, seed)
        for i, p in enumerate(self.slots):
            self.pool.state(p).copy_(self.st["S"][i].cuda())
            self.pool.window(p).copy_(self.st["win"][i].cuda())
        L = gdn.REPLAY_LOG_SLOTS
        g = torch.Generator().manual_seed(seed + 7)
        # log rows already in place (as earlier appends left them), zeros elsewhere
        self.log_x = torch.randn(N, L, sh.conv_dim, generator=g).to(sh.torch_in()).cuda()
        self.log_g = (-0.1 * torch.nn.functional.softplus(torch.randn(N, L, sh.num_v_heads, generator=g))).cuda()
        self.log_b = torch.sigmoid(torch.randn(N, L, sh.num_v_heads, generator=g)).cuda()
        self.log_len = torch.zeros(N, dtype=torch.int32, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.ckpt = dev(self.slots, torch.int32)
        self.w = inputs.conv_weights(sh, seed)

    def kw(self):
        return dict(ckpt_slot=self.ckpt, log_x=self.log_x, log_g=self.log_g, log_beta=self.log_b,
                    log_len=self.log_len, conv_w=dev(self.w), dev_error=self.err)

    def host_log(self):
        return self.log_x.cpu().float().numpy(), self.log_g.cpu().numpy(), self.log_b.cpu().numpy()

    def append(self, ti, m):
        o = torch.full((self.N, m, self.sh.num_v_heads, self.sh.head_dim_v), float("nan"),
                       dtype=self.sh.torch_out(), device="cuda")
        gdn.gdn_replay_append(self.sh, self.pool, x_new=dev(ti["x"]).view(self.N, m, -1),
                              g_new=dev(ti["g"]).view(self.N, m, -1),
                              beta_new=dev(ti["beta"]).view(self.N, m, -1), o=o, **self.kw())
        torch.cuda.synchronize()
        return o.cpu()


def _append_case(sh, lens, m, seed):
    N = len(lens)
    R = Log(sh, N, seed)
    R.log_len.copy_(torch.tensor(lens, dtype=torch.int32))
    lx, lg, lb = R.host_log()
    ti = inputs.token_inputs(sh, N * m, seed=seed + 1)
    o = R.append(ti, m)
    assert R.err.item() == 0
    assert R.log_len.cpu().tolist() == [n + m for n in lens]
    xs, gs, bs = ti["x"].view(N, m, -1), ti["g"].view(N, m, -1), ti["beta"].view(N, m, -1)
    o_ref = oracle.replay_append(dims(sh), R.w, R.st["S"].double().numpy(), R.st["win"].float().numpy(),
                                 lx, lg, lb, lens, xs, gs, bs)
    assert_out_close(o, o_ref, list(range(N + 1)))
    # the new rows sit after the kept ones, bit for bit; earlier rows untouched
    for r, n in enumerate(lens):
        assert torch.equal(R.log_x[r, n:n + m].cpu(), xs[r])
        assert torch.equal(R.log_g[r, n:n + m].cpu(), gs[r])
        assert torch.equal(R.log_b[r, n:n + m].cpu(), bs[r])
        assert np.array_equal(R.log_x[r, :n].cpu().float().numpy(), lx[r, :n])
    return R, o


@pytest.mark.parametrize("n,m", [(0, 1), (0, 16), (0, 17), (0, 32), (5, 11), (16, 1), (15, 2),
                                 (16, 16), (1, 31), (31, 1), (9, 23)])
def test_append_matches_oracle_at_every_length(n, m):
    _append_case(SH, [n] * 3, m, seed=10 * n + m)


def test_append_mixed_log_lengths_in_one_launch():
    # requests of one launch take the 16-row and the 32-row variant side by side
    _append_case(SH, [0, 16, 3, 12, 7, 1, 15, 10], 16, seed=5)


def test_append_gqa_group_of_three():
    # 3 value heads per qk head: the first head of each group copies the q / k channels
    sh = inputs.LayerShape(2, 6, 128, 128, 64, 16)
    _append_case(sh, [4, 0, 13], 9, seed=8)


def test_append_is_deterministic_and_leaves_the_checkpoint():
    R, o1 = _append_case(SH, [7, 0, 21], 11, seed=9)
    before = torch.stack([R.pool.payload(p) for p in R.slots]).cpu()
    R.log_len.copy_(torch.tensor([7, 0, 21], dtype=torch.int32))
    ti = inputs.token_inputs(SH, 3 * 11, seed=10)
    o2 = R.append(ti, 11)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(torch.stack([R.pool.payload(p) for p in R.slots]).cpu(), before)


@pytest.mark.parametrize("lens", [[1, 2, 3], [16, 17, 15], [32, 31, 30], [24, 8, 32]])
def test_flush_of_kept_logs_matches_oracle(lens):
    N = len(lens)
    R = Log(SH, N, seed=sum(lens))
    R.log_len.copy_(torch.tensor(lens, dtype=torch.int32))
    lx, lg, lb = R.host_log()
    gdn.gdn_replay_flush(SH, R.pool, **R.kw())
    torch.cuda.synchronize()
    assert R.err.item() == 0 and R.log_len.cpu().tolist() == [0] * N
    S_ref, win_ref = oracle.replay_flush(dims(SH), R.w, R.st["S"].double().numpy(), R.st["win"].float().numpy(),
                                         lx, lg, lb, lens)
    assert_state_close(torch.stack([R.pool.state(p) for p in R.slots]).cpu(), S_ref)
    for r, p in enumerate(R.slots):
        assert torch.equal(R.pool.window(p).cpu().float(), torch.as_tensor(win_ref[r], dtype=torch.float32))


def test_append_overflow_and_bad_page_are_reported():
    R = Log(SH, 2, seed=3)
    R.log_len.copy_(torch.tensor([20, 3], dtype=torch.int32))
    o = R.append(inputs.token_inputs(SH, 2 * 16, seed=4), 16)   # 20 + 16 > 32 for request 0
    assert R.err.item() == gdn.STATUS_CODE["GDN_ERR_LOG_OVERFLOW"]
    assert R.log_len.cpu().tolist() == [20, 19]
    assert torch.isnan(o[0].float()).all() and torch.isfinite(o[1].float()).all()
    R.err.zero_()
    R.ckpt.copy_(torch.tensor([R.slots[0], 99], dtype=torch.int32))
    R.log_len.copy_(torch.tensor([0, 0], dtype=torch.int32))
    o = R.append(inputs.token_inputs(SH, 2 * 4, seed=5), 4)
    assert R.err.item() == gdn.STATUS_CODE["GDN_ERR_PAGE_RANGE"]
    assert R.log_len.cpu().tolist() == [4, 0]
    assert torch.isnan(o[1].float()).all()


@pytest.mark.parametrize("lens,bjs", [([5, 16, 17, 32], [2, 16, 3, 31]), ([20, 9, 32, 1], [17, 0, 32, 1]),
                                      ([12, 30], [0, 29])])
def test_flush_writes_the_block_boundary_checkpoint(lens, bjs):
    """Replay with prefix caching: the state and conv window after the first
    j kept rows go to the boundary page, the checkpoint absorbs all rows."""
    N = len(lens)
    R = Log(SH, N, seed=sum(lens) + 3, extra_pages=N + 1)
    bpages = R.perm[N:2 * N]
    R.log_len.copy_(torch.tensor(lens, dtype=torch.int32))
    lx, lg, lb = R.host_log()
    before = {p: R.pool.payload(p).cpu().clone() for p in bpages}
    gdn.gdn_replay_flush(SH, R.pool, boundary_rows=dev(bjs, torch.int32), boundary_page=dev(bpages, torch.int32),
                         **R.kw())
    torch.cuda.synchronize()
    assert R.err.item() == 0 and R.log_len.cpu().tolist() == [0] * N
    d, S0, w0 = dims(SH), R.st["S"].double().numpy(), R.st["win"].float().numpy()
    S_ref, win_ref = oracle.replay_flush(d, R.w, S0, w0, lx, lg, lb, lens)
    assert_state_close(torch.stack([R.pool.state(p) for p in R.slots]).cpu(), S_ref)
    Sb_ref, winb_ref = oracle.replay_flush(d, R.w, S0, w0, lx, lg, lb, [max(b, 0) for b in bjs])
    for r, (p, bp, bj) in enumerate(zip(R.slots, bpages, bjs)):
        assert torch.equal(R.pool.window(p).cpu().float(), torch.as_tensor(win_ref[r], dtype=torch.float32))
        if bj > 0:
            assert_state_close(R.pool.state(bp).cpu()[None], Sb_ref[r:r + 1])
            assert torch.equal(R.pool.window(bp).cpu().float(), torch.as_tensor(winb_ref[r], dtype=torch.float32))
        else:
            assert torch.equal(R.pool.payload(bp).cpu(), before[bp])


def test_flush_boundary_errors_leave_the_request_unchanged():
    N = 3
    R = Log(SH, N, seed=41, extra_pages=N + 1)
    free = R.perm[N]
    R.log_len.copy_(torch.tensor([8, 8, 8], dtype=torch.int32))
    before = torch.stack([R.pool.payload(p) for p in R.slots]).cpu()
    # request 0: j beyond the log; 1: boundary page = its checkpoint; 2: page outside the pool
    bjs = dev([9, 4, 4], torch.int32)
    for bp, code in (([free, R.slots[1], free], "GDN_ERR_INVALID_ARG"),):
        gdn.gdn_replay_flush(SH, R.pool, boundary_rows=bjs, boundary_page=dev(bp, torch.int32), **R.kw())
        torch.cuda.synchronize()
        assert R.err.item() == gdn.STATUS_CODE[code]
    after = torch.stack([R.pool.payload(p) for p in R.slots]).cpu()
    assert torch.equal(after[:2], before[:2]) and R.log_len.cpu().tolist()[:2] == [8, 8]
    assert R.log_len.cpu().tolist()[2] == 0      # request 2 had a valid boundary
    R.err.zero_()
    R.log_len.copy_(torch.tensor([8, 8, 8], dtype=torch.int32))
    gdn.gdn_replay_flush(SH, R.pool, boundary_rows=dev([0, 0, 4], torch.int32),
                         boundary_page=dev([free, free, 1000], torch.int32), **R.kw())
    torch.cuda.synchronize()
    assert R.err.item() == gdn.STATUS_CODE["GDN_ERR_PAGE_RANGE"]
    assert R.log_len.cpu().tolist() == [0, 0, 8]
