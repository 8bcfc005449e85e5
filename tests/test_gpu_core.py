"""The packed core ("Hybrid linear attention (gated DeltaNet)", "Packed-core
traces"): packed q | k | v | z and b | a rows in, gated-normalised value rows
out, against the fp64 oracle (oracle.core_prefill / core_decode)."""
import numpy as np
import pytest
import torch

import oracle
import gated_deltanet_state_gb300 as gdn
from gated_deltanet_state_gb300 import inputs

from harness import assert_out_close, assert_state_close, dev, dims

pytestmark = pytest.mark.gpu


def _core_inputs(sh, T, seed):
    g = torch.Generator().manual_seed(seed)
    qkvz = torch.randn(T, sh.conv_dim + sh.num_v_heads * sh.head_dim_v, generator=g).to(sh.torch_in())
    ba = torch.randn(T, 2 * sh.num_v_heads, generator=g).to(sh.torch_in())
    A_log = torch.log(0.05 + 0.45 * torch.rand(sh.num_v_heads, generator=g)).float()
    dt_bias = (0.5 * torch.randn(sh.num_v_heads, generator=g)).float()
    norm_w = (1.0 + 0.1 * torch.randn(sh.head_dim_v, generator=g)).float()
    return qkvz, ba, A_log, dt_bias, norm_w


NORM_EPS = 1e-6


@pytest.mark.parametrize("path", [gdn.PREFILL_FUSED, gdn.PREFILL_TWO_KERNELS], ids=["fused", "two_kernels"])
def test_core_prefill_matches_oracle_cold_and_resumed(path):
    sh = inputs.LayerShape(2, 6, 128, 128, block_size=128, chunk_size=64)
    lens = [300, 65, 200]
    start = [0, 0, 256]
    init = [-1, -1, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    qkvz, ba, A_log, dt_bias, norm_w = _core_inputs(sh, T, 91)
    w = inputs.conv_weights(sh, 91)
    st = inputs.random_state(sh, 1, seed=92)
    pool = gdn.StatePool(sh, 12, fill=0xFF)
    pool.state(9).copy_(st["S"][0].cuda())
    pool.window(9).copy_(st["win"][0].cuda())
    bt = [[3, 4, -1, -1], [-1] * 4, [-1, -1, 5, -1]]        # boundaries 128, 256 | - | 384
    o = torch.full((T, sh.num_v_heads, sh.head_dim_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_core_prefill(sh, pool, cu_seqlens=dev(cu, torch.int32), start_pos=dev(start, torch.int64),
                         init_page=dev(init, torch.int32), block_table=dev(bt, torch.int32),
                         out_slot=dev([0, 1, 2], torch.int32), qkvz=dev(qkvz), ba=dev(ba), conv_w=dev(w),
                         A_log=dev(A_log), dt_bias=dev(dt_bias), norm_w=dev(norm_w), norm_eps=NORM_EPS, o=o,
                         dev_error=err, start_pos_host=start, init_page_host=init, max_seq_len=max(lens), path=path)
    torch.cuda.synchronize()
    assert err.item() == 0
    S0 = np.zeros((3, sh.num_v_heads, sh.head_dim_v, sh.head_dim_k))
    W0 = np.zeros((3, 3, sh.conv_dim))
    S0[2] = st["S"][0].double().numpy()
    W0[2] = st["win"][0].float().numpy()
    ref = oracle.core_prefill(dims(sh), cu, start, 128, qkvz, ba, w, A_log, dt_bias, norm_w, NORM_EPS, S0, W0)
    assert_out_close(o.cpu(), ref["y"], cu)
    assert_state_close(torch.stack([pool.state(s) for s in range(3)]).cpu(), ref["S"])
    assert_state_close(torch.stack([pool.state(p) for p in (3, 4, 5)]).cpu(), ref["ck_S"])
    for i, p in enumerate((3, 4, 5)):
        assert torch.equal(pool.window(p).cpu().float(), torch.as_tensor(ref["ck_win"][i], dtype=torch.float32))
    for s in range(3):
        assert torch.equal(pool.window(s).cpu().float(), torch.as_tensor(ref["win"][s], dtype=torch.float32))


@pytest.mark.parametrize("shape", [inputs.LayerShape(2, 6, 128, 128, 64, 16), inputs.QWEN4B,
                                   inputs.LayerShape(2, 4, 64, 64, 64, 16)])
def test_core_decode_matches_oracle(shape):
    sh = shape
    N = 7
    qkvz, ba, A_log, dt_bias, norm_w = _core_inputs(sh, N, 93)
    w = inputs.conv_weights(sh, 93)
    st = inputs.random_state(sh, N, seed=94)
    pool = gdn.StatePool(sh, N, fill=0)
    for p in range(N):
        pool.state(p).copy_(st["S"][p].cuda())
        pool.window(p).copy_(st["win"][p].cuda())
    o = torch.full((N, sh.num_v_heads, sh.head_dim_v), float("nan"), dtype=sh.torch_out(), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_core_decode(sh, pool, qkvz=dev(qkvz), ba=dev(ba), conv_w=dev(w), A_log=dev(A_log),
                        dt_bias=dev(dt_bias), norm_w=dev(norm_w), norm_eps=NORM_EPS,
                        slot=dev(list(range(N)), torch.int32), o=o, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    y_ref, S_ref, win_ref = oracle.core_decode(dims(sh), qkvz, ba, w, A_log, dt_bias, norm_w, NORM_EPS,
                                               st["S"].double().numpy(), st["win"].float().numpy())
    assert_out_close(o.cpu(), y_ref, list(range(N + 1)))
    assert_state_close(torch.stack([pool.state(p) for p in range(N)]).cpu(), S_ref)
    for p in range(N):
        assert torch.equal(pool.window(p).cpu().float(), torch.as_tensor(win_ref[p], dtype=torch.float32))


def _core_call(sh, pool, cu, start, init, bt, slots, qkvz, ba, w, A_log, dt_bias, norm_w, path, workspace=None):
    T = int(cu[-1])
    o = torch.full((T, sh.num_v_heads, sh.head_dim_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = gdn.gdn_core_prefill(sh, pool, cu_seqlens=dev(cu, torch.int32), start_pos=dev(start, torch.int64),
                              init_page=dev(init, torch.int32), block_table=dev(bt, torch.int32),
                              out_slot=dev(slots, torch.int32), qkvz=dev(qkvz), ba=dev(ba), conv_w=dev(w),
                              A_log=dev(A_log), dt_bias=dev(dt_bias), norm_w=dev(norm_w), norm_eps=NORM_EPS, o=o,
                              dev_error=err, start_pos_host=start, init_page_host=init, workspace=workspace,
                              max_seq_len=int(np.max(np.diff(cu))), path=path, raise_on_error=False)
    torch.cuda.synchronize()
    return st, int(err.item()), o.cpu()


@pytest.mark.parametrize("case", ["gqa3_resumed", "overlap_27b", "overlap_27b_resumed"])
def test_core_prefill_two_kernels_give_the_fused_kernels_bits(case):
    """The packed core on the chunk + chain kernels gives the fused kernel's
    bits: outputs, states, checkpoints and windows.  gqa3_resumed runs the
    chain's gated-norm epilogue; the overlap cases run the overlapped levels,
    whose chains leave fp32 outputs for the separate gated-norm pass (cold,
    and resumed from a block boundary with a carried state and window)."""
    if case == "gqa3_resumed":
        sh = inputs.LayerShape(2, 6, 128, 128, block_size=128, chunk_size=64)
        lens, start, init = [300, 65, 200], [0, 0, 256], [-1, -1, 9]
        bt, slots, npages = [[3, 4, -1, -1], [-1] * 4, [-1, -1, 5, -1]], [0, 1, 2], 12
    else:
        sh = inputs.QWEN27B
        if case == "overlap_27b":
            lens, start, init = [4133], [0], [-1]
            bt, slots, npages = [[1, 2, 3, 4]], [0], 5
        else:   # tokens 1,792 .. 5,925: boundaries 2,688 .. 5,376 in blocks 2 .. 5
            lens, start, init = [4133], [2 * 896], [9]
            bt, slots, npages = [[-1, -1, 1, 2, 3, 4, -1]], [0], 10
        plan = gdn.gdn_prefill_plan_for(sh, 1, 4133, 0, gdn.PREFILL_TWO_KERNELS)
        if plan["chunk_launches"] < 2:
            pytest.skip(f"this GPU runs the two kernels one after the other: {plan}")
    cu = np.concatenate([[0], np.cumsum(lens)])
    qkvz, ba, A_log, dt_bias, norm_w = _core_inputs(sh, int(cu[-1]), 94)
    w = inputs.conv_weights(sh, 94)
    st = inputs.random_state(sh, 1, seed=95)
    res = []
    for path in (gdn.PREFILL_FUSED, gdn.PREFILL_TWO_KERNELS):
        pool = gdn.StatePool(sh, npages, fill=0x3C)
        if 9 < npages:
            pool.state(9).copy_(st["S"][0].cuda())
            pool.window(9).copy_(st["win"][0].cuda())
        status, err, o = _core_call(sh, pool, cu, start, init, bt, slots, qkvz, ba, w, A_log, dt_bias, norm_w, path)
        assert status == 0 and err == 0
        res.append((o, pool.buf.cpu()))
    (o_f, p_f), (o_2, p_2) = res
    assert torch.equal(o_f.view(torch.int16), o_2.view(torch.int16))
    assert torch.equal(p_f, p_2)


def test_core_prefill_workspace_of_the_gates_alone_keeps_the_fused_kernel():
    """A workspace of the gates alone: AUTO runs the fused kernel (the same
    bits as with the full workspace), the two kernels are refused."""
    sh = inputs.LayerShape(2, 6, 128, 128, block_size=128, chunk_size=64)
    lens = [700, 300]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    qkvz, ba, A_log, dt_bias, norm_w = _core_inputs(sh, T, 96)
    w = inputs.conv_weights(sh, 96)
    gates_only = gdn.workspace_for(-(-(2 * 4 * T * sh.num_v_heads) // 256) * 256)
    args = (cu, [0, 0], [-1, -1], [[2, 3, 4, 5, 6], [7, 8, -1, -1, -1]], [0, 1], qkvz, ba, w, A_log, dt_bias, norm_w)
    outs = []
    for path, ws in ((gdn.PREFILL_AUTO, gates_only), (gdn.PREFILL_AUTO, None)):
        pool = gdn.StatePool(sh, 9, fill=0)
        status, err, o = _core_call(sh, pool, *args, path=path, workspace=ws)
        assert status == 0 and err == 0
        outs.append((o, pool.buf.cpu()))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1], outs[1][1])
    pool = gdn.StatePool(sh, 9, fill=0)
    status, _, _ = _core_call(sh, pool, *args, path=gdn.PREFILL_TWO_KERNELS, workspace=gates_only)
    assert status == gdn.STATUS_CODE["GDN_ERR_WORKSPACE"]
