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


def test_core_prefill_matches_oracle_cold_and_resumed():
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
                         dev_error=err, start_pos_host=start, init_page_host=init)
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
