"""Mixed batches: prefill sequences and single decode tokens packed in one
varlen batch ("Hybrid linear attention (gated DeltaNet)", "The part that is
easy to get wrong": the mixed regime runs the prefill kernels and
gdn_decode_mixed together).  Every sequence must get exactly the bits of the
corresponding separate prefill or decode call, and match the oracle."""
import numpy as np
import pytest
import torch

import oracle
import gated_deltanet_state_gb300 as gdn
from gated_deltanet_state_gb300 import inputs

from harness import assert_out_close, assert_state_close, dev, dims

pytestmark = pytest.mark.gpu

# regimes: prefill 300 cold, decode, prefill 130 resumed at 128, decode, decode
LENS = [300, 1, 130, 1, 1]
DECODE = [0, 1, 0, 1, 1]
START = [0, 0, 128, 0, 0]


@pytest.mark.parametrize("shape", [inputs.LayerShape(2, 6, 128, 128, 64, 64),    # tensor-core prefill
                                   inputs.LayerShape(2, 4, 64, 64, 64, 16)],     # scan prefill
                         ids=["tc", "scan"])
def test_mixed_batch_equals_separate_calls_and_oracle(shape):
    sh = shape
    N = len(LENS)
    cu = np.concatenate([[0], np.cumsum(LENS)]).astype(np.int64)
    T = int(cu[-1])
    ti = inputs.token_inputs(sh, T, seed=71)
    w = inputs.conv_weights(sh, 71)
    st = inputs.random_state(sh, 4, seed=72)
    # pages: slots 0..4 (one per sequence), 5 = resume page of sequence 2, 6..11 checkpoints
    slot = [0, 1, 2, 3, 4]
    init = [-1, -1, 5, -1, -1]
    bt = [[6, 7, 8, 9], [-1] * 4, [-1, -1, 10, 11], [-1] * 4, [-1] * 4]

    def fresh_pool():
        pool = gdn.StatePool(sh, 12, fill=0)
        for i, p in enumerate([1, 3, 4, 5]):        # decode slots and the resume page
            pool.state(p).copy_(st["S"][i].cuda())
            pool.window(p).copy_(st["win"][i].cuda())
        return pool

    # the mixed call
    pool_m = fresh_pool()
    o_m = torch.zeros(T, sh.num_v_heads, sh.head_dim_v, dtype=sh.torch_out(), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_mixed_step(sh, pool_m, cu_seqlens=dev(cu, torch.int32), is_decode=dev(DECODE, torch.int8),
                       start_pos=dev(START, torch.int64), init_page=dev(init, torch.int32),
                       block_table=dev(bt, torch.int32), slot=dev(slot, torch.int32), x=dev(ti["x"]),
                       g=dev(ti["g"]), beta=dev(ti["beta"]), conv_w=dev(w), o=o_m, dev_error=err,
                       start_pos_host=START, init_page_host=init)
    torch.cuda.synchronize()
    assert err.item() == 0

    # the same work as separate calls
    pool_s = fresh_pool()
    o_s = torch.zeros_like(o_m)
    pre = [s for s in range(N) if not DECODE[s]]
    dec = [s for s in range(N) if DECODE[s]]
    rows = torch.cat([torch.arange(int(cu[s]), int(cu[s + 1])) for s in pre])
    cu_p = np.concatenate([[0], np.cumsum([LENS[s] for s in pre])])
    o_p = torch.zeros(len(rows), sh.num_v_heads, sh.head_dim_v, dtype=sh.torch_out(), device="cuda")
    gdn.gdn_prefill_chunked(sh, pool_s, cu_seqlens=dev(cu_p, torch.int32),
                            start_pos=dev([START[s] for s in pre], torch.int64),
                            init_page=dev([init[s] for s in pre], torch.int32),
                            block_table=dev([bt[s] for s in pre], torch.int32),
                            out_slot=dev([slot[s] for s in pre], torch.int32), x=dev(ti["x"][rows]),
                            g=dev(ti["g"][rows]), beta=dev(ti["beta"][rows]), conv_w=dev(w), o=o_p,
                            dev_error=err, start_pos_host=[START[s] for s in pre],
                            init_page_host=[init[s] for s in pre])
    drows = torch.tensor([int(cu[s]) for s in dec])
    o_d = torch.zeros(len(dec), sh.num_v_heads, sh.head_dim_v, dtype=sh.torch_out(), device="cuda")
    gdn.gdn_decode_step(sh, pool_s, x=dev(ti["x"][drows]), g=dev(ti["g"][drows]), beta=dev(ti["beta"][drows]),
                        conv_w=dev(w), slot=dev([slot[s] for s in dec], torch.int32), o=o_d, dev_error=err)
    o_s[rows.cuda()] = o_p
    o_s[drows.cuda()] = o_d
    torch.cuda.synchronize()
    assert err.item() == 0
    bits = torch.int16 if o_m.element_size() == 2 else torch.int32
    assert torch.equal(o_m.view(bits), o_s.view(bits))
    assert torch.equal(pool_m.buf, pool_s.buf)

    # and the oracle: the decode tokens, and the resumed prefill
    o_ref, S_ref, win_ref = oracle.decode(dims(sh), ti["x"][drows], ti["g"][drows], ti["beta"][drows], w,
                                          st["S"][:3].double().numpy(), st["win"][:3].float().numpy())
    assert_out_close(o_m[drows.cuda()].cpu(), o_ref, list(range(len(dec) + 1)))
    assert_state_close(torch.stack([pool_m.state(slot[s]) for s in dec]).cpu(), S_ref)
    a, b = int(cu[2]), int(cu[3])
    ref = oracle.prefill(dims(sh), [0, b - a], [128], 64, ti["x"][a:b], ti["g"][a:b], ti["beta"][a:b], w,
                         st["S"][3:4].double().numpy(), st["win"][3:4].float().numpy())
    assert_out_close(o_m[a:b].cpu(), ref["o"], [0, b - a])
    assert_state_close(pool_m.state(2).cpu()[None], ref["S"])


def test_mixed_batch_of_decode_tokens_only_equals_decode_step():
    sh = inputs.LayerShape(2, 4, 128, 128, 64, 64)
    N = 6
    st = inputs.random_state(sh, N, seed=81)
    ti = inputs.token_inputs(sh, N, seed=82)
    w = inputs.conv_weights(sh, 82)
    pools = []
    for _ in range(2):
        pool = gdn.StatePool(sh, N, fill=0)
        for p in range(N):
            pool.state(p).copy_(st["S"][p].cuda())
            pool.window(p).copy_(st["win"][p].cuda())
        pools.append(pool)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o1 = torch.zeros(N, sh.num_v_heads, sh.head_dim_v, dtype=torch.bfloat16, device="cuda")
    o2 = torch.zeros_like(o1)
    gdn.gdn_mixed_step(sh, pools[0], cu_seqlens=dev(list(range(N + 1)), torch.int32),
                       is_decode=dev([1] * N, torch.int8), start_pos=dev([0] * N, torch.int64),
                       init_page=dev([-1] * N, torch.int32), block_table=None,
                       slot=dev(list(range(N)), torch.int32), x=dev(ti["x"]), g=dev(ti["g"]),
                       beta=dev(ti["beta"]), conv_w=dev(w), o=o1, dev_error=err)
    gdn.gdn_decode_step(sh, pools[1], x=dev(ti["x"]), g=dev(ti["g"]), beta=dev(ti["beta"]), conv_w=dev(w),
                        slot=dev(list(range(N)), torch.int32), o=o2, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(pools[0].buf, pools[1].buf)
