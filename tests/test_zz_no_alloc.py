"""gdn_prefill_chunked_noalloc against gdn_prefill_chunked.

The allocation-free prefill serves callers that cannot hand the library any
device memory for scratch (a runtime whose free GPU memory is all reserved for
its pools, or a C caller without an allocator).  It keeps its scratch in a
fixed 64 MiB device array of the library instead.  This file runs last so
that a failure here leaves every other test already run; it also passes alone
in a fresh process, because the first call does the per-device set-up.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_state_gb300 as gdn
from gated_deltanet_state_gb300 import inputs

from harness import assert_out_close, assert_state_close, dev

pytestmark = pytest.mark.gpu

SHAPE = inputs.with_(inputs.QWEN27B, block_size=128, chunk_size=64)
LENS = [300, 500]


def _args(seed):
    cu = np.concatenate([[0], np.cumsum(LENS)])
    ti = inputs.token_inputs(SHAPE, int(cu[-1]), seed)
    bt = [[2 + 4 * s + j if j < LENS[s] // 128 else -1 for j in range(4)] for s in range(len(LENS))]
    return dict(cu_seqlens=dev(cu, torch.int32), start_pos=dev([0, 0], torch.int64),
                init_page=dev([-1, -1], torch.int32), block_table=dev(bt, torch.int32),
                out_slot=dev([0, 1], torch.int32), x=dev(ti["x"]), g=dev(ti["g"]), beta=dev(ti["beta"]),
                conv_w=dev(inputs.conv_weights(SHAPE, seed)), start_pos_host=[0, 0], init_page_host=[-1, -1])


def _run(fn, seed, **extra):
    a = _args(seed)
    pool = gdn.StatePool(SHAPE, 12, fill=0)
    o = torch.empty(sum(LENS), SHAPE.num_v_heads, SHAPE.head_dim_v, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn(SHAPE, pool, o=o, dev_error=err, **a, **extra)
    torch.cuda.synchronize()
    assert err.item() == 0
    states = torch.stack([pool.state(p) for p in range(12)]).cpu()
    return o.cpu(), states, pool.buf.cpu()


def test_noalloc_prefill_matches_the_workspace_prefill_on_two_calls_in_a_row():
    assert gdn.gdn_prefill_workspace_size(SHAPE, len(LENS), sum(LENS)) <= gdn.NOALLOC_SCRATCH_BYTES
    cu = np.concatenate([[0], np.cumsum(LENS)])
    for seed in (41, 42):   # the second call reuses the scratch the first one left
        o_ref, s_ref, _ = _run(gdn.gdn_prefill_chunked, seed)
        o_na, s_na, _ = _run(gdn.gdn_prefill_chunked_noalloc, seed)
        assert_out_close(o_na, o_ref.double().numpy(), cu)
        used = [0, 1] + [p for p in range(2, 12) if s_ref[p].abs().sum() > 0]
        assert_state_close(s_na[used], s_ref[used].double().numpy())


def test_noalloc_prefill_rejects_calls_beyond_its_scratch():
    T = 2000   # 27B-shaped rows need ~41 KB of scratch each: more than 64 MiB
    assert gdn.gdn_prefill_workspace_size(SHAPE, 1, T) > gdn.NOALLOC_SCRATCH_BYTES
    ti = inputs.token_inputs(SHAPE, T, 1)
    pool = gdn.StatePool(SHAPE, 2, fill=0)
    o = torch.empty(T, SHAPE.num_v_heads, SHAPE.head_dim_v, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_prefill_chunked_noalloc(
            SHAPE, pool, cu_seqlens=dev([0, T], torch.int32), start_pos=dev([0], torch.int64),
            init_page=dev([-1], torch.int32), block_table=dev([[-1] * 16], torch.int32),
            out_slot=dev([0], torch.int32), x=dev(ti["x"]), g=dev(ti["g"]), beta=dev(ti["beta"]),
            conv_w=dev(inputs.conv_weights(SHAPE, 1)), o=o, dev_error=err)
    assert ei.value.status == gdn.STATUS_CODE["GDN_ERR_WORKSPACE"]
