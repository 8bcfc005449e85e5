"""gdn_prefill_chunked_noalloc against gdn_prefill_chunked.

The allocation-free prefill serves callers that cannot hand the library any
device memory for scratch (a runtime whose free GPU memory is all reserved for
its pools, or a C caller without an allocator).  It keeps its scratch in a
fixed 64 MiB device array of the library instead.  Layers on the tensor-core
path take the fused kernel, which needs no scratch at all (the same kernel as
gdn_prefill_chunked without a workspace); layers on the conv pre-pass path
(here d = 64) use the array and are limited by it.  This file runs last so
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

SHAPE = inputs.with_(inputs.QWEN27B, block_size=128, chunk_size=64)              # tensor-core path
SHAPE_SCAN = inputs.with_(SHAPE, head_dim_k=64, head_dim_v=64)                     # conv pre-pass path
LENS = [300, 500]


def _args(shape, lens, seed):
    cu = np.concatenate([[0], np.cumsum(lens)])
    ti = inputs.token_inputs(shape, int(cu[-1]), seed)
    nb = max(lens) // 128
    bt = [[2 + nb * s + j if j < lens[s] // 128 else -1 for j in range(nb)] for s in range(len(lens))]
    n = len(lens)
    return dict(cu_seqlens=dev(cu, torch.int32), start_pos=dev([0] * n, torch.int64),
                init_page=dev([-1] * n, torch.int32), block_table=dev(bt, torch.int32),
                out_slot=dev(list(range(n)), torch.int32), x=dev(ti["x"]), g=dev(ti["g"]),
                beta=dev(ti["beta"]), conv_w=dev(inputs.conv_weights(shape, seed)),
                start_pos_host=[0] * n, init_page_host=[-1] * n), 2 + nb * n


def _run(fn, shape, lens, seed, **extra):
    a, pages = _args(shape, lens, seed)
    pool = gdn.StatePool(shape, pages, fill=0)
    o = torch.empty(sum(lens), shape.num_v_heads, shape.head_dim_v, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn(shape, pool, o=o, dev_error=err, **a, **extra)
    torch.cuda.synchronize()
    assert err.item() == 0
    states = torch.stack([pool.state(p) for p in range(pages)]).cpu()
    return o.cpu(), states


@pytest.mark.parametrize("shape", [SHAPE, SHAPE_SCAN], ids=["tensor_core_path", "pre_pass_path"])
def test_noalloc_prefill_matches_the_workspace_prefill_on_two_calls_in_a_row(shape):
    tc = shape is SHAPE
    assert tc or gdn.gdn_prefill_workspace_size(shape, len(LENS), sum(LENS)) <= gdn.NOALLOC_SCRATCH_BYTES
    # the tensor-core layer's allocation-free call is the fused kernel, as is
    # gdn_prefill_chunked without a workspace
    extra = {"workspace": False} if tc else {}
    for seed in (41, 42):   # the second call reuses the scratch the first one left
        o_ref, s_ref = _run(gdn.gdn_prefill_chunked, shape, LENS, seed, **extra)
        o_na, s_na = _run(gdn.gdn_prefill_chunked_noalloc, shape, LENS, seed)
        # the same kernels on the same inputs: the same bits
        assert torch.equal(o_na.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(s_na.view(torch.int32), s_ref.view(torch.int32))


def test_noalloc_prefill_has_no_limit_on_the_tensor_core_path():
    """8,192 tokens of the 27B-shaped layer: the fused kernel needs no scratch,
    so the allocation-free call runs whatever its length (a workspace prefill
    of this call would need more than the array holds): the bits of
    gdn_prefill_chunked without a workspace, and the two-kernel path's
    results within the parity bounds."""
    T = 8192
    assert gdn.gdn_prefill_workspace_size(SHAPE, 1, T) > gdn.NOALLOC_SCRATCH_BYTES
    o_ref, s_ref = _run(gdn.gdn_prefill_chunked, SHAPE, [T], 43, workspace=False)
    o_na, s_na = _run(gdn.gdn_prefill_chunked_noalloc, SHAPE, [T], 43)
    assert torch.equal(o_na.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(s_na.view(torch.int32), s_ref.view(torch.int32))
    o_2k, s_2k = _run(gdn.gdn_prefill_chunked, SHAPE, [T], 43)
    assert_out_close(o_na, o_2k.double().numpy(), [0, T])
    used = [0] + [p for p in range(2, s_2k.shape[0]) if s_2k[p].abs().sum() > 0]
    assert_state_close(s_na[used], s_2k[used].double().numpy())


def test_noalloc_prefill_rejects_calls_beyond_its_scratch():
    SHAPE = SHAPE_SCAN
    T = 4000   # these rows need ~21 KB of scratch each: more than 64 MiB
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
