"""The tensor-core chunk prefill (d = 128, bf16, block size a multiple of 64)
against the fp64 oracle: lengths around the 64-row chunk edges, GQA groups of
three, resumes from arbitrary states, strong decays, and the special cases
that reduce to exact identities."""
import numpy as np
import pytest
import torch

import oracle
import gated_deltanet_state_gb300 as gdn
from gated_deltanet_state_gb300 import inputs

from harness import assert_out_close, assert_state_close, dims, oracle_head, run_prefill

pytestmark = pytest.mark.gpu


def _tables(lens, B, first_page):
    nb = max(1, max(lens) // B)
    bt = np.full((len(lens), nb), -1)
    page = first_page
    for s, L in enumerate(lens):
        for jb in range(L // B):
            bt[s, jb] = page
            page += 1
    return bt, page


def _last_rows(x, a, b):
    """The window a cold sequence x[a:b] leaves: its last three pre-conv rows,
    zeros in front when it is shorter."""
    rows = x[max(a, b - 3):b]
    return torch.cat([rows.new_zeros(3 - rows.shape[0], x.shape[1]), rows])


def test_chunk_edges_gqa3_match_oracle():
    sh = inputs.LayerShape(2, 6, 128, 128, block_size=128, chunk_size=64)
    lens = [1, 63, 64, 65, 127, 128, 129, 300, 700]
    cu = np.concatenate([[0], np.cumsum(lens)])
    N = len(lens)
    ti = inputs.token_inputs(sh, int(cu[-1]), seed=21)
    w = inputs.conv_weights(sh, 21)
    bt, npages = _tables(lens, 128, N)
    pool = gdn.StatePool(sh, npages, fill=0xFF)
    o, err, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, cu, [0] * N, [-1] * N, bt, list(range(N)))
    assert err == 0
    ref = oracle.prefill(dims(sh), cu, [0] * N, 128, ti["x"], ti["g"], ti["beta"], w)
    assert_out_close(o, ref["o"], cu)
    assert_state_close(torch.stack([pool.state(s) for s in range(N)]).cpu(), ref["S"])
    k = 0
    for s, L in enumerate(lens):
        for jb in range(L // 128):
            p = int(bt[s, jb])
            assert_state_close(pool.state(p).cpu()[None], ref["ck_S"][k][None])
            assert torch.equal(pool.window(p).cpu().float(), torch.as_tensor(ref["ck_win"][k], dtype=torch.float32))
            k += 1
    for s in range(N):
        assert torch.equal(pool.window(s).cpu(), _last_rows(ti["x"], int(cu[s]), int(cu[s + 1])))


def test_resume_in_place_strong_decay_and_q_scale_match_oracle():
    sh = inputs.LayerShape(1, 2, 128, 128, block_size=192, chunk_size=64, q_scale=0.5)
    st = inputs.random_state(sh, 1, seed=31)
    T = 450
    ti = inputs.token_inputs(sh, T, seed=32)
    # a stretch of very strong decays (a = e^-30): the chunk's running decay
    # underflows toward zero inside one chunk
    ti["g"][100:140] = -30.0
    w = inputs.conv_weights(sh, 32)
    pool = gdn.StatePool(sh, 4, fill=0)
    pool.state(1).copy_(st["S"][0].cuda())
    pool.window(1).copy_(st["win"][0].cuda())
    # resume at 384 (two blocks); boundaries at 576 and 768 fall at rows 192, 384
    o, err, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, [0, T], [384], [1], [[-1, -1, 2, 3]], [1])
    assert err == 0
    ref = oracle.prefill(dims(sh), [0, T], [384], 192, ti["x"], ti["g"], ti["beta"], w,
                         st["S"].double().numpy(), st["win"].float().numpy())
    assert_out_close(o, ref["o"], [0, T])
    assert_state_close(pool.state(1).cpu()[None], ref["S"])
    assert_state_close(pool.state(2).cpu()[None], ref["ck_S"][0][None])
    assert_state_close(pool.state(3).cpu()[None], ref["ck_S"][1][None])


def test_no_write_no_decay_keeps_the_state_bitwise():
    """b = 0 and g = 0 (a = 1): every chunk adds exact zeros to gam_C S0 = S0,
    so the state comes back with the same bits, and the outputs are S0 q^."""
    sh = inputs.LayerShape(1, 2, 128, 128, block_size=128, chunk_size=64)
    st = inputs.random_state(sh, 1, seed=41)
    T = 200
    ti = inputs.token_inputs(sh, T, seed=42)
    ti["g"].zero_()
    ti["beta"].zero_()
    w = inputs.conv_weights(sh, 42)
    pool = gdn.StatePool(sh, 3, fill=0)
    pool.state(1).copy_(st["S"][0].cuda())
    pool.window(1).copy_(st["win"][0].cuda())
    o, err, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, [0, T], [128], [1], [[-1, 2, -1]], [0])
    assert err == 0
    assert torch.equal(pool.state(0).cpu().view(torch.int32), st["S"][0].view(torch.int32))
    assert torch.equal(pool.state(2).cpu().view(torch.int32), st["S"][0].view(torch.int32))
    ref = oracle.prefill(dims(sh), [0, T], [128], 128, ti["x"], ti["g"], ti["beta"], w,
                         st["S"].double().numpy(), st["win"].float().numpy())
    assert_out_close(o, ref["o"], [0, T])


def test_cold_equals_resume_bitwise_at_64_multiple_blocks():
    sh = inputs.LayerShape(2, 4, 128, 128, block_size=320, chunk_size=64)
    T = 1000
    ti = inputs.token_inputs(sh, T, seed=51)
    w = inputs.conv_weights(sh, 51)
    pool = gdn.StatePool(sh, 10, fill=0)
    o_cold, err, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, [0, T], [0], [-1], [[1, 2, 3]], [0])
    assert err == 0
    P = 320
    o_res, err, _ = run_prefill(sh, pool, ti["x"][P:], ti["g"][P:], ti["beta"][P:], w, [0, T - P], [P], [1],
                                [[-1, 5, 6]], [4])
    assert err == 0
    assert torch.equal(o_res.view(torch.int16), o_cold[P:].view(torch.int16))
    assert torch.equal(pool.payload(4).cpu(), pool.payload(0).cpu())
    assert torch.equal(pool.payload(5).cpu(), pool.payload(2).cpu())
    assert torch.equal(pool.payload(6).cpu(), pool.payload(3).cpu())


def test_pieces_over_several_launches_equal_one_launch_bitwise():
    """Four sequences of the 27B-shaped layer are 192 (sequence, v head)
    chains, more than the GPU has SMs, so the prefill cuts them into pieces run
    over several launches (a piece starts from the state the one before it
    left in the final slot).  One sequence alone is 48 chains, one launch.
    Outputs, final states, checkpoints and windows must be the same bits, with
    block boundaries at piece ends, a resumed sequence, a sequence that ends
    inside its second piece and one shorter than a piece.  (The single
    sequences take the fused kernel: the two kernels would cut even one
    sequence into overlapped levels.)"""
    sh = inputs.LayerShape(16, 48, 128, 128, block_size=1024, chunk_size=64, page_bytes=inputs.QWEN27B.page)
    lens = [2048, 1800, 77, 1536]
    start = [0, 0, 0, 1024]
    init = [-1, -1, -1, 4]
    bt = [[5, 6], [7, -1], [-1, -1], [-1, 8]]
    N = len(lens)
    plan = gdn.gdn_prefill_plan_for(sh, N, max(lens))
    assert plan["levels"] == 2 and plan["launches"] > 1, plan
    assert gdn.gdn_prefill_plan_for(sh, 1, max(lens), 0, gdn.PREFILL_FUSED)["launches"] == 1
    cu = np.concatenate([[0], np.cumsum(lens)])
    ti = inputs.token_inputs(sh, int(cu[-1]), seed=61)
    w = inputs.conv_weights(sh, 61)
    st = inputs.random_state(sh, 1, seed=62)
    pools = []
    for _ in range(2):
        pool = gdn.StatePool(sh, 9, fill=0)
        pool.state(4).copy_(st["S"][0].cuda())
        pool.window(4).copy_(st["win"][0].cuda())
        pools.append(pool)
    o_all, err, _ = run_prefill(sh, pools[0], ti["x"], ti["g"], ti["beta"], w, cu, start, init, bt,
                                list(range(N)), max_seq_len=max(lens))
    assert err == 0
    for s in range(N):
        a, b = int(cu[s]), int(cu[s + 1])
        o_one, err, _ = run_prefill(sh, pools[1], ti["x"][a:b], ti["g"][a:b], ti["beta"][a:b], w, [0, b - a],
                                    [start[s]], [init[s]], [bt[s]], [s], max_seq_len=b - a, workspace=False,
                                    path=gdn.PREFILL_FUSED)
        assert err == 0
        assert torch.equal(o_all[a:b].view(torch.int16), o_one.view(torch.int16)), s
    for page in [0, 1, 2, 3, 5, 6, 7, 8]:
        assert torch.equal(pools[0].payload(page).cpu(), pools[1].payload(page).cpu()), page
    # a bad page for a boundary inside a later piece (sequence 0's block 1,
    # reached in its second piece) is reported like one in the first
    bad = [list(r) for r in bt]
    bad[0][1] = 99
    pool = gdn.StatePool(sh, 9, fill=0)
    pool.state(4).copy_(st["S"][0].cuda())
    _, err, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, cu, start, init, bad, list(range(N)),
                            max_seq_len=max(lens))
    assert err == gdn.STATUS_CODE["GDN_ERR_PAGE_RANGE"]
    # and against the oracle on two heads of the resumed sequence
    a, b = int(cu[3]), int(cu[4])
    for h in (0, 47):
        ref = oracle_head(sh, ti["x"][a:b], ti["g"][a:b], ti["beta"][a:b], w, h, [0, b - a], [1024], 1024,
                          st["S"].double().numpy(), st["win"].float().numpy())
        assert_out_close(o_all[a:b, h:h + 1], ref["o"], [0, b - a])
        assert_state_close(pools[0].state(3).cpu()[None, h:h + 1], ref["S"])


def _both_paths(sh, lens, start, init, bt, seed, npages, fill_state=None, max_seq_len=0):
    """The same call through the fused kernel (no workspace) and the chunk +
    chain kernels (with one): outputs, pool pages and error words."""
    cu = np.concatenate([[0], np.cumsum(lens)])
    ti = inputs.token_inputs(sh, int(cu[-1]), seed=seed)
    w = inputs.conv_weights(sh, seed)
    res = []
    for ws, path in ((False, gdn.PREFILL_FUSED), (None, gdn.PREFILL_TWO_KERNELS)):
        pool = gdn.StatePool(sh, npages, fill=0x3C)
        if fill_state is not None:
            page, st = fill_state
            pool.state(page).copy_(st["S"][0].cuda())
            pool.window(page).copy_(st["win"][0].cuda())
        o, err, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, cu, start, init, bt,
                                list(range(len(lens))), max_seq_len=max_seq_len, workspace=ws, path=path)
        assert err == 0
        res.append((o, pool.buf.cpu()))
    return res


@pytest.mark.parametrize("case", ["edges_gqa3", "resumed_27b", "pieces_27b", "overlap_27b", "overlap_27b_resumed"])
def test_two_kernel_path_gives_the_fused_kernels_bits(case):
    """The chunk + chain kernels split and multiply every operand as the fused
    kernel does, so a call gives the same bits on either path: a prefix hit
    reproduces a cold run's bits whichever path each call takes.  The overlap
    cases run the two kernels' overlapped levels (the chain on a second
    stream, four checkpoints inside levels), cold and resumed."""
    if case == "edges_gqa3":
        sh = inputs.LayerShape(2, 6, 128, 128, block_size=128, chunk_size=64)
        lens = [1, 63, 64, 65, 127, 128, 129, 300, 700]
        bt, npages = _tables(lens, 128, len(lens))
        res = _both_paths(sh, lens, [0] * len(lens), [-1] * len(lens), bt, 81, npages)
    elif case == "resumed_27b":
        sh = inputs.with_(inputs.QWEN27B, block_size=256)
        st = inputs.random_state(sh, 1, seed=83)
        res = _both_paths(sh, [700, 300], [512, 0], [5, -1], [[-1, -1, 6, 7], [8, -1, -1, -1]], 82, 9,
                          fill_state=(5, st))
    elif case == "overlap_27b":
        sh = inputs.QWEN27B
        lens = [4133]
        plan = gdn.gdn_prefill_plan_for(sh, 1, max(lens), 0, gdn.PREFILL_TWO_KERNELS)
        if plan["chunk_launches"] < 2:
            pytest.skip(f"this GPU runs the two kernels one after the other: {plan}")
        res = _both_paths(sh, lens, [0], [-1], [[1, 2, 3, 4]], 85, 5, max_seq_len=max(lens))
    elif case == "overlap_27b_resumed":
        # tokens 1,792 .. 5,925 from a carried state and window in page 9
        sh = inputs.QWEN27B
        lens = [4133]
        plan = gdn.gdn_prefill_plan_for(sh, 1, max(lens), 0, gdn.PREFILL_TWO_KERNELS)
        if plan["chunk_launches"] < 2:
            pytest.skip(f"this GPU runs the two kernels one after the other: {plan}")
        st = inputs.random_state(sh, 1, seed=86)
        res = _both_paths(sh, lens, [2 * 896], [9], [[-1, -1, 1, 2, 3, 4, -1]], 86, 10, fill_state=(9, st),
                          max_seq_len=max(lens))
    else:
        sh = inputs.LayerShape(16, 48, 128, 128, block_size=1024, chunk_size=64, page_bytes=inputs.QWEN27B.page)
        lens = [2048, 1800, 77, 1536]
        assert gdn.gdn_prefill_plan_for(sh, len(lens), max(lens))["levels"] == 2
        res = _both_paths(sh, lens, [0] * 4, [-1] * 4, [[5, 6], [7, -1], [-1, -1], [8, -1]], 84, 9,
                          max_seq_len=max(lens))
    (o_f, pool_f), (o_2, pool_2) = res
    assert torch.equal(o_f.view(torch.int16), o_2.view(torch.int16))
    assert torch.equal(pool_f, pool_2)


@pytest.mark.parametrize("case", ["serial", "overlap", "one_per_group"])
def test_six_value_heads_a_group_two_kernels(case):
    """Six value heads to a qk head: the chunk kernel forms the gates of its
    first four heads during the conv and the later ones inside the head loop
    (both modes: v convolved in the chain, serial here; v's image, overlapped
    levels); and one value head to a qk head (no next head to prepare).  The
    two kernels give the fused kernel's bits, and the serial cases match the
    oracle."""
    if case in ("serial", "one_per_group"):
        sh = inputs.LayerShape(1, 6, 128, 128, block_size=128, chunk_size=64) if case == "serial" else \
            inputs.LayerShape(2, 2, 128, 128, block_size=128, chunk_size=64)
        lens = [700, 129, 1, 300]
        plan = gdn.gdn_prefill_plan_for(sh, len(lens), max(lens), 0, gdn.PREFILL_TWO_KERNELS)
        assert plan["chunk_launches"] == 1
        bt, npages = _tables(lens, 128, len(lens))
        res = _both_paths(sh, lens, [0] * len(lens), [-1] * len(lens), bt, 87, npages)
        cu = np.concatenate([[0], np.cumsum(lens)])
        ti = inputs.token_inputs(sh, int(cu[-1]), seed=87)
        ref = oracle.prefill(dims(sh), cu, [0] * len(lens), 128, ti["x"], ti["g"], ti["beta"],
                             inputs.conv_weights(sh, 87))
        assert_out_close(res[1][0], ref["o"], cu)
    else:
        sh = inputs.LayerShape(8, 48, 128, 128, block_size=1024, chunk_size=64, page_bytes=inputs.QWEN27B.page)
        lens = [4133]
        plan = gdn.gdn_prefill_plan_for(sh, 1, max(lens), 0, gdn.PREFILL_TWO_KERNELS)
        if plan["chunk_launches"] < 2:
            pytest.skip(f"this GPU runs the two kernels one after the other: {plan}")
        res = _both_paths(sh, lens, [0], [-1], [[1, 2, 3, 4]], 88, 5, max_seq_len=max(lens))
    (o_f, pool_f), (o_2, pool_2) = res
    assert torch.equal(o_f.view(torch.int16), o_2.view(torch.int16))
    assert torch.equal(pool_f, pool_2)


def test_overlapped_levels_resume_bitwise():
    """A long sequence on the two kernels' overlapped levels, then the same
    sequence resumed from its second checkpoint (a shorter call, its own
    levels): the resumed call reproduces the cold call's outputs, later
    checkpoints and final state bit for bit, and both match the oracle on
    two heads."""
    sh = inputs.QWEN27B
    T, B = 6000, sh.block_size
    nb = T // B                                   # 6 checkpoints
    P = 2 * B
    for L in (T, T - P):
        plan = gdn.gdn_prefill_plan_for(sh, 1, L, 0, gdn.PREFILL_TWO_KERNELS)
        if plan["chunk_launches"] < 2:
            pytest.skip(f"this GPU runs the two kernels one after the other: {plan}")
    ti = inputs.token_inputs(sh, T, seed=86)
    w = inputs.conv_weights(sh, 86)
    pool = gdn.StatePool(sh, 2 + 2 * nb, fill=0)
    kw = dict(workspace=None, path=gdn.PREFILL_TWO_KERNELS)
    cold_pages = list(range(1, nb + 1))
    o_cold, err, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, [0, T], [0], [-1], [cold_pages],
                                 [0], max_seq_len=T, **kw)
    assert err == 0
    res_pages = [-1, -1] + list(range(nb + 2, 2 * nb))
    o_res, err, _ = run_prefill(sh, pool, ti["x"][P:], ti["g"][P:], ti["beta"][P:], w, [0, T - P], [P], [2],
                                [res_pages], [nb + 1], max_seq_len=T - P, **kw)
    assert err == 0
    assert torch.equal(o_res.view(torch.int16), o_cold[P:].view(torch.int16))
    assert torch.equal(pool.payload(nb + 1).cpu(), pool.payload(0).cpu())
    for j in range(2, nb):
        assert torch.equal(pool.payload(res_pages[j]).cpu(), pool.payload(cold_pages[j]).cpu()), j
    for h in (0, 47):
        ref = oracle_head(sh, ti["x"], ti["g"], ti["beta"], w, h, [0, T], [0], B)
        assert_out_close(o_cold[:, h:h + 1], ref["o"], [0, T])
        assert_state_close(pool.state(0).cpu()[None, h:h + 1], ref["S"])
        for j, page in enumerate(cold_pages):
            assert_state_close(pool.state(page).cpu()[None, h:h + 1], ref["ck_S"][j][None])


def _paths_with_error(sh, lens, bt, seed, npages, max_seq_len=0, two_max_seq_len=None):
    """The same call on the fused kernel and on the two kernels, each into a
    fresh pool: (outputs, pool bytes, error word) per path."""
    cu = np.concatenate([[0], np.cumsum(lens)])
    ti = inputs.token_inputs(sh, int(cu[-1]), seed=seed)
    w = inputs.conv_weights(sh, seed)
    res = []
    for ws, path, L in ((False, gdn.PREFILL_FUSED, max_seq_len),
                        (None, gdn.PREFILL_TWO_KERNELS, max_seq_len if two_max_seq_len is None else two_max_seq_len)):
        pool = gdn.StatePool(sh, npages, fill=0x3C)
        o, err, _ = run_prefill(sh, pool, ti["x"], ti["g"], ti["beta"], w, cu, [0] * len(lens), [-1] * len(lens),
                                bt, list(range(len(lens))), max_seq_len=L, workspace=ws, path=path)
        res.append((o, pool.buf.cpu(), err))
    return cu, res


def test_two_kernel_path_empty_sequences():
    """Empty sequences among others: both paths give the same bits (the empty
    sequences' final slots included), and no error."""
    sh = inputs.LayerShape(2, 6, 128, 128, block_size=128, chunk_size=64)
    lens = [0, 300, 0, 129, 64, 0]
    bt, npages = _tables(lens, 128, len(lens))
    cu, ((o_f, pool_f, e_f), (o_2, pool_2, e_2)) = _paths_with_error(sh, lens, bt, 87, npages)
    assert e_f == 0 and e_2 == 0
    assert torch.equal(o_f.view(torch.int16), o_2.view(torch.int16))
    assert torch.equal(pool_f, pool_2)


def test_two_kernel_path_refuses_a_sequence_past_max_seq_len():
    """max_seq_len sizes the two kernels' grid: a longer sequence sets
    GDN_ERR_INVALID_ARG and gets no outputs; the sequences within the bound
    are unaffected (the fused kernel's bits)."""
    sh = inputs.LayerShape(2, 6, 128, 128, block_size=128, chunk_size=64)
    lens = [300, 700]
    bt, npages = _tables(lens, 128, len(lens))
    cu, ((o_f, pool_f, e_f), (o_2, pool_2, e_2)) = _paths_with_error(sh, lens, bt, 88, npages, max_seq_len=700,
                                                                      two_max_seq_len=300)
    assert e_f == 0
    assert e_2 == gdn.STATUS_CODE["GDN_ERR_INVALID_ARG"]
    assert torch.equal(o_f[:300].view(torch.int16), o_2[:300].view(torch.int16))
    assert torch.isnan(o_2[300:].float()).all()
    page = sh.page
    for p_ in [0] + [int(x) for x in bt[0] if x >= 0]:     # sequence 0's final slot and checkpoints
        assert torch.equal(pool_f[p_ * page:p_ * page + sh.state_bytes], pool_2[p_ * page:p_ * page + sh.state_bytes])
    for p_ in [1] + [int(x) for x in bt[1] if x >= 0]:     # sequence 1: no state written
        assert (pool_2[p_ * page:p_ * page + sh.state_bytes] == 0x3C).all()


def test_two_kernel_path_bad_page_in_a_later_level():
    """A checkpoint page outside the pool, reached in the second of the
    overlapped levels: GDN_ERR_PAGE_RANGE, as on the fused kernel, and the
    same bits everywhere else."""
    sh = inputs.QWEN27B
    plan = gdn.gdn_prefill_plan_for(sh, 1, 4133, 0, gdn.PREFILL_TWO_KERNELS)
    if plan["chunk_launches"] < 2:
        pytest.skip(f"this GPU runs the two kernels one after the other: {plan}")
    level_tokens = plan["piece_chunks"] * 64
    jb = next(j for j in range(4) if (j + 1) * sh.block_size > level_tokens)   # a boundary past level 0
    bt = [[1, 2, 3, 4]]
    bt[0][jb] = 99
    cu, ((o_f, pool_f, e_f), (o_2, pool_2, e_2)) = _paths_with_error(sh, [4133], bt, 89, 5, max_seq_len=4133)
    assert e_f == e_2 == gdn.STATUS_CODE["GDN_ERR_PAGE_RANGE"]
    assert torch.equal(o_f.view(torch.int16), o_2.view(torch.int16))
    assert torch.equal(pool_f, pool_2)


def test_overlapped_levels_capture_into_a_cuda_graph():
    """The two kernels' overlapped levels (a fork onto the second stream and a
    join back per call) captured into a CUDA graph: a replay gives the eager
    call's bits (outputs and pool)."""
    sh = inputs.QWEN27B
    T = 4133
    plan = gdn.gdn_prefill_plan_for(sh, 1, T, 0, gdn.PREFILL_TWO_KERNELS)
    if plan["chunk_launches"] < 2:
        pytest.skip(f"this GPU runs the two kernels one after the other: {plan}")
    ti = inputs.token_inputs(sh, T, seed=90)
    w = inputs.conv_weights(sh, 90).cuda()
    x, g, beta = ti["x"].cuda(), ti["g"].cuda(), ti["beta"].cuda()
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    start = torch.zeros(1, dtype=torch.int64, device="cuda")
    init = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    bt = torch.tensor([[1, 2, 3, 4]], dtype=torch.int32, device="cuda")
    slot = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = gdn.workspace_for(gdn.gdn_prefill_workspace_size(sh, 1, T))
    runs = []
    for _ in range(2):
        pool = gdn.StatePool(sh, 5, fill=0)
        o = torch.full((T, sh.num_v_heads, sh.head_dim_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        runs.append((pool, o, err))
    call = lambda pool, o, err: gdn.gdn_prefill_chunked(
        sh, pool, cu_seqlens=cu, start_pos=start, init_page=init, block_table=bt, out_slot=slot, x=x, g=g,
        beta=beta, conv_w=w, o=o, dev_error=err, start_pos_host=[0], init_page_host=[-1], workspace=ws,
        max_seq_len=T, path=gdn.PREFILL_TWO_KERNELS)
    call(*runs[0])                       # eager (also makes the second stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(*runs[1])
    graph.replay()
    torch.cuda.synchronize()
    (p0, o0, e0), (p1, o1, e1) = runs
    assert e0.item() == 0 and e1.item() == 0
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(p0.buf, p1.buf)
