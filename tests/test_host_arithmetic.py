"""Host arithmetic of the engine (libgdn.so) against the pages' worked values.

Integer results must match bit for bit.  Fixtures: tests/golden/page_arithmetic.json.
"""
import json
import os

import pytest

import gated_deltanet_state_gb300 as gdn
from gated_deltanet_state_gb300 import inputs

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_arithmetic.json")))
MIB = 1 << 20


def _shape(d):
    return inputs.LayerShape(d["Hqk"], d["Hv"], d["dk"], d["dv"], block_size=64, chunk_size=64,
                             in_dtype=inputs.BF16, out_dtype=inputs.BF16)


def test_mamba_page_bytes_27b():
    for e in GOLD["mamba_page_bytes"]:
        assert gdn.gdn_mamba_page_bytes(_shape(e["desc"])) == e["bytes"]
    e = GOLD["mib_rounding"][0]
    assert f"{e['bytes'] / MIB:.2f}" == e["mib_2dp"]
    assert f"{e['bytes'] / 1e6:.2f}" == e["mb_2dp"]
    e = GOLD["per_sequence_state"][0]
    assert f"{e['bytes_per_layer'] * e['gdn_layers'] / 1e6:.1f}" == e["mb_1dp"]
    e = GOLD["attn_bytes_per_token"][0]
    assert e["per_layer"] * e["attn_layers"] == e["total"]


def test_state_bytes_4b_fits_page():
    e = GOLD["state_bytes_4b"][0]
    sh = _shape(e["desc"])
    assert sh.state_bytes == e["state_bytes"] == 2 * MIB
    assert gdn.gdn_mamba_page_bytes(sh) == 2_146_304 <= e["page_bytes"]
    assert inputs.QWEN4B.page == e["page_bytes"]


def test_block_size_for():
    for e in GOLD["block_size_for"]:
        assert gdn.gdn_block_size_for(e["mamba_page"], e["attn_bytes_per_token"], e["alignment"]) == e["block"]
    assert gdn.gdn_block_size_for(0, 4096, 16) == -1


def test_pages_and_blocks_per_request():
    for e in GOLD["pages_per_request"]:
        pages = gdn.gdn_mamba_pages_per_request(e["gdn_layers"], e["prefix_caching"], e["spec"])
        assert pages == e["pages"]
        assert gdn.gdn_pool_blocks_for_pages(pages, e["layers_per_block"]) == e["blocks"]


def test_chunk_end_floors_to_blocks():
    for e in GOLD["chunk_end"]:
        assert gdn.gdn_chunk_end(e["computed"], e["tokens"], e["budget"], e["block"]) == e["end"]
    # never 2048 at block 784, whatever the start inside the schedule
    for start in range(0, 20 * 784, 784):
        assert gdn.gdn_chunk_end(start, 10**9, 2048, 784) - start in (784, 1568)
    # the final chunk may end inside a block
    assert gdn.gdn_chunk_end(896, 1000, 1024, 896) == 1000
    # a budget below one block schedules nothing before the final chunk
    assert gdn.gdn_chunk_end(896, 10**6, 500, 896) == 896


def test_cached_tokens_rule():
    for e in GOLD["cached_tokens"]:
        assert gdn.gdn_cached_tokens(e["shared"], e["block"]) == e["cached"]
    for shared in range(0, 5000, 37):
        c = gdn.gdn_cached_tokens(shared, 896)
        assert c == (max(0, shared // 896 - 1)) * 896
        assert c % 896 == 0 and (c == 0 or c <= shared - 896)


def test_resume_block():
    for e in GOLD["resume_block"]:
        assert gdn.gdn_resume_block(e["hit"], e["block"]) == e["resume"]
    assert gdn.gdn_resume_block(0, 896) == -1
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_resume_block(200_000, 896)
    assert ei.value.status == gdn.STATUS_CODE["GDN_ERR_NOT_BLOCK_ALIGNED"]


def test_spec_copy_and_replay_bytes():
    e = GOLD["spec_copy_bytes"][0]
    b = gdn.gdn_spec_copy_bytes(e["draft"], e["layers"], e["page_bytes"])
    assert b == e["bytes"] and b == e["mib"] * MIB
    e2 = GOLD["spec_copy_bytes"][1]
    per = gdn.gdn_spec_copy_bytes(16, 24, e2["page_bytes"]) - gdn.gdn_spec_copy_bytes(15, 24, e2["page_bytes"])
    assert per == e2["per_draft_token_mib"] * MIB
    e = GOLD["replay_bytes"][0]
    assert e["slot_bytes"] == inputs.QWEN4B.conv_dim * 2
    assert gdn.gdn_replay_bytes_per_request(e["layers"], e["page_bytes"], e["slots"], e["slot_bytes"]) == e["mib"] * MIB


def test_27b_config_block_geometry():
    sh = inputs.QWEN27B
    page = gdn.gdn_mamba_page_bytes(sh)
    assert gdn.gdn_block_size_for(page, 4096, 128) == sh.block_size == 896
    assert sh.page == 896 * 4096 >= page
    # config 5: a prefix of 200,000 shared tokens resumes from block 222
    # (state after 199,808 tokens); the cached-token rule stops one block earlier
    assert gdn.gdn_resume_block(200_000 // 896 * 896, 896) == 222
    assert gdn.gdn_cached_tokens(200_000, 896) == 198_912


def _boundary_rows_brute(absorbed, kept, block):
    # the states after 1..kept more rows sit at absorbed + j; block boundaries are positive multiples
    hits = [j for j in range(1, kept + 1) if (absorbed + j) % block == 0]
    return 0 if not hits else (hits[0] if len(hits) == 1 else -1)


def test_replay_boundary_rows():
    # a flush of kept rows crosses at most one boundary for blocks above 32 rows
    cases = [(0, 16, 64, 0), (60, 16, 64, 4), (64, 16, 64, 0), (48, 16, 64, 16), (63, 1, 64, 1),
             (10, 200, 64, -1), (199808 - 5, 16, 896, 5), (199808, 32, 896, 0), (0, 0, 64, 0)]
    for absorbed, kept, block, want in cases:
        assert gdn.gdn_replay_boundary_rows(absorbed, kept, block) == want, (absorbed, kept, block)
    for block in (16, 64, 784, 896):
        for absorbed in list(range(0, 3 * block, 7)) + [5 * block - 1, 5 * block]:
            for kept in (0, 1, 15, 16, 17, 31, 32):
                assert gdn.gdn_replay_boundary_rows(absorbed, kept, block) == \
                    _boundary_rows_brute(absorbed, kept, block), (absorbed, kept, block)
    assert gdn.gdn_replay_boundary_rows(-1, 4, 64) == -1
    assert gdn.gdn_replay_boundary_rows(0, -1, 64) == -1
    assert gdn.gdn_replay_boundary_rows(0, 4, 0) == -1
