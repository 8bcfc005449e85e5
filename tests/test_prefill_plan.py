"""The prefill's launch plan (host arithmetic, no GPU): when the (sequence,
value head) chains outnumber the SMs, the chains are cut into pieces run level
by level over several launches.  The CTA -> piece map of the kernel is played
out here for many shapes and SM counts: every chain gets each of its pieces
once, in launches that strictly increase with the piece, no launch holds two
pieces of one chain or more CTAs than the GPU has SMs, and the pieces cover a
chain's chunks exactly once for any length up to the bound (the last piece
runs to the end, so even a longer sequence is covered)."""
import itertools

import pytest

import gated_deltanet_state_gb300 as gdn
from gated_deltanet_state_gb300 import inputs


def _play(plan, N, Hv):
    """chain -> [(launch, level)] as the kernel maps CTA (h, b) of launch t."""
    per = plan["ctas_per_launch"] // Hv
    pairs = plan["levels"] * N
    runs = {}
    for t in range(plan["launches"]):
        base = t * per
        s0, level0 = base % N, base // N
        cnt = min(per, pairs - base)
        assert cnt >= 1
        seen = set()
        for b in range(cnt):
            s, level = s0 + b, level0
            if s >= N:
                s, level = s - N, level + 1
            assert s not in seen, "two pieces of one chain in one launch"
            seen.add(s)
            for h in range(Hv):
                runs.setdefault((s, h), []).append((t, level))
        assert cnt * Hv <= max(plan["ctas_per_launch"], 1)
    return runs


def _chunks(plan, level, nch):
    P = plan["piece_chunks"]
    lo = level * P
    hi = nch if level == plan["levels"] - 1 else min(nch, lo + P)
    return range(lo, hi) if (lo < nch or level == 0) else range(0)


SHAPES = [(48, 1), (48, 3), (48, 4), (48, 5), (48, 8), (48, 64), (32, 8), (32, 5), (6, 40), (64, 3), (2, 200)]
LENS = [0, 64, 500, 1024, 2048, 8192, 229376]
SMS = [152, 148, 132, 16]


@pytest.mark.parametrize("path", [gdn.PREFILL_FUSED, gdn.PREFILL_TWO_KERNELS], ids=["fused", "chain"])
@pytest.mark.parametrize("Hv,N", SHAPES)
def test_plan_runs_every_piece_once_in_order(Hv, N, path):
    sh = inputs.LayerShape(max(1, Hv // 3) if Hv % 3 == 0 else Hv, Hv, 128, 128, block_size=896, chunk_size=64)
    for max_len, sms in itertools.product(LENS, SMS):
        plan = gdn.gdn_prefill_plan_for(sh, N, max_len, sms, path)
        assert plan.pop("two_kernels") == (path == gdn.PREFILL_TWO_KERNELS)
        assert plan["chains"] == Hv * N
        maxc = -(-max_len // 64)
        chunk_launches = plan.pop("chunk_launches")
        if chunk_launches > 1:
            # only the two kernels, with one round of chains of 32 chunks or more
            assert path == gdn.PREFILL_TWO_KERNELS and 0 < Hv * N <= sms and maxc >= 32
            # levels of every chain, each after the chunk launch of its chunks
            assert chunk_launches == plan["levels"] == plan["launches"] > 1
            assert plan["ctas_per_launch"] == Hv * N and 16 <= plan["piece_chunks"] <= maxc // 2
            assert plan["levels"] <= 64
            segs = [range(lv * plan["piece_chunks"], min(maxc, (lv + 1) * plan["piece_chunks"]))
                    for lv in range(chunk_launches)]
            assert [c for r in segs for c in r] == list(range(maxc))
            for lv in range(plan["levels"]):
                # level lv reads only chunks the launches up to lv produced
                assert all(c < segs[lv].stop for c in _chunks(plan, lv, maxc))
        else:
            assert chunk_launches == (int(Hv * N > 0) if path == gdn.PREFILL_TWO_KERNELS else 0)
        if plan["levels"] > 1:
            P = plan["piece_chunks"]
            assert P >= 4 and P % 2 == 0, "pieces start at even chunks"
            assert plan["ctas_per_launch"] <= sms and plan["ctas_per_launch"] % Hv == 0
            assert plan["launches"] <= 64
        else:
            assert plan["launches"] == 1 and plan["ctas_per_launch"] == Hv * N
        runs = _play(plan, N, Hv)
        assert len(runs) == Hv * N
        for key, lst in runs.items():
            assert [lv for _, lv in lst] == list(range(plan["levels"])), key
            assert all(t0 < t1 for (t0, _), (t1, _) in zip(lst, lst[1:])), key
        # coverage for lengths up to the bound, and past it
        for nch in sorted({0, 1, maxc // 2, max(maxc - 1, 0), maxc, maxc + 3}):
            covered = [c for lv in range(plan["levels"]) for c in _chunks(plan, lv, nch)]
            assert covered == list(range(nch)), (max_len, sms, nch)


def test_benchmark_shape_plan():
    # 4 x 8,192 tokens of the 27B-shaped layer on 152 SMs: 44-chunk pieces
    # (the last 40), three (level, sequence) pairs of 48 CTAs a launch, 12
    # pairs in 4 launches: ~4 x 44 chunk times against 2 x 128 in one launch
    for path in (gdn.PREFILL_FUSED, gdn.PREFILL_TWO_KERNELS):
        two = int(path == gdn.PREFILL_TWO_KERNELS)
        plan = gdn.gdn_prefill_plan_for(inputs.QWEN27B, 4, 8192, 152, path)
        assert plan == {"chains": 192, "piece_chunks": 44, "levels": 3, "ctas_per_launch": 144, "launches": 4,
                        "two_kernels": two, "chunk_launches": two}
        # a large batch (3,072 chains) stays one launch
        assert gdn.gdn_prefill_plan_for(inputs.QWEN27B, 64, 8192, 152, path)["launches"] == 1
    # one long sequence (48 chains): one launch of the fused kernel; the two
    # kernels overlap 20 levels of 180 chunks with the chunk kernel
    assert gdn.gdn_prefill_plan_for(inputs.QWEN27B, 1, 229376, 152, gdn.PREFILL_FUSED)["launches"] == 1
    plan = gdn.gdn_prefill_plan_for(inputs.QWEN27B, 1, 229376, 152, gdn.PREFILL_TWO_KERNELS)
    assert plan == {"chains": 48, "piece_chunks": 180, "levels": 20, "ctas_per_launch": 48, "launches": 20,
                    "two_kernels": 1, "chunk_launches": 20}
    # 1 x 8,192: four levels of 32 chunks; 2 x 8,192 (96 chains leave 56 SMs
    # idle) runs the two kernels one after the other
    plan = gdn.gdn_prefill_plan_for(inputs.QWEN27B, 1, 8192, 152, gdn.PREFILL_TWO_KERNELS)
    assert (plan["piece_chunks"], plan["levels"], plan["chunk_launches"]) == (32, 4, 4)
    for N in (2, 3):
        plan = gdn.gdn_prefill_plan_for(inputs.QWEN27B, N, 8192, 152, gdn.PREFILL_TWO_KERNELS)
        assert (plan["levels"], plan["launches"], plan["chunk_launches"]) == (1, 1, 1)


def test_auto_path_follows_the_model():
    """The model behind GDN_PREFILL_AUTO (both paths give the same bits),
    fitted to 17 measured calls of the 27B-shaped layer on 152 SMs, in every
    one of which the two kernels measured faster (e.g. 0.80 / 2.04 / 4.07 ms
    for 1 / 4 / 8 sequences of 8,192 tokens against the fused kernel's 1.80 /
    2.45 / 4.83; 0.129 against 0.161 ms for one of 512): those calls take the
    two kernels; calls of a few chunks, whose chunk kernel and second launch
    cost more than they save, take the fused kernel."""
    auto = lambda N, L: gdn.gdn_prefill_plan_for(inputs.QWEN27B, N, L, 152)["two_kernels"]
    for N, L in [(1, 512), (1, 768), (1, 1024), (2, 1024), (4, 1024), (4, 2048), (8, 2048), (16, 1024),
                 (32, 2048), (64, 512), (1, 8192), (2, 8192), (3, 8192), (4, 8192), (8, 8192), (64, 8192),
                 (1, 65536), (1, 229376)]:
        assert auto(N, L) == 1, (N, L)
    assert auto(1, 64) == 0 and auto(1, 256) == 0


def test_plan_rejects_the_scan_path_and_bad_arguments():
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_prefill_plan_for(inputs.TINY, 4, 1024, 152)
    assert ei.value.status == gdn.STATUS_CODE["GDN_ERR_UNSUPPORTED_SHAPE"]
    with pytest.raises(gdn.GdnError):
        gdn.gdn_prefill_plan_for(inputs.QWEN27B, -1, 1024, 152)
    assert gdn.gdn_prefill_plan_for(inputs.QWEN27B, 0, 1024, 152)["launches"] == 0
