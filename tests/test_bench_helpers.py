"""Host helpers of bench.py on CPU: the count of score elements the forward computes (tile fill)
against a brute-force count, and the DRAM-traffic lookup that trusts a committed ncu summary
only while the kernel sources are unchanged."""
import numpy as np
import pytest

import bench
import oracle
from oracle import masks as om
from workloads import byte_stream, workload


def _brute_elements(rp, ci, block, causal, heads, n_tokens):
    """Per 128-token query tile: the set of (key block) visible to any of its query rows, taken
    token by token from the CSR, times 32-key chunks of 128 rows."""
    nb = rp.shape[1] - 1
    total = 0
    for s in range(rp.shape[0]):
        for q0 in range(0, n_tokens, 128):
            blocks = set()
            for i in range(q0, min(n_tokens, q0 + 128)):
                I = i // block
                for J in ci[rp[s, I]:rp[s, I + 1]]:
                    if not causal or J <= I:
                        blocks.add(int(J))
            total += len(blocks) * max(1, block // 32)
    return total * 32 * 128 * heads


@pytest.mark.parametrize("block,causal,mode", [(32, 0, "bigbird"), (64, 1, "topk"), (128, 1, "topk"),
                                               (32, 1, "full")])
def test_tile_elements_match_brute_force(block, causal, mode):
    n = 1024
    if mode == "topk":
        cfg = workload("tiny_topk")
        p = om.MaskParams(mode="topk", block=block, n_tokens=n, causal=1, window_blocks=2, global_blocks=1, topk=3)
        data = np.resize(byte_stream(cfg)[0], (2, n))
        rp, ci = om.build_csr(p, oracle.block_ratios(data, block, 6), 2)
    elif mode == "bigbird":
        p = om.MaskParams(mode="bigbird", block=block, n_tokens=n, causal=0, window_blocks=4, global_blocks=1,
                          random_blocks=1, seed=7)
        rp, ci = om.build_csr(p, None, 1)
    else:
        p = om.MaskParams(mode="full", block=block, n_tokens=n, causal=1)
        rp, ci = om.build_csr(p, None, 1)
    got = bench._csr_tile_elements(rp, ci, block, causal, 3)
    assert got == _brute_elements(rp, ci, block, causal, 3, n)
    # every mask edge lies inside a computed chunk
    assert bench._csr_edges(rp, ci, block, causal, 3) <= got


def test_recorded_traffic_only_for_unchanged_sources(monkeypatch):
    got = bench.recorded_traffic("attn_fwd_bytelm_topk_8k.md", bench.ATTN_FWD_SOURCES)
    digest = bench.source_digest(bench.ATTN_FWD_SOURCES)
    with open(bench.os.path.join(bench.ROOT, "profiles", "attn_fwd_bytelm_topk_8k.md")) as f:
        text = f.read()
    if f"kernel_source_sha256_16: {digest}" in text:
        assert isinstance(got, int) and got > 150_000_000     # at least Q, K, V of the 8K workload
    else:
        assert got is None
    monkeypatch.setattr(bench, "source_digest", lambda names: "0" * 16)
    assert bench.recorded_traffic("attn_fwd_bytelm_topk_8k.md", bench.ATTN_FWD_SOURCES) is None
    assert bench.recorded_traffic("no_such_profile.md", bench.ATTN_FWD_SOURCES) is None
