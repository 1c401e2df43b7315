"""Split-row combine of the block-sparse forward: long key lists cut into parts that write
partial (O, LSE) to the workspace and are merged by log-sum-exp.

A launch splits when it has few work items (query tiles x heads x sequences: fewer than
four per SM at d = 32 or 64, fewer than one per SM at d = 128), its longest key list exceeds
1.25x an even share and its workspace has room for partial results; the shapes below are
chosen so that it does (one or two sequences and heads with long rows: the full causal mask, BigBird's
global rows that attend to every key). Each case is compared with the float64 oracle on
every row, and the workspace's split header (list length, split entries, key tiles per part,
split items; 16 bytes at offset 64) must show that items were split. The same call with a
256-byte workspace (no room for partial results, so no split) must agree within tolerance.
"""
import numpy as np
import pytest

import content_adaptive_sparse_gb300 as sa
import oracle
from oracle import masks as om
from workloads import bf16_bits_to_f64, bf16_normal_bits
from gpu_helpers import assert_attention_close, bf16_to_f64, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


def _split_header(ws):
    h = ws[64:80].cpu().numpy().view(np.int32)
    return {"list_len": int(h[0]), "n_split": int(h[1]), "part_tiles": int(h[2]), "n_split_items": int(h[3])}


def _run(p: om.MaskParams, bt, h, hkv, d, seed, qmul=2.0, ratios=None, csr_shared=False, rows=None):
    torch = torch_cuda()
    rng = np.random.default_rng(seed)
    n, b = p.n_tokens, p.block
    qb = bf16_normal_bits(rng, (bt, n, h, d), 0.25 * qmul)
    kb = bf16_normal_bits(rng, (bt, n, hkv, d), 0.25)
    vb = bf16_normal_bits(rng, (bt, n, hkv, d), 0.25)
    ncsr = 1 if csr_shared else bt
    if rows is None:
        prm = sa.mask_params(p.mode, b, n, ncsr, p.causal, p.window_blocks, p.global_blocks, p.topk,
                             p.random_blocks, p.seed, p.components)
        r = None if ratios is None else torch.from_numpy(np.ascontiguousarray(ratios)).cuda()
        rp_d, ci_d = sa.build_mask(prm, r)
        rp_o, ci_o = om.build_csr(p, ratios, ncsr)
    else:
        nb = n // b
        rp_o = np.zeros((ncsr, nb + 1), dtype=np.int32)
        cols = []
        for s in range(ncsr):
            rp_o[s, 0] = len(cols)
            for I, row in enumerate(rows):
                cols += row
                rp_o[s, I + 1] = len(cols)
        ci_o = np.array(cols, dtype=np.int32)
        rp_d, ci_d = torch.from_numpy(rp_o).cuda(), torch.from_numpy(ci_o).cuda()
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    ws = sa.fwd_workspace(q, b, csr_shared)
    o = torch.empty_like(q)
    lse = torch.empty((bt, h, n), dtype=torch.float32, device="cuda")
    sa.sa_attn_fwd(q, k, v, rp_d, ci_d, b, p.causal, o, lse, csr_shared, workspace=ws)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    hdr = _split_header(ws)
    assert hdr["n_split_items"] > 0 and hdr["n_split"] >= 2 * hdr["n_split_items"], hdr
    f = bf16_bits_to_f64
    o_ref, lse_ref = oracle.attention_csr(f(qb), f(kb), f(vb), rp_o, ci_o, b, p.causal)
    errs = assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                                  f"split {p} d={d}")
    # the same launch without room for partial results (no split)
    small = torch.empty((256,), dtype=torch.uint8, device="cuda")
    o2 = torch.empty_like(q)
    lse2 = torch.empty_like(lse)
    sa.sa_attn_fwd(q, k, v, rp_d, ci_d, b, p.causal, o2, lse2, csr_shared, workspace=small)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    assert_attention_close(bf16_to_f64(o2), lse2.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                           f"unsplit {p} d={d}")
    return hdr, errs


@pytest.mark.parametrize("d,b", [(64, 64), (128, 128), (32, 32)])
def test_split_full_causal_long_rows(d, b):
    """Full causal mask at 8192 tokens with one sequence and two heads: the last query tiles
    hold up to 64 key tiles and are cut into parts."""
    _run(om.MaskParams("full", b, 8192, 1), 1, 2, 1, d, seed=d + b)


def test_split_bigbird_global_rows():
    """BigBird at 4096 tokens, one sequence, two heads: the global block's rows attend to every
    key (32 key tiles), the other rows to about 16 blocks."""
    p = om.MaskParams("bigbird", 32, 4096, 0, 8, 1, 0, 1, 45)
    hdr, _ = _run(p, 1, 2, 2, 64, seed=3, csr_shared=True)


def test_split_ragged_tail_and_empty_rows():
    """65 blocks of 32 tokens (the last query tile holds one block), with some query blocks
    that have no key block at all and one that sees every earlier block."""
    nb = 65
    rows = []
    for I in range(nb):
        if I % 7 == 3:
            rows.append([])
        elif I == nb - 1:
            rows.append(list(range(nb)))
        else:
            rows.append(sorted({0, max(0, I - 1), I}))
    _run(om.MaskParams("full", 32, nb * 32, 1), 1, 1, 1, 64, seed=9, rows=rows)


def test_split_topk_two_sequences_gqa():
    """Compression-guided top-k rows, two sequences with their own CSRs and grouped-query
    attention (2 KV heads for 4 query heads), 4096 tokens."""
    n, b = 4096, 64
    rng = np.random.default_rng(21)
    ratios = (rng.integers(20, 80, (2, n // b)) / np.float32(b)).astype(np.float32)
    p = om.MaskParams("topk", b, n, 1, 4, 1, 40)
    _run(p, 2, 4, 2, 64, seed=22, ratios=ratios)
