"""Full-size workloads against the float64 oracle, on whole query tiles.

Each workload runs at its full size in the launch configuration the bench times, and
every row of several whole 128-row query tiles is compared for every head: the first and
the last tile of the pass, a BigBird global-row tile (its rows attend to every key,
"BigBird" section 2 "Derivation"), and tiles whose key list is longer than one batch of
sixteen 128-key tiles that the kernel's planner publishes at a time. The oracle evaluates
each query block of those tiles from the CSR definition (``attention_csr_block``).
The full causal mask at 16K is also checked against the second, dense route of
"Parameter-free Adaptive Sparse Attention via Compression-Based Content Selection",
section 5 "Limitations" (N x N scores masked by multiplication): a causal query prefix
only sees keys of the prefix, so the dense route on the first 1024 tokens is exact for
those rows.
"""
import functools

import numpy as np
import pytest

import content_adaptive_sparse_gb300 as sa
import oracle
from oracle import masks as om
from workloads import bf16_bits_to_f64, byte_stream, qkv_bits, workload
from gpu_helpers import assert_attention_close, bf16_to_f64, to_dev, torch_cuda

pytestmark = pytest.mark.gpu

TILE = 128          # query rows per work item of the forward kernel
BATCH_KEYS = 16 * 128   # keys the planner publishes per batch entry


@functools.lru_cache(maxsize=2)
def _qkv(name: str):
    return qkv_bits(workload(name))


def _mask_on_gpu(p: om.MaskParams, batch: int, ratios=None):
    torch = torch_cuda()
    prm = sa.mask_params(p.mode, p.block, p.n_tokens, batch, p.causal, p.window_blocks, p.global_blocks, p.topk,
                         p.random_blocks, p.seed, p.components)
    r = None if ratios is None else torch.from_numpy(np.ascontiguousarray(ratios)).cuda()
    return sa.build_mask(prm, r)


def _tile_union_keys(rp, ci, block, causal, s, tile, nb):
    """Keys in the union of the CSR rows of a query tile (what the kernel iterates)."""
    cs = s if rp.shape[0] > 1 else 0
    blocks = set()
    for I in range(tile * TILE // block, min(nb, (tile + 1) * TILE // block)):
        row = ci[rp[cs, I]:rp[cs, I + 1]]
        blocks.update(int(J) for J in row if not causal or J <= I)
    return len(blocks) * block


def _run_and_check_tiles(cfg, p: om.MaskParams, csr_batch, ratios_gpu, ratios_oracle, tiles, need_long=False):
    torch = torch_cuda()
    qb, kb, vb = _qkv(cfg["name"])
    rp_d, ci_d = _mask_on_gpu(p, csr_batch, ratios_gpu)
    shared = csr_batch == 1 and cfg["batch"] > 1
    o, lse = sa.attn_fwd(to_dev(qb), to_dev(kb), to_dev(vb), rp_d, ci_d, p.block, p.causal, csr_shared=shared)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    rp_o, ci_o = om.build_csr(p, ratios_oracle, csr_batch)
    # the GPU mask is bit-exact with the oracle's (its own tests check every workload)
    assert np.array_equal(rp_d.cpu().numpy(), rp_o)
    o_np = bf16_to_f64(o)
    lse_np = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o_np)) and np.all(np.isfinite(lse_np))   # no row is empty in these graphs
    b, nb, h = p.block, p.nb, cfg["heads"]
    if need_long:
        assert any(_tile_union_keys(rp_o, ci_o, b, p.causal, s, t, nb) > BATCH_KEYS for s, t in tiles)
    og, lg, orf, lrf = [], [], [], []
    for s, t in tiles:
        for I in range(t * TILE // b, min(nb, (t + 1) * TILE // b)):
            rows = slice(I * b, (I + 1) * b)
            for hh in range(h):
                ob, lb = oracle.attention_csr_block(qb, kb, vb, rp_o, ci_o, b, p.causal, s, I, hh,
                                                    convert=bf16_bits_to_f64)
                og.append(o_np[s, rows, hh])
                lg.append(lse_np[s, hh, rows])
                orf.append(ob)
                lrf.append(lb)
    return assert_attention_close(np.concatenate(og), np.concatenate(lg), np.concatenate(orf), np.concatenate(lrf),
                                  f"{cfg['name']} tiles {tiles}")


def test_bytelm_topk_8k_whole_tiles():
    cfg = workload("bytelm_topk_8k")
    data = byte_stream(cfg)
    p = om.MaskParams("topk", cfg["block"], cfg["n_tokens"], 1, cfg["window_blocks"], cfg["global_blocks"],
                      cfg["topk"])
    last = cfg["n_tokens"] // TILE - 1
    tiles = [(0, 0), (cfg["batch"] - 1, last), (1, 1), (2, 31), (0, 47), (3, 12), (1, last - 1), (2, 50)]
    _run_and_check_tiles(cfg, p, cfg["batch"], sa.sa_block_ratios(data, cfg["block"]),
                         oracle.block_ratios(data, cfg["block"]), tiles)


@pytest.mark.parametrize("name", ["bigbird_4k", "bigbird_16k"])
def test_bigbird_whole_tiles(name):
    cfg = workload(name)
    b = cfg["block"]
    p = om.MaskParams("bigbird", b, cfg["n_tokens"], 0, cfg["window_tokens"] // b, cfg["global_tokens"] // b, 0,
                      cfg["random_tokens"] // b, cfg["seed"])
    last = cfg["n_tokens"] // TILE - 1
    # tile 0 holds the global block's rows (every key: several batches of key tiles)
    tiles = [(0, 0), (cfg["batch"] - 1, last), (5, 0), (3, 1), (2, last // 2), (6, last - 3), (1, last - 1),
             (4, 7)]
    _run_and_check_tiles(cfg, p, 1, None, None, tiles, need_long=True)


@pytest.mark.parametrize("topk", [16, 64, 256])
def test_long_topk_64k_whole_tiles(topk):
    """The 64K compression-guided workload, d = 128, b = 128, with top-k swept over the
    workload's {16, 64, 256}."""
    cfg = workload("long_topk_64k", topk=topk)
    data = byte_stream(cfg)
    p = om.MaskParams("topk", cfg["block"], cfg["n_tokens"], 1, cfg["window_blocks"], cfg["global_blocks"], topk)
    last = cfg["n_tokens"] // TILE - 1
    tiles = [(0, 0), (0, last), (0, 1), (0, 5), (0, 100), (0, 255), (0, 400), (0, last - 1)]
    _run_and_check_tiles(cfg, p, 1, sa.sa_block_ratios(data, cfg["block"]), oracle.block_ratios(data, cfg["block"]),
                         tiles, need_long=topk >= 64)


def test_full_causal_16k_whole_tiles_and_dense_route():
    """The full causal mask at N = 16384, d = 128: whole tiles against the CSR oracle, and
    the first 1024 rows of every head against the dense masked route."""
    torch = torch_cuda()
    cfg = workload("full_16k")
    p = om.MaskParams("full", cfg["block"], cfg["n_tokens"], 1)
    last = cfg["n_tokens"] // TILE - 1
    tiles = [(0, 0), (0, last), (0, 1), (0, 20), (0, 64), (0, 90), (0, 126), (0, last - 1)]
    _run_and_check_tiles(cfg, p, 1, None, None, tiles, need_long=True)
    # dense route on the causal prefix
    qb, kb, vb = _qkv(cfg["name"])
    m = 1024
    rp_d, ci_d = _mask_on_gpu(p, 1)
    o, lse = sa.attn_fwd(to_dev(qb), to_dev(kb), to_dev(vb), rp_d, ci_d, p.block, 1)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    f = bf16_bits_to_f64
    o_ref, lse_ref = oracle.dense_masked_attention(f(qb[:, :m]), f(kb[:, :m]), f(vb[:, :m]),
                                                   np.tril(np.ones((m, m), dtype=bool)))
    assert_attention_close(bf16_to_f64(o)[:, :m], lse.cpu().numpy().astype(np.float64)[:, :, :m], o_ref, lse_ref,
                           "full 16k vs dense route, first 1024 rows")


def test_cas_heads_8k_whole_tiles():
    """[CAS] head groups at 4 x 8192, b = 128: whole tiles of every head, each head
    against the CSR of its group."""
    torch = torch_cuda()
    cfg = workload("cas_heads_8k")
    data = byte_stream(cfg)
    b, n, bt, h = cfg["block"], cfg["n_tokens"], cfg["batch"], cfg["heads"]
    r_gpu = sa.sa_block_ratios(data, b, cfg["zlib_level"])
    r_ora = oracle.block_ratios(data, b, cfg["zlib_level"])
    comps = list(cfg["head_components"])
    assert comps == oracle.cas_head_components(h)
    parts = sorted(set(comps))
    head_mask = [parts.index(c) for c in comps]
    qb, kb, vb = qkv_bits(cfg)
    csrs_d, csrs_o = [], []
    for c in parts:
        p = om.MaskParams("literal_mean", b, n, 1, cfg["window_blocks"], components=c)
        csrs_d.append(_mask_on_gpu(p, bt, r_gpu))
        csrs_o.append(om.build_csr(p, r_ora, bt))
    o, lse = sa.attn_fwd_heads(to_dev(qb), to_dev(kb), to_dev(vb), csrs_d, head_mask, b, 1)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    o_np, lse_np = bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)
    last = n // TILE - 1
    tiles = [(0, 0), (bt - 1, last), (1, 1), (2, 31), (3, 40), (0, last - 1), (1, 20), (2, 60)]
    og, lg, orf, lrf = [], [], [], []
    for s, t in tiles:
        I = t   # b = 128: one query block per tile
        for hh in range(h):
            rp_o, ci_o = csrs_o[head_mask[hh]]
            ob, lb = oracle.attention_csr_block(qb, kb, vb, rp_o, ci_o, b, 1, s, I, hh, convert=bf16_bits_to_f64)
            og.append(o_np[s, I * b:(I + 1) * b, hh])
            lg.append(lse_np[s, hh, I * b:(I + 1) * b])
            orf.append(ob)
            lrf.append(lb)
    assert_attention_close(np.concatenate(og), np.concatenate(lg), np.concatenate(orf), np.concatenate(lrf),
                           "cas_heads_8k tiles")
