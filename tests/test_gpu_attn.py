"""Block-sparse attention forward (tcgen05 kernel) vs the float64 oracle."""
import numpy as np
import pytest

import content_adaptive_sparse_gb300 as sa
import oracle
from oracle import masks as om
from workloads import bf16_bits_to_f64, bf16_normal_bits, byte_stream, qkv_bits, workload
from gpu_helpers import assert_attention_close, bf16_to_f64, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


def _mask_on_gpu(p: om.MaskParams, batch: int, ratios=None):
    torch = torch_cuda()
    mode = {"topk": 0, "bigbird": 1, "full": 2, "literal_mean": 3}[p.mode]
    prm = sa.mask_params(mode, p.block, p.n_tokens, batch, p.causal, p.window_blocks, p.global_blocks, p.topk,
                         p.random_blocks, p.seed, p.components)
    r = None if ratios is None else torch.from_numpy(np.ascontiguousarray(ratios)).cuda()
    return sa.build_mask(prm, r)


def _run_case(p: om.MaskParams, bt, h, hkv, d, seed=0, qmul=1.0, ratios=None, csr_shared=False, std=0.125):
    """Full comparison at a size the oracle finishes in seconds."""
    torch = torch_cuda()
    rng = np.random.default_rng(seed)
    n = p.n_tokens
    qb = bf16_normal_bits(rng, (bt, n, h, d), std * qmul)
    kb = bf16_normal_bits(rng, (bt, n, hkv, d), std)
    vb = bf16_normal_bits(rng, (bt, n, hkv, d), std)
    rp_d, ci_d = _mask_on_gpu(p, 1 if csr_shared else bt, ratios)
    o, lse = sa.attn_fwd(to_dev(qb), to_dev(kb), to_dev(vb), rp_d, ci_d, p.block, p.causal, csr_shared=csr_shared)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    rp_o, ci_o = om.build_csr(p, ratios, 1 if csr_shared else bt)
    o_ref, lse_ref = oracle.attention_csr(bf16_bits_to_f64(qb), bf16_bits_to_f64(kb), bf16_bits_to_f64(vb), rp_o,
                                          ci_o, p.block, p.causal)
    return assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                                  f"{p} d={d}")


def test_tiny_topk_workload():
    cfg = workload("tiny_topk")
    data = byte_stream(cfg)
    ratios = oracle.block_ratios(data, cfg["block"])
    p = om.MaskParams("topk", cfg["block"], cfg["n_tokens"], 1, cfg["window_blocks"], cfg["global_blocks"],
                      cfg["topk"])
    for qmul in (1.0, 8.0):   # 8x: softmax far from uniform (stress of the running max)
        _run_case(p, 1, cfg["heads"], cfg["kv_heads"], cfg["head_dim"], seed=43, qmul=qmul, ratios=ratios,
                  std=cfg["std"])


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("b", [32, 64, 128])
def test_full_causal_all_shapes(d, b):
    _run_case(om.MaskParams("full", b, 512, 1), 2, 2, 2, d, seed=d + b, qmul=4.0)


@pytest.mark.parametrize("d,b", [(64, 32), (128, 128), (32, 64)])
def test_full_bidirectional(d, b):
    _run_case(om.MaskParams("full", b, 384, 0), 1, 3, 1, d, seed=7)


@pytest.mark.parametrize("b,d", [(64, 64), (128, 128), (32, 32), (32, 64)])
def test_topk_several_tiles_gqa(b, d):
    n = 2048
    rng = np.random.default_rng(b * d)
    ratios = (rng.integers(20, 80, (2, n // b)) / np.float32(b)).astype(np.float32)
    p = om.MaskParams("topk", b, n, 1, 3, 1, 5)
    _run_case(p, 2, 4, 2, d, seed=3, qmul=3.0, ratios=ratios)


def test_bigbird_small_shared_csr():
    p = om.MaskParams("bigbird", 32, 1024, 0, 8, 1, 0, 1, 45)
    _run_case(p, 2, 2, 2, 64, seed=11, qmul=2.0, csr_shared=True)


def test_literal_mean_mode():
    n, b = 2048, 64
    rng = np.random.default_rng(5)
    ratios = (rng.integers(20, 90, (2, n // b)) / np.float32(b)).astype(np.float32)
    for causal in (1, 0):
        _run_case(om.MaskParams("literal_mean", b, n, causal, 1), 2, 2, 2, 64, seed=causal, ratios=ratios)


def test_ragged_tail_tile():
    # 13 blocks of 32: the last 128-row tile holds one query block
    p = om.MaskParams("full", 32, 416, 1)
    _run_case(p, 1, 2, 2, 64, seed=5, qmul=2.0)
    p = om.MaskParams("bigbird", 32, 416, 0, 4, 1, 0, 2, 3)
    _run_case(p, 2, 2, 1, 64, seed=6)


def test_empty_rows_and_strided_inputs():
    torch = torch_cuda()
    rng = np.random.default_rng(9)
    bt, n, h, d, b = 2, 256, 2, 64, 32
    packed = bf16_normal_bits(rng, (bt, n, 3, h, d), 0.5)   # q, k, v interleaved: strided views
    t = to_dev(packed)
    q, k, v = t[:, :, 0], t[:, :, 1], t[:, :, 2]
    nb = n // b
    rows = [[0], [], [0, 1], [2], [], [1, 3, 5], [6], [0, 7]]
    rp = np.zeros((bt, nb + 1), dtype=np.int32)
    cols = []
    for s in range(bt):
        rp[s, 0] = len(cols)
        for I, row in enumerate(rows):
            cols += row
            rp[s, I + 1] = len(cols)
    ci = np.array(cols, dtype=np.int32)
    o, lse = sa.attn_fwd(q, k, v, torch.from_numpy(rp).cuda(), torch.from_numpy(ci).cuda(), b, 1)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    f = bf16_bits_to_f64(packed)
    o_ref, lse_ref = oracle.attention_csr(f[:, :, 0], f[:, :, 1], f[:, :, 2], rp, ci, b, 1)
    assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, "empty rows")
    assert np.all(bf16_to_f64(o)[:, 32:64] == 0)


@pytest.mark.parametrize("steep", [6.0, 2.0])
@pytest.mark.parametrize("d,b", [(64, 64), (128, 128), (64, 32), (32, 32)])
def test_running_max_rescale_paths(d, b, steep):
    """Logits that grow along the sequence (and jump inside a key tile) force the
    running-max updates: first-tile init, O rescale, and (steep = 2: the logits of each
    128-key tile exceed the running max by far more than 2^32 / 128) a tile recomputed
    against its exact max."""
    torch = torch_cuda()
    rng = np.random.default_rng(d + b)
    n, h = 768, 2
    base = np.arange(n, dtype=np.float32)[None, :, None, None] / np.float32(steep)
    sign = np.where(rng.random((1, n, h, 1)) < 0.5, -1.0, 1.0).astype(np.float32)
    qf = np.ones((1, n, h, d), np.float32) * 0.5 + 0.05 * rng.standard_normal((1, n, h, d), dtype=np.float32)
    kf = (base * (1.0 + 0.3 * sign)) * np.ones((1, n, h, d), np.float32) / np.float32(np.sqrt(d))
    vf = rng.standard_normal((1, n, h, d), dtype=np.float32)
    from workloads import _f32_to_bf16_bits
    qb, kb, vb = (_f32_to_bf16_bits(a) for a in (qf, kf, vf))
    for mode in ("full", "topk"):
        if mode == "full":
            p = om.MaskParams("full", b, n, 1)
            ratios = None
        else:
            p = om.MaskParams("topk", b, n, 1, 2, 1, 3)
            ratios = (rng.integers(20, 60, (1, n // b)) / np.float32(b)).astype(np.float32)
        rp_d, ci_d = _mask_on_gpu(p, 1, ratios)
        o, lse = sa.attn_fwd(to_dev(qb), to_dev(kb), to_dev(vb), rp_d, ci_d, b, 1)
        torch.cuda.synchronize()
        assert sa.sa_device_status() == 0
        rp_o, ci_o = om.build_csr(p, ratios, 1)
        o_ref, lse_ref = oracle.attention_csr(bf16_bits_to_f64(qb), bf16_bits_to_f64(kb), bf16_bits_to_f64(vb),
                                              rp_o, ci_o, b, 1)
        assert np.max(lse_ref) > 60.0          # the logit range really spans many 2^8 steps
        assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                               f"rescale {mode} d={d} b={b}")


def test_bounded_wait_times_out_and_context_survives():
    """A wait on a barrier nothing completes gives up after the wait limit and reports
    SA_ERR_TIMEOUT; the status is cleared by the read and the device keeps working."""
    torch = torch_cuda()
    sa.sa_selftest_bounded_wait()
    assert sa.sa_device_status() == -5
    assert sa.sa_device_status() == 0
    _run_case(om.MaskParams("full", 64, 256, 1), 1, 2, 2, 64, seed=12)


def test_bad_csr_index_is_reported():
    torch = torch_cuda()
    bt, n, h, d, b = 1, 256, 1, 64, 64
    x = torch.zeros((bt, n, h, d), dtype=torch.bfloat16, device="cuda")
    rp = torch.tensor([[0, 1, 3, 4, 5]], dtype=torch.int32, device="cuda")
    ci = torch.tensor([0, 0, 9, 2, 3], dtype=torch.int32, device="cuda")   # 9 is out of range
    o, lse = sa.attn_fwd(x, x, x, rp, ci, b, 1)
    assert sa.sa_device_status() == -6
    assert sa.sa_device_status() == 0          # the status word was cleared


# Full-size workloads (whole query tiles of every head) are in test_gpu_fullsize.py.


# ---------------------------------------------------------------- head groups (per-head CSR)

def _head_group_case(bt, n, b, h, hkv, d, w, causal, comps, seed, ratios, qmul=2.0):
    torch = torch_cuda()
    rng = np.random.default_rng(seed)
    qb = bf16_normal_bits(rng, (bt, n, h, d), 0.125 * qmul)
    kb = bf16_normal_bits(rng, (bt, n, hkv, d), 0.125)
    vb = bf16_normal_bits(rng, (bt, n, hkv, d), 0.125)
    parts = sorted(set(comps))
    head_mask = [parts.index(c) for c in comps]
    csrs_d, csrs_o = [], []
    for c in parts:
        p = om.MaskParams("literal_mean", b, n, causal, w, components=c)
        csrs_d.append(_mask_on_gpu(p, bt, ratios))
        csrs_o.append(om.build_csr(p, ratios, bt))
    o, lse = sa.attn_fwd_heads(to_dev(qb), to_dev(kb), to_dev(vb), csrs_d, head_mask, b, causal)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    o_ref, lse_ref = oracle.attention_csr_heads(bf16_bits_to_f64(qb), bf16_bits_to_f64(kb), bf16_bits_to_f64(vb),
                                                csrs_o, head_mask, b, causal)
    assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                           f"head groups b={b} d={d} causal={causal}")


@pytest.mark.parametrize("b,d,causal", [(128, 64, 1), (64, 64, 0), (32, 128, 1), (128, 32, 0)])
def test_head_groups_against_oracle(b, d, causal):
    """The page's split (6 local, 3 long-range, 3 hybrid heads) with 3 KV heads, so that
    KV groups straddle head groups (KV head 1 serves local heads 4-5 and literal heads
    6-7; KV head 2 serves literal head 8 and hybrid heads 9-11)."""
    n, bt = 1536, 2
    rng = np.random.default_rng(b + d)
    ratios = (rng.integers(20, 90, (bt, n // b)) / np.float32(b)).astype(np.float32)
    comps = oracle.cas_head_components(12)
    _head_group_case(bt, n, b, 12, 3, d, 1, causal, comps, seed=b * d + causal, ratios=ratios)


def test_head_groups_interleaved_and_single_mask():
    """Heads that alternate between CSRs, and n_masks = 1 through the per-head entry
    point, which must equal sa_attn_fwd bit for bit."""
    torch = torch_cuda()
    n, b, bt = 1024, 64, 1
    rng = np.random.default_rng(77)
    ratios = (rng.integers(20, 90, (bt, n // b)) / np.float32(b)).astype(np.float32)
    _head_group_case(bt, n, b, 5, 5, 64, 2, 1, [2, 1, 0, 1, 2], seed=3, ratios=ratios, qmul=4.0)
    p = om.MaskParams("literal_mean", b, n, 1, 1)
    rp, ci = _mask_on_gpu(p, bt, ratios)
    q, k, v = (to_dev(bf16_normal_bits(rng, (bt, n, 3, 64), 0.25)) for _ in range(3))
    o1, l1 = sa.attn_fwd(q, k, v, rp, ci, b, 1)
    o2, l2 = sa.attn_fwd_heads(q, k, v, [(rp, ci)], [0, 0, 0], b, 1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_head_groups_eight_masks_sixteen_heads():
    """The maximum of 8 CSRs, 16 query heads over 4 KV heads, two masks unused, heads of
    one KV group spread over several masks."""
    torch = torch_cuda()
    n, b, bt, h, hkv = 1024, 64, 2, 16, 4
    rng = np.random.default_rng(88)
    ratios = (rng.integers(20, 90, (bt, n // b)) / np.float32(b)).astype(np.float32)
    params = [om.MaskParams("topk", b, n, 1, 2, 1, 3), om.MaskParams("topk", b, n, 1, 1, 0, 6),
              om.MaskParams("full", b, n, 1), om.MaskParams("literal_mean", b, n, 1, 1, components=1),
              om.MaskParams("literal_mean", b, n, 1, 1, components=2), om.MaskParams("literal_mean", b, n, 1, 2),
              om.MaskParams("topk", b, n, 1, 4, 2, 1), om.MaskParams("full", b, n, 1)]
    head_mask = [int(x) for x in rng.integers(0, 6, h)]          # masks 6 and 7 unused
    qb = bf16_normal_bits(rng, (bt, n, h, 64), 0.4)
    kb, vb = (bf16_normal_bits(rng, (bt, n, hkv, 64), 0.25) for _ in range(2))
    csrs_d = [_mask_on_gpu(p, bt, ratios) for p in params]
    csrs_o = [om.build_csr(p, ratios, bt) for p in params]
    o, lse = sa.attn_fwd_heads(to_dev(qb), to_dev(kb), to_dev(vb), csrs_d, head_mask, b, 1)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    o_ref, lse_ref = oracle.attention_csr_heads(bf16_bits_to_f64(qb), bf16_bits_to_f64(kb), bf16_bits_to_f64(vb),
                                                csrs_o, head_mask, b, 1)
    assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, "8 masks")


def test_concurrent_launches_on_four_streams():
    """Four forward launches in flight at once on four streams (each launch takes a work
    counter slot of its own; both forward kernels and both head-dimension paths); every
    result matches the oracle."""
    torch = torch_cuda()
    shapes = [(64, 64, 1), (32, 32, 1), (64, 128, 0), (128, 64, 1)]   # (d, b, causal)
    n, bt, h = 1024, 2, 2
    cases = []
    for i, (d, b, causal) in enumerate(shapes):
        rng = np.random.default_rng(300 + i)
        p = om.MaskParams("full", b, n, causal)
        bits = [bf16_normal_bits(rng, (bt, n, h, d), 0.25) for _ in range(3)]
        rp_d, ci_d = _mask_on_gpu(p, bt)
        cases.append((p, bits, rp_d, ci_d))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in shapes]
    outs = []
    for s, (p, bits, rp_d, ci_d) in zip(streams, cases):
        with torch.cuda.stream(s):
            q, k, v = (to_dev(x) for x in bits)
            outs.append(sa.attn_fwd(q, k, v, rp_d, ci_d, p.block, p.causal))
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    for (p, bits, _, _), (o, lse), (d, _, _) in zip(cases, outs, shapes):
        rp_o, ci_o = om.build_csr(p, None, bt)
        f = [bf16_bits_to_f64(x) for x in bits]
        o_ref, lse_ref = oracle.attention_csr(f[0], f[1], f[2], rp_o, ci_o, p.block, p.causal)
        assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                               f"stream case d={d} b={p.block} causal={p.causal}")


@pytest.mark.parametrize("d", [32, 64, 128])
def test_items_spanning_several_tile_batches(d):
    """Full causal mask at 4096 tokens with 32-token blocks: the last query tiles' key lists
    hold 128 blocks = 32 key tiles of 128 keys, published in more than one batch of tiles;
    the item's output must not depend on where the batches split it."""
    _run_case(om.MaskParams("full", 32, 4096, 1), 1, 1, 1, d, seed=40 + d, qmul=2.0)


@pytest.mark.parametrize("d", [64, 128])
def test_many_items_per_cta_with_keyless_items(d):
    """640 work items (more than four per SM, so no split and each CTA runs a stream of
    several items) over a random causal CSR in which about a third of the query blocks have
    no key block at all: items without key tiles interleave with items of one to eight key
    tiles, so the hand-over of each item's output, and of O to the next item, happens many
    times per CTA (at d = 128 through the epilogue warps)."""
    torch = torch_cuda()
    rng = np.random.default_rng(70 + d)
    bt, n, h, hkv, b = 4, 2048, 10, 5, 128
    nb = n // b
    rp = np.zeros((bt, nb + 1), dtype=np.int32)
    cols = []
    for s in range(bt):
        rp[s, 0] = len(cols)
        for I in range(nb):
            row = []
            if rng.random() >= 0.35:
                picks = set(rng.integers(0, I + 1, size=int(rng.integers(1, 9))).tolist())
                if rng.random() < 0.5:
                    picks.add(I)
                row = sorted(picks)
            cols += row
            rp[s, I + 1] = len(cols)
    ci = np.array(cols, dtype=np.int32)
    qb = bf16_normal_bits(rng, (bt, n, h, d), 0.25)
    kb = bf16_normal_bits(rng, (bt, n, hkv, d), 0.25)
    vb = bf16_normal_bits(rng, (bt, n, hkv, d), 0.25)
    o, lse = sa.attn_fwd(to_dev(qb), to_dev(kb), to_dev(vb), torch.from_numpy(rp).cuda(),
                         torch.from_numpy(ci).cuda(), b, 1)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    f = bf16_bits_to_f64
    o_ref, lse_ref = oracle.attention_csr(f(qb), f(kb), f(vb), rp, ci, b, 1)
    assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                           f"many items d={d}")
    # rows of key-less query blocks: O = 0 and LSE = -inf
    empty = [(s, I) for s in range(bt) for I in range(nb) if rp[s, I + 1] == rp[s, I]]
    assert empty
    oh, lh = bf16_to_f64(o), lse.cpu().numpy()
    for s, I in empty[:8]:
        assert np.all(oh[s, I * b:(I + 1) * b] == 0) and np.all(np.isneginf(lh[s, :, I * b:(I + 1) * b]))
