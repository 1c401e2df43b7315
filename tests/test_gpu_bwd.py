"""Block-sparse attention backward (tcgen05 kernels) vs the float64 oracle."""
import numpy as np
import pytest

import content_adaptive_sparse_gb300 as sa
import oracle
from oracle import masks as om
from workloads import bf16_bits_to_f64, bf16_normal_bits, byte_stream, qkv_bits, workload
from gpu_helpers import assert_grad_close, bf16_to_f64, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


def _mask_on_gpu(p: om.MaskParams, batch: int, ratios=None):
    torch = torch_cuda()
    mode = {"topk": 0, "bigbird": 1, "full": 2, "literal_mean": 3}[p.mode]
    prm = sa.mask_params(mode, p.block, p.n_tokens, batch, p.causal, p.window_blocks, p.global_blocks, p.topk,
                         p.random_blocks, p.seed, p.components)
    r = None if ratios is None else torch.from_numpy(np.ascontiguousarray(ratios)).cuda()
    return sa.build_mask(prm, r)


def _fwd_bwd(qb, kb, vb, dob, rp_d, ci_d, block, causal, csr_shared=False):
    torch = torch_cuda()
    q, k, v, do = (to_dev(x) for x in (qb, kb, vb, dob))
    o, lse = sa.attn_fwd(q, k, v, rp_d, ci_d, block, causal, csr_shared=csr_shared)
    dq, dk, dv = sa.attn_bwd(q, k, v, o, lse, do, rp_d, ci_d, block, causal, csr_shared=csr_shared)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    return dq, dk, dv


def _run_case(p: om.MaskParams, bt, h, hkv, d, seed=0, qmul=1.0, ratios=None, csr_shared=False, std=0.25):
    rng = np.random.default_rng(seed)
    n = p.n_tokens
    qb = bf16_normal_bits(rng, (bt, n, h, d), std * qmul)
    kb = bf16_normal_bits(rng, (bt, n, hkv, d), std)
    vb = bf16_normal_bits(rng, (bt, n, hkv, d), std)
    dob = bf16_normal_bits(rng, (bt, n, h, d), std)
    rp_d, ci_d = _mask_on_gpu(p, 1 if csr_shared else bt, ratios)
    dq, dk, dv = _fwd_bwd(qb, kb, vb, dob, rp_d, ci_d, p.block, p.causal, csr_shared)
    rp_o, ci_o = om.build_csr(p, ratios, 1 if csr_shared else bt)
    f = bf16_bits_to_f64
    rq, rk, rv = oracle.attention_csr_backward(f(qb), f(kb), f(vb), f(dob), rp_o, ci_o, p.block, p.causal)
    what = f"{p} d={d}"
    assert_grad_close(bf16_to_f64(dq), rq, "dQ " + what)
    assert_grad_close(bf16_to_f64(dk), rk, "dK " + what)
    assert_grad_close(bf16_to_f64(dv), rv, "dV " + what)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("b", [32, 64, 128])
def test_full_causal_all_shapes(d, b):
    _run_case(om.MaskParams("full", b, 512, 1), 2, 2, 1, d, seed=d + b, qmul=3.0)


@pytest.mark.parametrize("d,b", [(64, 64), (128, 128), (32, 32)])
def test_topk_several_tiles_gqa(d, b):
    n = 2048
    rng = np.random.default_rng(b * d)
    ratios = (rng.integers(20, 80, (2, n // b)) / np.float32(b)).astype(np.float32)
    _run_case(om.MaskParams("topk", b, n, 1, 3, 1, 5), 2, 4, 2, d, seed=3, qmul=3.0, ratios=ratios)


def test_bigbird_shared_csr_bidirectional():
    _run_case(om.MaskParams("bigbird", 32, 1024, 0, 8, 1, 0, 1, 45), 2, 2, 2, 64, seed=11, qmul=2.0,
              csr_shared=True)


def test_literal_mean_both_directions():
    n, b = 1024, 64
    rng = np.random.default_rng(5)
    ratios = (rng.integers(20, 90, (2, n // b)) / np.float32(b)).astype(np.float32)
    for causal in (1, 0):
        _run_case(om.MaskParams("literal_mean", b, n, causal, 1), 2, 2, 2, 64, seed=causal, ratios=ratios)


def test_ragged_tail_and_empty_key_tiles():
    # 13 blocks of 32: the last 128-row tile holds one block; BigBird leaves key tiles
    # that only some query tiles reach
    _run_case(om.MaskParams("full", 32, 416, 1), 1, 2, 2, 64, seed=5, qmul=2.0)
    _run_case(om.MaskParams("bigbird", 32, 416, 0, 4, 1, 0, 2, 3), 2, 2, 1, 64, seed=6)


def test_empty_rows_and_unreached_keys_strided():
    """Rows without keys give dQ = 0, key blocks no row reaches give dK = dV = 0; inputs
    are strided views of one packed buffer."""
    torch = torch_cuda()
    rng = np.random.default_rng(9)
    bt, n, h, d, b = 2, 256, 2, 64, 32
    packed = bf16_normal_bits(rng, (bt, n, 3, h, d), 0.5)
    t = to_dev(packed)
    q, k, v = t[:, :, 0], t[:, :, 1], t[:, :, 2]
    dob = bf16_normal_bits(rng, (bt, n, h, d), 0.5)
    do = to_dev(dob)
    nb = n // b
    rows = [[0], [], [0, 1], [2], [], [1, 3, 5], [6], [0, 7]]     # block 4 is never a key
    rp = np.zeros((bt, nb + 1), dtype=np.int32)
    cols = []
    for s in range(bt):
        rp[s, 0] = len(cols)
        for I, row in enumerate(rows):
            cols += row
            rp[s, I + 1] = len(cols)
    ci = np.array(cols, dtype=np.int32)
    rp_d, ci_d = torch.from_numpy(rp).cuda(), torch.from_numpy(ci).cuda()
    o, lse = sa.attn_fwd(q, k, v, rp_d, ci_d, b, 1)
    # dq / dk / dv strided like q / k / v
    gt = torch.empty((bt, n, 3, h, d), dtype=torch.bfloat16, device="cuda")
    dq, dk, dv = gt[:, :, 0], gt[:, :, 1], gt[:, :, 2]
    ws = torch.empty((sa.sa_attn_bwd_workspace_size(bt, n, h, b, bt, ci.size),), dtype=torch.uint8, device="cuda")
    # d_o must share o's strides: o is contiguous, so is do
    sa.sa_attn_bwd(q, k, v, o, do, lse, rp_d, ci_d, b, 1, dq, dk, dv, ws)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    f = bf16_bits_to_f64(packed)
    rq, rk, rv = oracle.attention_csr_backward(f[:, :, 0], f[:, :, 1], f[:, :, 2], bf16_bits_to_f64(dob), rp, ci, b, 1)
    assert_grad_close(bf16_to_f64(dq), rq, "dQ empty rows")
    assert_grad_close(bf16_to_f64(dk), rk, "dK empty rows")
    assert_grad_close(bf16_to_f64(dv), rv, "dV empty rows")
    assert np.all(bf16_to_f64(dq)[:, 32:64] == 0) and np.all(bf16_to_f64(dq)[:, 128:160] == 0)
    assert np.all(bf16_to_f64(dk)[:, 128:160] == 0) and np.all(bf16_to_f64(dv)[:, 128:160] == 0)


def test_backward_is_deterministic():
    torch = torch_cuda()
    n, b = 1024, 64
    rng = np.random.default_rng(8)
    ratios = (rng.integers(20, 80, (1, n // b)) / np.float32(b)).astype(np.float32)
    p = om.MaskParams("topk", b, n, 1, 2, 1, 4)
    qb, kb, vb, dob = (bf16_normal_bits(rng, (1, n, 2, 64), 0.3) for _ in range(4))
    rp_d, ci_d = _mask_on_gpu(p, 1, ratios)
    a = _fwd_bwd(qb, kb, vb, dob, rp_d, ci_d, b, 1)
    c = _fwd_bwd(qb, kb, vb, dob, rp_d, ci_d, b, 1)
    for x, y in zip(a, c):
        assert torch.equal(x, y)


# ---------------------------------------------------------------- full-size workload, sampled rows

def test_bytelm_topk_8k_sampled_and_invariants():
    torch = torch_cuda()
    cfg = workload("bytelm_topk_8k")
    data = byte_stream(cfg)
    b, n, bt, h = cfg["block"], cfg["n_tokens"], cfg["batch"], cfg["heads"]
    p = om.MaskParams("topk", b, n, 1, cfg["window_blocks"], cfg["global_blocks"], cfg["topk"])
    qb, kb, vb = qkv_bits(cfg)
    dob = bf16_normal_bits(np.random.default_rng(77), qb.shape, cfg["std"])
    rp_d, ci_d = _mask_on_gpu(p, bt, sa.sa_block_ratios(data, b))
    dq, dk, dv = _fwd_bwd(qb, kb, vb, dob, rp_d, ci_d, b, 1)
    dq_np, dk_np, dv_np = bf16_to_f64(dq), bf16_to_f64(dk), bf16_to_f64(dv)
    assert np.all(np.isfinite(dq_np)) and np.all(np.isfinite(dk_np)) and np.all(np.isfinite(dv_np))
    rp_o, ci_o = om.build_csr(p, oracle.block_ratios(data, b), bt)
    rng = np.random.default_rng(1)
    smp = [(int(rng.integers(bt)), int(rng.integers(n)), int(rng.integers(h))) for _ in range(24)]
    smp += [(0, 0, 0), (3, n - 1, 11), (1, 4095, 5)]
    ref = oracle.attention_rows_dq(qb, kb, vb, dob, rp_o, ci_o, b, 1, smp, convert=bf16_bits_to_f64)
    got = np.stack([dq_np[s, i, hh] for s, i, hh in smp])
    assert_grad_close(got, ref, "dQ sampled 8K")
    smp_kv = [(int(rng.integers(bt)), int(rng.integers(64, n)), int(rng.integers(h))) for _ in range(6)]
    smp_kv += [(2, n - 1, 4), (1, 100, 7)]
    rk, rv = oracle.attention_rows_dkdv(qb, kb, vb, dob, rp_o, ci_o, b, 1, smp_kv, convert=bf16_bits_to_f64)
    assert_grad_close(np.stack([dk_np[s, j, hk] for s, j, hk in smp_kv]), rk, "dK sampled 8K")
    assert_grad_close(np.stack([dv_np[s, j, hk] for s, j, hk in smp_kv]), rv, "dV sampled 8K")
    # invariants of the exact gradients at full size: sum_j dK_j = 0, sum_j dV_j = sum_i dO_i
    do_f = bf16_bits_to_f64(dob)
    sum_dv = dv_np.sum(axis=1)
    want_dv = do_f.sum(axis=1)
    assert np.abs(sum_dv - want_dv).max() <= 2e-2 * np.abs(want_dv).max()
    assert np.abs(dk_np.sum(axis=1)).max() <= 2e-2 * np.abs(dk_np).max() * np.sqrt(n)


# ---------------------------------------------------------------- head groups

@pytest.mark.parametrize("b,d,causal", [(128, 64, 1), (64, 64, 0), (32, 128, 1)])
def test_head_group_backward(b, d, causal):
    """The page's 6/3/3 split with 3 KV heads (KV groups straddle head groups)."""
    n, bt, h, hkv = 1024, 2, 12, 3
    rng = np.random.default_rng(b + d + causal)
    ratios = (rng.integers(20, 90, (bt, n // b)) / np.float32(b)).astype(np.float32)
    comps = oracle.cas_head_components(h)
    parts = sorted(set(comps))
    head_mask = [parts.index(c) for c in comps]
    qb = bf16_normal_bits(rng, (bt, n, h, d), 0.5)
    kb, vb = (bf16_normal_bits(rng, (bt, n, hkv, d), 0.25) for _ in range(2))
    dob = bf16_normal_bits(rng, (bt, n, h, d), 0.25)
    csrs_d, csrs_o = [], []
    for c in parts:
        p = om.MaskParams("literal_mean", b, n, causal, 1, components=c)
        csrs_d.append(_mask_on_gpu(p, bt, ratios))
        csrs_o.append(om.build_csr(p, ratios, bt))
    torch = torch_cuda()
    q, k, v, do = (to_dev(x) for x in (qb, kb, vb, dob))
    o, lse = sa.attn_fwd_heads(q, k, v, csrs_d, head_mask, b, causal)
    dq, dk, dv = sa.attn_bwd_heads(q, k, v, o, lse, do, csrs_d, head_mask, b, causal)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    f = bf16_bits_to_f64
    rq, rk, rv = oracle.attention_csr_backward_heads(f(qb), f(kb), f(vb), f(dob), csrs_o, head_mask, b, causal)
    what = f"head groups b={b} d={d} causal={causal}"
    assert_grad_close(bf16_to_f64(dq), rq, "dQ " + what)
    assert_grad_close(bf16_to_f64(dk), rk, "dK " + what)
    assert_grad_close(bf16_to_f64(dv), rv, "dV " + what)
