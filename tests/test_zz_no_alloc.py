"""The backward entry point that allocates nothing (sa_attn_bwd_noalloc).

Some callers cannot allocate device memory when they run the backward: a plugin whose host
application owns every allocation, a service that allocates only at start-up, or a caller
that cannot afford the device synchronisation cudaMalloc implies. sa_attn_bwd_noalloc keeps
its scratch in a fixed array inside the library instead of a caller workspace. These tests
call it through the C ABI and compare it with sa_attn_bwd, which takes a caller workspace.

The file is named so that pytest collects it last: a run that stops at the first failure
has then already run every other test.
"""
import numpy as np
import pytest

import content_adaptive_sparse_gb300 as sa
import oracle
from oracle import masks as om
from workloads import bf16_bits_to_f64, bf16_normal_bits
from gpu_helpers import assert_grad_close, bf16_to_f64, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


def _case(seed, n, b, bt, h, hkv, d, w, g, k):
    """Inputs, the GPU CSR and the forward's outputs of one top-k case."""
    torch = torch_cuda()
    rng = np.random.default_rng(seed)
    ratios = (rng.integers(20, 80, (bt, n // b)) / np.float32(b)).astype(np.float32)
    p = om.MaskParams("topk", b, n, 1, w, g, k)
    prm = sa.mask_params("topk", b, n, bt, 1, w, g, k)
    rp_d, ci_d = sa.build_mask(prm, torch.from_numpy(ratios).cuda())
    qb = bf16_normal_bits(rng, (bt, n, h, d), 0.3)
    kb, vb = (bf16_normal_bits(rng, (bt, n, hkv, d), 0.3) for _ in range(2))
    dob = bf16_normal_bits(rng, (bt, n, h, d), 0.3)
    q, k_, v, do = (to_dev(x) for x in (qb, kb, vb, dob))
    o, lse = sa.attn_fwd(q, k_, v, rp_d, ci_d, b, 1)
    return dict(p=p, ratios=ratios, bits=(qb, kb, vb, dob), dev=(q, k_, v, do, o, lse), csr=(rp_d, ci_d), b=b)


def test_noalloc_matches_workspace_call_on_two_calls_in_a_row():
    """Two calls in a row on different shapes and masks (the second with fewer CSR entries
    than the first, so stale scratch from the first call would show): each equals the
    workspace call within the gradient tolerance, and the oracle too."""
    torch = torch_cuda()
    cases = [_case(31, 1024, 64, 2, 4, 2, 64, 2, 1, 3), _case(32, 768, 32, 1, 3, 3, 32, 3, 1, 1)]
    for c in cases:
        q, k, v, do, o, lse = c["dev"]
        rp_d, ci_d = c["csr"]
        dq1, dk1, dv1 = sa.attn_bwd(q, k, v, o, lse, do, rp_d, ci_d, c["b"], 1)
        dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        sa.sa_attn_bwd_noalloc(q, k, v, o, do, lse, rp_d, ci_d, c["b"], 1, dq2, dk2, dv2)
        torch.cuda.synchronize()
        assert sa.sa_device_status() == 0
        for name, x, y in (("dQ", dq2, dq1), ("dK", dk2, dk1), ("dV", dv2, dv1)):
            assert_grad_close(bf16_to_f64(x), bf16_to_f64(y), f"{name} noalloc vs workspace call")
        f = bf16_bits_to_f64
        qb, kb, vb, dob = c["bits"]
        rp_o, ci_o = om.build_csr(c["p"], c["ratios"], qb.shape[0])
        rq, rk, rv = oracle.attention_csr_backward(f(qb), f(kb), f(vb), f(dob), rp_o, ci_o, c["b"], 1)
        assert_grad_close(bf16_to_f64(dq2), rq, "dQ noalloc")
        assert_grad_close(bf16_to_f64(dk2), rk, "dK noalloc")
        assert_grad_close(bf16_to_f64(dv2), rv, "dV noalloc")


def test_noalloc_refuses_shapes_beyond_its_scratch():
    """A shape whose scratch exceeds the library's 16 MiB is refused before any launch."""
    torch = torch_cuda()
    c = _case(33, 1024, 64, 1, 2, 2, 64, 2, 1, 3)
    q, k, v, do, o, lse = c["dev"]
    rp_d, ci_d = c["csr"]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    with pytest.raises(sa.SAError) as e:
        sa.sa_attn_bwd_noalloc(q, k, v, o, do, lse, rp_d, ci_d, c["b"], 1, dq, dk, dv, col_capacity=8 << 20)
    assert e.value.code == -3
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0


def test_noalloc_short_col_capacity_is_reported_by_device_status():
    """A col_capacity below the CSR's real entry count is only seen on the device: the
    transposed lists are clamped to it and sa_device_status reports SA_ERR_CAPACITY."""
    torch = torch_cuda()
    c = _case(34, 1024, 64, 1, 2, 2, 64, 2, 1, 3)
    q, k, v, do, o, lse = c["dev"]
    rp_d, ci_d = c["csr"]
    nnz = int(rp_d[0, -1].item())
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    sa.sa_attn_bwd_noalloc(q, k, v, o, do, lse, rp_d, ci_d, c["b"], 1, dq, dk, dv, col_capacity=nnz // 2)
    assert sa.sa_device_status() == -3
    assert sa.sa_device_status() == 0
