"""GPU block-CSR builder vs the oracle: bit-exact row_ptr and col_idx."""
import numpy as np
import pytest

import content_adaptive_sparse_gb300 as sa
import oracle
from oracle import masks as om
from workloads import byte_stream, bytes_zipf_text, workload
from gpu_helpers import torch_cuda

pytestmark = pytest.mark.gpu


def _gpu_csr(p: om.MaskParams, batch: int, ratios=None):
    torch = torch_cuda()
    mode = {"topk": 0, "bigbird": 1, "full": 2, "literal_mean": 3}[p.mode]
    prm = sa.mask_params(mode, p.block, p.n_tokens, batch, p.causal, p.window_blocks, p.global_blocks, p.topk,
                         p.random_blocks, p.seed, p.components)
    r_dev = None if ratios is None else torch.from_numpy(np.ascontiguousarray(ratios)).cuda()
    rp, ci = sa.build_mask(prm, r_dev)
    torch.cuda.synchronize()
    return rp.cpu().numpy(), ci.cpu().numpy()


def _compare(p, batch, ratios_gpu, ratios_oracle):
    rp_g, ci_g = _gpu_csr(p, batch, ratios_gpu)
    rp_o, ci_o = om.build_csr(p, ratios_oracle, batch)
    assert np.array_equal(rp_g, rp_o)
    assert np.array_equal(ci_g[:len(ci_o)], ci_o)


def _topk_case(name, **over):
    cfg = workload(name, **over)
    data = byte_stream(cfg)
    p = om.MaskParams("topk", cfg["block"], cfg["n_tokens"], 1, cfg["window_blocks"], cfg["global_blocks"],
                      cfg["topk"])
    # each side computes its own ratios (library zlib vs oracle zlib)
    return p, cfg["batch"], sa.sa_block_ratios(data, cfg["block"]), oracle.block_ratios(data, cfg["block"])


@pytest.mark.parametrize("name,over", [
    ("tiny_topk", {}),
    ("bytelm_topk_8k", {}),
    ("long_topk_64k", {"topk": 16}),
    ("long_topk_64k", {"topk": 64}),
    ("long_topk_64k", {"topk": 256}),
])
def test_topk_workloads(name, over):
    p, batch, rg, ro = _topk_case(name, **over)
    _compare(p, batch, rg, ro)


@pytest.mark.parametrize("n", [4096, 16384])
def test_bigbird_workloads(n):
    cfg = workload("bigbird_16k" if n == 16384 else "bigbird_4k")
    b = cfg["block"]
    p = om.MaskParams("bigbird", b, n, 0, cfg["window_tokens"] // b, cfg["global_tokens"] // b, 0,
                      cfg["random_tokens"] // b, cfg["seed"])
    _compare(p, 2, None, None)


def test_full_16k():
    _compare(om.MaskParams("full", 128, 16384, 1), 1, None, None)
    _compare(om.MaskParams("full", 64, 4096, 0), 2, None, None)


@pytest.mark.parametrize("causal", [1, 0])
@pytest.mark.parametrize("b,w", [(128, 1), (64, 2), (32, 0)])
def test_literal_mean(causal, b, w):
    n = 8192
    data = np.stack([bytes_zipf_text(100 + s, n) for s in range(3)])
    p = om.MaskParams("literal_mean", b, n, causal, w)
    _compare(p, 3, sa.sa_block_ratios(data, b), oracle.block_ratios(data, b))


@pytest.mark.parametrize("causal", [1, 0])
def test_literal_mean_long_sequences(causal):
    """1280 blocks per sequence (more than the 1024 whose literal prefixes the CTAs keep in
    shared memory for the entry counts of earlier sequences), three sequences: the CTAs of later
    sequences derive the earlier ones' counts one after another."""
    n, b = 40960, 32
    data = np.stack([bytes_zipf_text(300 + s, n) for s in range(3)])
    p = om.MaskParams("literal_mean", b, n, causal, 1)
    _compare(p, 3, sa.sa_block_ratios(data, b), oracle.block_ratios(data, b))


@pytest.mark.parametrize("components", [1, 2])
@pytest.mark.parametrize("causal", [1, 0])
def test_literal_mean_components(causal, components):
    n, b, w = 8192, 64, 2
    data = np.stack([bytes_zipf_text(200 + s, n) for s in range(2)])
    p = om.MaskParams("literal_mean", b, n, causal, w, components=components)
    _compare(p, 2, sa.sa_block_ratios(data, b), oracle.block_ratios(data, b))


def test_random_parameter_sweep():
    rng = np.random.default_rng(2024)
    for trial in range(40):
        b = int(rng.choice([32, 64, 128]))
        nb = int(rng.integers(1, 70))
        n = nb * b
        mode = ["topk", "bigbird", "full", "literal_mean"][trial % 4]
        batch = int(rng.integers(1, 4))
        ratios = (rng.integers(20, 60, (batch, nb)) / np.float32(b)).astype(np.float32)  # many ties
        if mode == "topk":
            p = om.MaskParams("topk", b, n, 1, int(rng.integers(0, 6)), int(rng.integers(0, 3)),
                              int(rng.integers(0, 12)))
        elif mode == "bigbird":
            p = om.MaskParams("bigbird", b, n, 0, int(rng.integers(0, 10)), int(rng.integers(0, 3)), 0,
                              int(rng.integers(0, 5)), int(rng.integers(0, 2**63)))
        elif mode == "full":
            p = om.MaskParams("full", b, n, int(rng.integers(0, 2)))
        else:
            p = om.MaskParams("literal_mean", b, n, int(rng.integers(0, 2)), int(rng.integers(0, 4)),
                              components=int(rng.integers(0, 4)))
        needs = mode in ("topk", "literal_mean")
        _compare(p, batch, ratios if needs else None, ratios if needs else None)


def test_mask_is_deterministic():
    p, batch, rg, _ = _topk_case("bytelm_topk_8k")
    a = _gpu_csr(p, batch, rg)
    b = _gpu_csr(p, batch, rg)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("name,mode", [("bytelm_topk_8k", "topk"), ("cas_heads_8k", "literal_mean")])
def test_mask_from_host_bytes(name, mode):
    """sa_build_mask_from_bytes (host ratios, their upload and the mask build in one call)
    writes the oracle's CSR bit for bit, and the host ratios it returns equal the oracle's."""
    torch = torch_cuda()
    cfg = workload(name)
    data = byte_stream(cfg)
    b, n, bt = cfg["block"], cfg["n_tokens"], cfg["batch"]
    level = cfg.get("zlib_level", 6)
    if mode == "topk":
        p = om.MaskParams("topk", b, n, 1, cfg["window_blocks"], cfg["global_blocks"], cfg["topk"])
    else:
        p = om.MaskParams("literal_mean", b, n, 1, cfg["window_blocks"])
    prm = sa.mask_params(mode, b, n, bt, p.causal, p.window_blocks, p.global_blocks, p.topk, 0, 0, 0)
    cap = sa.sa_mask_nnz_bound(prm)
    h_ratio = torch.empty((bt, n // b), dtype=torch.float32).pin_memory()
    d_ratio = torch.empty((bt, n // b), dtype=torch.float32, device="cuda")
    rp = torch.empty((bt, n // b + 1), dtype=torch.int32, device="cuda")
    ci = torch.empty((cap,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    sa.sa_build_mask_from_bytes(prm, data, h_ratio, d_ratio, rp, ci, level=level, stream=stream)
    stream.synchronize()
    assert sa.sa_device_status() == 0
    r_ora = oracle.block_ratios(data, b, level)
    assert np.array_equal(h_ratio.numpy(), r_ora)
    assert np.array_equal(d_ratio.cpu().numpy(), r_ora)
    rp_o, ci_o = om.build_csr(p, r_ora, bt)
    assert np.array_equal(rp.cpu().numpy(), rp_o)
    assert np.array_equal(ci.cpu().numpy()[:len(ci_o)], ci_o)
