"""Host-side checks of libsa.so that need no GPU: the library loads, exports every
symbol include/sa_api.h declares, and its host-only entry points (size bound,
Fibonacci offsets, zlib ratios, argument validation) agree with the oracle."""
import ctypes
import math
import os
import re
from fractions import Fraction

import numpy as np
import pytest

import content_adaptive_sparse_gb300 as sa
import oracle
from oracle import masks as om
from workloads import byte_stream, bytes_phrase_random, workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    sa.build_library()
    return sa.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "sa_api.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(sa_\w+)\s*\(", text, flags=re.M)))


def test_header_symbols_exported(lib):
    names = _declared_functions()
    assert {"sa_build_mask", "sa_attn_fwd", "sa_attn_fwd_heads", "sa_offset_attn_fwd", "sa_pow2_offsets",
            "sa_offset_attn_fwd_list",
            "sa_attn_bwd", "sa_attn_bwd_workspace_size", "sa_attn_bwd_noalloc", "sa_offset_attn_interp_fwd",
            "sa_attn_bwd_heads", "sa_selftest_bounded_wait", "sa_attn_fwd_workspace_size", "sa_build_mask_from_bytes",
            "sa_layer_alpha", "sa_fib_offsets", "sa_block_ratios",
            "sa_mask_nnz_bound", "sa_device_status", "sa_status_string", "sa_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert lib.sa_version() == 1
    assert lib.sa_status_string(-3) == b"SA_ERR_CAPACITY"


@pytest.mark.parametrize("name", ["tiny_topk", "bytelm_topk_8k", "long_topk_64k"])
def test_block_ratios_match_oracle(lib, name):
    cfg = workload(name, batch=1) if name == "long_topk_64k" else workload(name)
    data = byte_stream(cfg)
    r_lib = sa.sa_block_ratios(data, cfg["block"], 6)
    r_ora = oracle.block_ratios(data, cfg["block"], 6)
    assert r_lib.dtype == np.float32 and np.array_equal(r_lib, r_ora)


@pytest.mark.parametrize("block", [32, 64, 128])
def test_block_ratios_every_level_and_content(lib, block):
    """Each worker reuses one deflate stream across its blocks: every level, and neighbouring
    blocks of very different content (zeros, random bytes, short periods, text-like phrases),
    must give the lengths of independent one-shot compressions."""
    rng = np.random.default_rng(block)
    n_blocks = 48
    parts = []
    for i in range(n_blocks):
        kind = i % 4
        if kind == 0:
            parts.append(np.zeros(block, np.uint8))
        elif kind == 1:
            parts.append(rng.integers(0, 256, block, dtype=np.uint8))
        elif kind == 2:
            period = 1 + i % 7
            parts.append(np.resize(rng.integers(0, 256, period, dtype=np.uint8), block))
        else:
            parts.append(bytes_phrase_random(i, block))
    data = np.concatenate(parts).reshape(2, -1)
    for level in range(10):
        r_lib = sa.sa_block_ratios(data, block, level, n_threads=3)
        r_ora = oracle.block_ratios(data, block, level)
        assert np.array_equal(r_lib, r_ora), level


def _ratios_in_child(data):
    return sa.sa_block_ratios(data, 64, 6)


@pytest.mark.filterwarnings("ignore:This process .* is multi-threaded:DeprecationWarning")
def test_ratio_workers_after_fork(lib):
    """The ratio pass keeps host worker threads between calls; a child forked after the parent
    used them has none of them and must build its own (same ratios, no hang)."""
    import multiprocessing
    data = np.stack([bytes_phrase_random(s, 8192) for s in range(2)])
    parent = sa.sa_block_ratios(data, 64, 6)          # the parent's workers exist from here on
    with multiprocessing.get_context("fork").Pool(1) as pool:
        child = pool.apply_async(_ratios_in_child, (data,)).get(timeout=120)
    assert np.array_equal(parent, child)
    assert np.array_equal(parent, oracle.block_ratios(data, 64, 6))


def test_fib_offsets_match_oracle(lib):
    for lo, hi in (((1, 2), (2, 1)), ((1, 2), (3, 2))):
        for alpha in oracle.alpha_schedule(16, lo, hi):
            for W in (6, 8, 10, 12):
                for n in (2048, 8192):
                    want = [d for d in oracle.fib_offsets(alpha, oracle.fib_rungs(15)) if W < d < n]
                    got = sa.sa_fib_offsets(alpha.numerator, alpha.denominator, 15, W, n)
                    assert got == want
                    want_all = [d for d in oracle.fib_offsets(alpha, oracle.fib_rungs_upto(n)) if W < d < n]
                    assert sa.sa_fib_offsets(alpha.numerator, alpha.denominator, 0, W, n) == want_all


def test_pow2_offsets_and_layer_alpha_match_oracle(lib):
    for lo, hi in (((1, 2), (2, 1)), ((1, 2), (3, 2))):
        for stride in (1, 7, 3):
            want_alphas = oracle.alpha_schedule(16, lo, hi, stride=stride)
            for l in range(16):
                num, den = sa.sa_layer_alpha(l, 16, lo, hi, stride)
                assert Fraction(num, den) == want_alphas[l] and math.gcd(num, den) == 1
        for alpha in oracle.alpha_schedule(16, lo, hi):
            for W in (6, 8, 12):
                for n in (2048, 8192):
                    want = [d for d in oracle.fib_offsets(alpha, oracle.pow2_rungs(11)) if W < d < n]
                    assert sa.sa_pow2_offsets(alpha.numerator, alpha.denominator, 11, W, n) == want
                    want_all = [d for d in oracle.fib_offsets(alpha, oracle.pow2_rungs_upto(n)) if W < d < n]
                    assert sa.sa_pow2_offsets(alpha.numerator, alpha.denominator, 0, W, n) == want_all
    # a stride sharing a factor with the layer count is refused
    num, den = ctypes.c_int32(0), ctypes.c_int32(0)
    assert lib.sa_layer_alpha(0, 16, 1, 2, 3, 2, 4, ctypes.byref(num), ctypes.byref(den)) == -1


def _params(p: om.MaskParams, batch: int):
    mode = {"topk": 0, "bigbird": 1, "full": 2, "literal_mean": 3}[p.mode]
    return sa.mask_params(mode, p.block, p.n_tokens, batch, p.causal, p.window_blocks, p.global_blocks, p.topk,
                          p.random_blocks, p.seed, p.components)


@pytest.mark.parametrize("p", [
    om.MaskParams("literal_mean", 64, 4096, 1, 3, components=1),
    om.MaskParams("literal_mean", 32, 1024, 0, 2, components=1),
    om.MaskParams("topk", 64, 8192, 1, 4, 1, 16),
    om.MaskParams("topk", 128, 65536, 1, 4, 1, 256),
    om.MaskParams("bigbird", 32, 16384, 0, 8, 1, 0, 1, 45),
    om.MaskParams("bigbird", 32, 1024, 0, 5, 2, 0, 3, 7),
    om.MaskParams("full", 128, 16384, 1),
    om.MaskParams("full", 32, 512, 0),
])
def test_nnz_bound_exact_for_data_independent_modes(lib, p):
    rng = np.random.default_rng(0)
    ratios = rng.random((2, p.nb)).astype(np.float32)
    _, ci = om.build_csr(p, ratios if p.mode in ("topk", "literal_mean") else None, 2)
    assert sa.sa_mask_nnz_bound(_params(p, 2)) == len(ci)


def test_argument_validation_before_any_launch(lib):
    bad = [
        sa.mask_params(0, 64, 8192, 1, causal=0, window_blocks=4),        # topk must be causal
        sa.mask_params(1, 32, 1024, 1, causal=1, window_blocks=8),        # bigbird bidirectional only
        sa.mask_params(0, 64, 1000, 1, window_blocks=4),                   # N % b != 0
        sa.mask_params(3, 64, 1024, 1, global_blocks=1),                   # literal_mean has no globals
        sa.mask_params(0, 1, 8192, 1),                                     # nb > 4096
        sa.mask_params(3, 64, 1024, 1, components=4),                      # unknown component bit
        sa.mask_params(0, 64, 8192, 1, window_blocks=4, components=1),     # components: literal_mean only
    ]
    expect = [-2, -2, -1, -2, -2, -1, -1]
    for prm, code in zip(bad, expect):
        out = ctypes.c_int64(0)
        assert lib.sa_mask_nnz_bound(ctypes.byref(prm), ctypes.byref(out)) == code
    ok = sa.mask_params(0, 64, 8192, 1, window_blocks=4, global_blocks=1, topk=16)
    # capacity short -> SA_ERR_CAPACITY, decided on the host before touching the device
    dummy = ctypes.c_void_p(16)
    assert lib.sa_build_mask(ctypes.byref(ok), dummy, dummy, dummy, 10, None) == -3
    I3 = ctypes.c_int64 * 3
    s = I3(8192 * 12 * 64, 12 * 64, 64)
    p16 = ctypes.c_void_p(256)
    # head_dim 48 unsupported, heads % kv_heads != 0 invalid, misaligned pointer unsupported
    assert lib.sa_attn_fwd(p16, p16, p16, s, s, s, 1, 8192, 12, 12, 48, 64, 1, p16, p16, 0,
                           ctypes.c_float(0.125), p16, p16, p16, 4096, None) == -2
    assert lib.sa_attn_fwd(p16, p16, p16, s, s, s, 1, 8192, 12, 5, 64, 64, 1, p16, p16, 0,
                           ctypes.c_float(0.125), p16, p16, p16, 4096, None) == -1
    assert lib.sa_attn_fwd(ctypes.c_void_p(258), p16, p16, s, s, s, 1, 8192, 12, 12, 64, 64, 1, p16, p16, 0,
                           ctypes.c_float(0.125), p16, p16, p16, 4096, None) == -2
    # the workspace: required, 256-byte aligned, at least 256 bytes
    assert lib.sa_attn_fwd(p16, p16, p16, s, s, s, 1, 8192, 12, 12, 64, 64, 1, p16, p16, 0,
                           ctypes.c_float(0.125), p16, p16, None, 4096, None) == -1
    assert lib.sa_attn_fwd(p16, p16, p16, s, s, s, 1, 8192, 12, 12, 64, 64, 1, p16, p16, 0,
                           ctypes.c_float(0.125), p16, p16, ctypes.c_void_p(272), 4096, None) == -2
    assert lib.sa_attn_fwd(p16, p16, p16, s, s, s, 1, 8192, 12, 12, 64, 64, 1, p16, p16, 0,
                           ctypes.c_float(0.125), p16, p16, p16, 128, None) == -3
    nbytes = ctypes.c_size_t(0)
    assert lib.sa_attn_fwd_workspace_size(4, 8192, 12, 64, 64, 4, 1, ctypes.byref(nbytes)) == 0
    # counter + plan (3072 items, 256 query-tile groups) + 608 slots of 128 x 65 floats
    assert 608 * 128 * 65 * 4 < nbytes.value < 608 * 128 * 65 * 4 + 3072 * 8 + 608 * 24 + 256 * 16
    assert lib.sa_attn_fwd_workspace_size(4, 8192, 12, 48, 64, 4, 1, ctypes.byref(nbytes)) == -2
    # per-head CSRs: head index out of range invalid, too many CSRs unsupported
    P2 = ctypes.c_void_p * 2
    rps, cis = P2(256, 512), P2(256, 512)
    hm = (ctypes.c_int32 * 12)(*([0] * 11 + [2]))
    assert lib.sa_attn_fwd_heads(p16, p16, p16, s, s, s, 1, 8192, 12, 12, 64, 64, 1, 2, rps, cis, hm, 0,
                                 ctypes.c_float(0.125), p16, p16, p16, 4096, None) == -1
    P9 = ctypes.c_void_p * 9
    rp9 = P9(*([256] * 9))
    assert lib.sa_attn_fwd_heads(p16, p16, p16, s, s, s, 1, 8192, 12, 12, 64, 64, 1, 9, rp9, rp9, hm, 0,
                                 ctypes.c_float(0.125), p16, p16, p16, 4096, None) == -2
    # interpolated gather: alpha must be positive, head_dim 32, 64 or 128
    assert lib.sa_offset_attn_interp_fwd(p16, p16, p16, s, s, s, 1, 8192, 8, 8, 64, 8, ctypes.c_double(-0.5), 15, 0,
                                         ctypes.c_float(0.125), p16, p16, None) == -1
    assert lib.sa_offset_attn_interp_fwd(p16, p16, p16, s, s, s, 1, 8192, 8, 8, 96, 8, ctypes.c_double(0.8), 15, 0,
                                         ctypes.c_float(0.125), p16, p16, None) == -2
    offs = (ctypes.c_int32 * 2)(5, 9)        # offset inside the window -> invalid
    assert lib.sa_offset_attn_fwd_list(p16, p16, p16, s, s, s, 1, 8192, 8, 8, 64, 8, offs, 2,
                                       ctypes.c_float(0.125), p16, p16, None) == -1
    # the page's parameters: alpha must be a positive fraction; head_dim 32, 64 or 128
    assert lib.sa_offset_attn_fwd(p16, p16, p16, s, s, s, 1, 8192, 8, 8, 64, 8, 1, 0, 15,
                                  ctypes.c_float(0.125), p16, p16, None) == -1
    assert lib.sa_offset_attn_fwd(p16, p16, p16, s, s, s, 1, 8192, 8, 8, 64, 8, -3, 2, 15,
                                  ctypes.c_float(0.125), p16, p16, None) == -1
    assert lib.sa_offset_attn_fwd(p16, p16, p16, s, s, s, 1, 8192, 8, 8, 96, 8, 1, 1, 15,
                                  ctypes.c_float(0.125), p16, p16, None) == -2


def test_compute_entry_points_refuse_without_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    ok = sa.mask_params(0, 64, 8192, 1, window_blocks=4, global_blocks=1, topk=16)
    dummy = ctypes.c_void_p(16)
    assert lib.sa_build_mask(ctypes.byref(ok), dummy, dummy, dummy, 10**6, None) == -4   # SA_ERR_CUDA


def test_bwd_noalloc_capacity_is_checked_on_the_host(lib):
    """The no-allocation backward refuses shapes whose scratch exceeds its 16 MiB before
    touching a device; shapes that fit get as far as the device check."""
    I3 = ctypes.c_int64 * 3
    s = I3(8192 * 12 * 64, 12 * 64, 64)
    p16 = ctypes.c_void_p(256)
    args = lambda batch, cap: (p16, p16, p16, p16, p16, p16, s, s, s, batch, 8192, 12, 12, 64, 64, 1, p16, p16,
                               ctypes.c_int64(cap), 0, ctypes.c_float(0.125), p16, p16, p16, None)
    assert lib.sa_attn_bwd_noalloc(*args(64, 10**5)) == -3        # 64 x 12 x 8192 x 4 B of D alone > 16 MiB
    ws = ctypes.c_size_t(0)
    assert lib.sa_attn_bwd_workspace_size(4, 8192, 12, 64, 4, 10**4, ctypes.byref(ws)) == 0
    assert ws.value < 16 << 20
    import torch
    if not torch.cuda.is_available():
        assert lib.sa_attn_bwd_noalloc(*args(4, 10**4)) == -4     # fits; no device here


def test_ratio_threads_are_deterministic(lib):
    data = np.stack([bytes_phrase_random(s, 4096) for s in range(3)])
    a = sa.sa_block_ratios(data, 32, 6, n_threads=1)
    b = sa.sa_block_ratios(data, 32, 6, n_threads=7)
    assert np.array_equal(a, b)
