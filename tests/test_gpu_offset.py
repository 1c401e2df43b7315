"""Window-plus-Fibonacci-offset attention kernel vs the float64 oracle."""
from fractions import Fraction

import numpy as np
import pytest

import content_adaptive_sparse_gb300 as sa
import oracle
from workloads import bf16_bits_to_f64, bf16_normal_bits, qkv_bits, workload
from gpu_helpers import LSE_MAX_ABS, O_MAX_ABS, assert_attention_close, bf16_to_f64, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


def _run(bt, n, h, hkv, window, alpha: Fraction, n_rungs=15, seed=0, qmul=1.0, ladder="fib", d=64):
    torch = torch_cuda()
    rng = np.random.default_rng(seed)
    qb = bf16_normal_bits(rng, (bt, n, h, d), 0.125 * qmul)
    kb = bf16_normal_bits(rng, (bt, n, hkv, d), 0.125)
    vb = bf16_normal_bits(rng, (bt, n, hkv, d), 0.125)
    if ladder == "fib":
        offs = sa.sa_fib_offsets(alpha.numerator, alpha.denominator, n_rungs, window, n)
        rungs = oracle.fib_rungs(n_rungs) if n_rungs else oracle.fib_rungs_upto(n)
    else:
        offs = sa.sa_pow2_offsets(alpha.numerator, alpha.denominator, n_rungs, window, n)
        rungs = oracle.pow2_rungs(n_rungs) if n_rungs else oracle.pow2_rungs_upto(n)
    assert offs == [d for d in oracle.fib_offsets(alpha, rungs) if window < d < n]
    o, lse = sa.offset_attn_fwd(to_dev(qb), to_dev(kb), to_dev(vb), window, offs)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    o_ref, lse_ref = oracle.attention_offsets(bf16_bits_to_f64(qb), bf16_bits_to_f64(kb), bf16_bits_to_f64(vb),
                                              window, oracle.fib_offsets(alpha, rungs))
    return assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                                  f"d={d} W={window} alpha={alpha}")


@pytest.mark.parametrize("window", [6, 8, 10, 12])
def test_windows_mid_alpha(window):
    _run(2, 1024, 2, 2, window, Fraction(7, 10), seed=window, qmul=4.0)


@pytest.mark.parametrize("alpha", [Fraction(1, 2), Fraction(1, 1), Fraction(3, 2), Fraction(2, 1)])
def test_alpha_range_gqa(alpha):
    _run(1, 2048, 4, 2, 8, alpha, seed=3)


@pytest.mark.parametrize("layer", [0, 1, 9, 15])
def test_pow2_base_coprime_stagger(layer):
    """Power-of-2 control rungs with the coprime-staggered alpha of a layer."""
    num, den = sa.sa_layer_alpha(layer, 16, (1, 2), (3, 2), 7)
    alpha = Fraction(num, den)
    assert alpha == oracle.alpha_schedule(16, (1, 2), (3, 2), stride=7)[layer]
    _run(1, 2048, 4, 2, 8, alpha, n_rungs=11, seed=20 + layer, qmul=3.0, ladder="pow2")


def test_all_rungs_up_to_n_and_ragged_tail():
    _run(1, 1000, 2, 1, 8, Fraction(13, 10), n_rungs=0, seed=4, qmul=2.0)


def test_small_edge_cases():
    _run(1, 130, 1, 1, 0, Fraction(1, 1), seed=5)          # window 0: self plus offsets
    _run(1, 64, 1, 1, 64, Fraction(1, 2), seed=6)          # window covers everything: dense causal


@pytest.mark.parametrize("window,hkv", [(6, 2), (8, 8), (8, 2), (10, 2), (12, 8), (12, 2)])
def test_fib_2k_full_layers(window, hkv):
    """The 2048-token Fibonacci workload (8 sequences, 8 heads of 64) in full, through the
    entry point that takes the page's parameters (W, alpha as a fraction, 15 rungs), for
    the first, a middle and the last layer of the 0.5 -> 2.0 ramp and of the page's own
    0.5 -> 1.5 ramp ("Depth-Staggered Fibonacci Spacing ...", section 3 "Run matrix": windows
    6 to 12, grouped-query attention with 2 KV heads)."""
    torch = torch_cuda()
    cfg = workload("fib_2k", window=window, kv_heads=hkv)
    for lo, hi in ((cfg["alpha_lo"], cfg["alpha_hi"]), ((1, 2), (3, 2))):
        for layer in (0, 7, 15):
            num, den = sa.sa_layer_alpha(layer, 16, lo, hi)
            alpha = Fraction(num, den)
            assert alpha == oracle.alpha_schedule(16, lo, hi)[layer]
            qb, kb, vb = qkv_bits(cfg, seed_offset=layer)
            o, lse = sa.fib_offset_attn_fwd(to_dev(qb), to_dev(kb), to_dev(vb), window, num, den, 15)
            torch.cuda.synchronize()
            assert sa.sa_device_status() == 0
            f = bf16_bits_to_f64
            o_ref, lse_ref = oracle.attention_offsets(f(qb), f(kb), f(vb), window,
                                                      oracle.fib_offsets(alpha, oracle.fib_rungs(15)))
            assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                                   f"fib 2k W={window} Hkv={hkv} layer {layer} alpha={alpha}")


@pytest.mark.parametrize("window,hkv,layer", [(8, 8, 11), (6, 2, 0), (10, 2, 15), (12, 8, 5)])
def test_fib_8k_whole_tiles(window, hkv, layer):
    """The 8192-token workload (4x the training length): every row of eight 128-query slices
    (the first, the last, others spread over the sequences) for every head."""
    torch = torch_cuda()
    cfg = workload("fib_8k", window=window, kv_heads=hkv)
    qb, kb, vb = qkv_bits(cfg, seed_offset=layer)
    num, den = sa.sa_layer_alpha(layer, 16, cfg["alpha_lo"], cfg["alpha_hi"])
    alpha = Fraction(num, den)
    n, bt, h = cfg["n_tokens"], cfg["batch"], cfg["heads"]
    o, lse = sa.fib_offset_attn_fwd(to_dev(qb), to_dev(kb), to_dev(vb), window, num, den, cfg["n_rungs"])
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    o_np = bf16_to_f64(o)
    lse_np = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o_np)) and np.all(np.isfinite(lse_np))
    slices = [(0, 0), (bt - 1, n - 128), (1, 128), (2, 1024), (3, 4096 - 64), (4, 6000), (5, 8000 - 128),
              (6, 987 - 60)]
    smp = [(s, i, hh) for s, i0 in slices for i in range(i0, i0 + 128) for hh in range(h)]
    o_ref, lse_ref = oracle.attention_offsets(qb, kb, vb, window, oracle.fib_offsets(alpha, oracle.fib_rungs(15)),
                                              samples=smp, convert=bf16_bits_to_f64)
    o_g = np.stack([o_np[s, i, hh] for s, i, hh in smp])
    l_g = np.array([lse_np[s, hh, i] for s, i, hh in smp])
    assert_attention_close(o_g, l_g, o_ref, lse_ref, f"fib_8k W={window} Hkv={hkv} layer {layer}")


def _run_offsets(q64, k64, v64, qd, kd, vd, window, offs, what):
    torch = torch_cuda()
    o, lse = sa.offset_attn_fwd(qd, kd, vd, window, offs)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    o_ref, lse_ref = oracle.attention_offsets(q64, k64, v64, window, offs)
    return assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, what)


@pytest.mark.parametrize("window,offs", [
    (8, [9, 31, 32, 33, 63, 64, 65, 79, 80, 96, 127, 128, 129, 500, 777]),   # both sides of the band limit
    (0, [1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 144, 233, 377, 610]),           # window 0, classic rungs
    (64, [65, 66, 100, 1000]),                                               # widest window
    (3, list(range(4, 68)) ),                                                # 64 offsets, all but 3 in the band
])
def test_explicit_offset_sets(window, offs):
    rng = np.random.default_rng(window + len(offs))
    n = 1100
    qb = bf16_normal_bits(rng, (2, n, 2, 64), 0.5)
    kb = bf16_normal_bits(rng, (2, n, 2, 64), 0.5)
    vb = bf16_normal_bits(rng, (2, n, 2, 64), 0.5)
    _run_offsets(bf16_bits_to_f64(qb), bf16_bits_to_f64(kb), bf16_bits_to_f64(vb), to_dev(qb), to_dev(kb),
                 to_dev(vb), window, offs, f"W={window} offsets={offs[:4]}..")


@pytest.mark.parametrize("d", [32, 64, 128])
def test_packed_strided_inputs(d):
    rng = np.random.default_rng(9 + d)
    bt, n, h = 2, 700, 4
    packed = bf16_normal_bits(rng, (bt, n, 3, h, d), 0.5 * (64 / d) ** 0.5)   # q, k, v interleaved per token
    t = to_dev(packed)
    f = bf16_bits_to_f64(packed)
    _run_offsets(f[:, :, 0], f[:, :, 1], f[:, :, 2], t[:, :, 0], t[:, :, 1], t[:, :, 2], 8,
                 [9, 13, 21, 34, 55, 89, 144, 233, 377, 610], f"packed qkv d={d}")
    # the interpolated gather on the same strided views
    torch = torch_cuda()
    o, lse = sa.offset_attn_interp_fwd(t[:, :, 0], t[:, :, 1], t[:, :, 2], 8, 0.91)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    o_ref, lse_ref = oracle.attention_offsets_interp(f[:, :, 0], f[:, :, 1], f[:, :, 2], 8,
                                                     oracle.interp_rungs(0.91, oracle.fib_rungs(15), 8))
    assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                           f"packed qkv interp d={d}")


# ---------------------------------------------------------------- interpolated gather (continuous alpha)

def _run_interp(bt, n, h, hkv, window, alpha, n_rungs=15, ladder=0, seed=0, qmul=1.0, d=64):
    torch = torch_cuda()
    rng = np.random.default_rng(seed)
    qb = bf16_normal_bits(rng, (bt, n, h, d), 0.125 * qmul)
    kb = bf16_normal_bits(rng, (bt, n, hkv, d), 0.125)
    vb = bf16_normal_bits(rng, (bt, n, hkv, d), 0.125)
    o, lse = sa.offset_attn_interp_fwd(to_dev(qb), to_dev(kb), to_dev(vb), window, alpha, n_rungs, ladder)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    if ladder == 0:
        rungs = oracle.fib_rungs(n_rungs) if n_rungs else oracle.fib_rungs_upto(n)
    else:
        rungs = oracle.pow2_rungs(n_rungs) if n_rungs else oracle.pow2_rungs_upto(n)
    lt = oracle.interp_rungs(alpha, rungs, window)
    o_ref, lse_ref = oracle.attention_offsets_interp(bf16_bits_to_f64(qb), bf16_bits_to_f64(kb),
                                                     bf16_bits_to_f64(vb), window, lt)
    return assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                                  f"interp d={d} W={window} alpha={alpha}")


@pytest.mark.parametrize("alpha", [0.8317, 1.2345, 0.5, 1.5])
def test_interp_alphas_gqa(alpha):
    _run_interp(1, 1000, 4, 2, 8, alpha, seed=int(alpha * 1000), qmul=3.0)


def test_interp_windows_pow2_and_all_rungs():
    _run_interp(2, 520, 2, 2, 0, 0.777, seed=1)                  # window 0: self plus rungs
    _run_interp(1, 700, 2, 1, 12, 1.1, ladder=1, n_rungs=11, seed=2, qmul=2.0)
    _run_interp(1, 900, 2, 2, 6, 0.9, n_rungs=0, seed=3)         # every rung up to N


def test_interp_integer_alpha_matches_integer_offset_kernel():
    """alpha = 1 and 2: the interpolated path and the integer-offset kernel see the same
    key set; both match the oracle, and each other to the combined tolerance."""
    torch = torch_cuda()
    rng = np.random.default_rng(12)
    n = 1024
    qb, kb, vb = (bf16_normal_bits(rng, (1, n, 2, 64), 0.3) for _ in range(3))
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    for alpha in (1, 2):
        o1, l1 = sa.offset_attn_interp_fwd(q, k, v, 8, float(alpha))
        offs = sa.sa_fib_offsets(alpha, 1, 15, 8, n)
        o2, l2 = sa.offset_attn_fwd(q, k, v, 8, offs)
        torch.cuda.synchronize()
        assert (o1.float() - o2.float()).abs().max().item() < 2 * O_MAX_ABS
        assert (l1 - l2).abs().max().item() < 2 * LSE_MAX_ABS


def test_interp_fib_8k_whole_slices():
    torch = torch_cuda()
    cfg = workload("fib_8k", layers=1)
    qb, kb, vb = qkv_bits(cfg)
    alpha = 0.5 + 1.0 / (1.0 + np.exp(-0.37))            # a learned-style alpha in (0.5, 1.5)
    o, lse = sa.offset_attn_interp_fwd(to_dev(qb), to_dev(kb), to_dev(vb), cfg["window"], alpha)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    bt, n, h = cfg["batch"], cfg["n_tokens"], cfg["heads"]
    # every row of eight 128-query slices, every head
    slices = [(0, 0), (bt - 1, n - 128), (3, 1), (5, 987 - 64), (1, 2048), (2, 4000), (4, 6100), (6, 7777)]
    smp = [(s, i, hh) for s, i0 in slices for i in range(i0, min(n, i0 + 128)) for hh in range(h)]
    lt = oracle.interp_rungs(alpha, oracle.fib_rungs(15), cfg["window"])
    o_ref, lse_ref = oracle.attention_offsets_interp(qb, kb, vb, cfg["window"], lt, samples=smp,
                                                     convert=bf16_bits_to_f64)
    o_np = bf16_to_f64(o)
    lse_np = lse.cpu().numpy().astype(np.float64)
    o_g = np.stack([o_np[s, i, hh] for s, i, hh in smp])
    l_g = np.array([lse_np[s, hh, i] for s, i, hh in smp])
    assert_attention_close(o_g, l_g, o_ref, lse_ref, "interp fib 8k")


def test_interp_band_boundary_and_wide_windows():
    """Rungs just inside and just past the 64-row band (floor distance 63 and 64, with and
    without a fractional part), and windows that need three to five 16-key steps."""
    _run_interp(1, 600, 2, 2, 8, 0.99, ladder=1, n_rungs=8, seed=41)      # 64 x 0.99 = 63.36
    _run_interp(1, 600, 2, 2, 8, 1.01, ladder=1, n_rungs=8, seed=42)      # 64.64
    _run_interp(1, 600, 2, 1, 8, 63 / 64, ladder=1, n_rungs=8, seed=43)   # 63.0 and 126.0
    _run_interp(1, 600, 2, 2, 8, 1.0, ladder=1, n_rungs=9, seed=44)       # 64.0, 128.0, 256.0
    _run_interp(1, 777, 2, 2, 40, 0.73, seed=45, qmul=2.0)
    _run_interp(2, 500, 2, 1, 64, 1.3, n_rungs=0, seed=46)


def test_interp_ragged_length_and_tiny_sequences():
    """Lengths that are not multiples of the 16-query warp tile or the 64-query CTA tile, and
    sequences shorter than the first rung."""
    _run_interp(2, 1003, 2, 1, 8, 0.6180, seed=31, qmul=2.0)
    _run_interp(1, 7, 1, 1, 3, 1.7, seed=32)
    _run_interp(1, 1, 1, 1, 0, 0.9, seed=33)


# ---------------------------------------------------------------- head dimensions 32 and 128

@pytest.mark.parametrize("d", [32, 128])
@pytest.mark.parametrize("window,alpha,hkv,n_rungs", [
    (8, Fraction(7, 10), 2, 15),     # GQA, the page's window
    (12, Fraction(3, 2), 1, 15),     # four query heads on one KV head
    (0, Fraction(2, 1), 2, 15),      # self plus offsets: one 16-key band step
    (64, Fraction(1, 2), 2, 15),     # the widest band: five 16-key steps
    (6, Fraction(13, 10), 2, 0),     # every rung up to N
])
def test_head_dims_32_128(d, window, alpha, hkv, n_rungs):
    """1000 tokens: a ragged tail for the 128-query (d <= 64) and 64-query (d = 128) tiles."""
    _run(2, 1000, 4, hkv, window, alpha, n_rungs=n_rungs, seed=100 + window + d, qmul=3.0, d=d)


@pytest.mark.parametrize("d", [32, 128])
def test_head_dims_pow2_and_short(d):
    _run(1, 2048, 4, 2, 8, Fraction(9, 10), n_rungs=11, seed=7 + d, qmul=2.0, ladder="pow2", d=d)
    _run(1, 130, 1, 1, 0, Fraction(1, 1), seed=8 + d, d=d)
    _run(1, 64, 1, 1, 64, Fraction(1, 2), seed=9 + d, d=d)     # dense causal


@pytest.mark.parametrize("d", [32, 128])
def test_interp_head_dims_32_128(d):
    _run_interp(2, 1003, 4, 2, 8, 0.8317, seed=200 + d, qmul=3.0, d=d)
    _run_interp(1, 600, 2, 2, 8, 0.99, ladder=1, n_rungs=8, seed=201 + d, d=d)     # 63.36: band side
    _run_interp(1, 600, 2, 2, 8, 1.01, ladder=1, n_rungs=8, seed=202 + d, d=d)     # 64.64: slab side
    _run_interp(2, 500, 2, 1, 64, 1.3, n_rungs=0, seed=203 + d, d=d)               # widest window, all rungs
    _run_interp(1, 7, 1, 1, 3, 1.7, seed=204 + d, d=d)


@pytest.mark.parametrize("d", [32, 128])
def test_interp_integer_alpha_matches_integer_offset_kernel_head_dims(d):
    torch = torch_cuda()
    rng = np.random.default_rng(300 + d)
    n = 1024
    qb, kb, vb = (bf16_normal_bits(rng, (1, n, 2, d), 0.3) for _ in range(3))
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    for alpha in (1, 2):
        o1, l1 = sa.offset_attn_interp_fwd(q, k, v, 8, float(alpha))
        offs = sa.sa_fib_offsets(alpha, 1, 15, 8, n)
        o2, l2 = sa.offset_attn_fwd(q, k, v, 8, offs)
        torch.cuda.synchronize()
        assert (o1.float() - o2.float()).abs().max().item() < 2 * O_MAX_ABS
        assert (l1 - l2).abs().max().item() < 2 * LSE_MAX_ABS


@pytest.mark.parametrize("d", [32, 128])
def test_head_dims_whole_8k_layer(d):
    """A whole 8K layer (2 sequences, 4 heads on 2 KV heads) at d = 32 and 128, every row
    compared: the 64-query tiles of d = 128 and the slab rings over many waves."""
    _run(2, 8192, 4, 2, 8, Fraction(2, 1), seed=400 + d, d=d)
    _run_interp(2, 8192, 4, 2, 8, 1.618, seed=401 + d, d=d)
