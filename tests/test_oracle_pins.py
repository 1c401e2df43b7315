"""Pins of the CPU oracle against facts that do not come from the oracle itself:
library routines (numpy Philox, gzip framing), closed forms printed on the pages,
brute force from token-level definitions, and an independent dense route.
"""
import gzip
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import masks as om
from workloads import bf16_bits_to_f64, bytes_phrase_random, bytes_zipf_text, qkv_bits, workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


# ------------------------------------------------------------------ Philox

def test_philox_matches_numpy_raw_stream():
    for seed in (0, 45, 12345, 2**63 + 7):
        ref = np.random.Philox(key=seed).random_raw(37)
        mine = [oracle.philox_word(seed, p) for p in range(37)]
        assert mine == [int(x) for x in ref]


def test_philox_known_answer_zero_key():
    # Random123 known-answer: philox4x64_10 with zero counter and zero key.
    out = oracle.philox4x64_10((0, 0, 0, 0), (0, 0))
    assert out == [0x16554d9eca36314c, 0xdb20fe9d672d0fdc, 0xd7e772cee186176b, 0x7e68b68aec7ba23b]


# ------------------------------------------------------------------ ratios (Eq. 1)

def test_ratio_is_compressed_length_over_block():
    data = bytes_phrase_random(3, 1024)
    r = oracle.block_ratios(data, 64)
    for i in range(16):
        n = r[i] * 64
        assert n == int(n) and n > 0
        # gzip framing = zlib framing + 12 bytes (10+8 header/trailer vs 2+4)
        chunk = data[i * 64:(i + 1) * 64].tobytes()
        assert len(gzip.compress(chunk, compresslevel=6, mtime=0)) == int(n) + 12


def test_ratio_extremes():
    rng = np.random.default_rng(0)
    same = np.full(128, 7, dtype=np.uint8)
    rnd = rng.integers(0, 256, 128, dtype=np.uint8)
    r = oracle.block_ratios(np.concatenate([same, rnd]), 128)
    assert r[0] < 0.2          # a run compresses to a few bytes
    assert r[1] > 1.0          # random bytes expand (so r in (0,1] does not hold)


def test_mean_threshold_is_exact_integer_compare():
    for seed in range(5):
        data = bytes_zipf_text(seed, 4096)
        r = oracle.block_ratios(data, 32)
        lens = [int(x * 32) for x in r]
        nb = len(lens)
        want = [L * nb > sum(lens) for L in lens]
        assert oracle.literal_flags(r) == want


# ------------------------------------------------------------------ topk

def _topk_by_rank(ratios, w, g, k):
    """Brute force by counting ranks (no sort): J is literal for I iff fewer than k
    candidates beat it on (ratio desc, index asc)."""
    nb = len(ratios)
    rows = []
    for I in range(nb):
        cand = [J for J in range(g, I - w + 1)]
        chosen = []
        for J in cand:
            beats = sum(1 for J2 in cand if ratios[J2] > ratios[J] or (ratios[J2] == ratios[J] and J2 < J))
            if beats < k:
                chosen.append(J)
        row = set(range(max(0, I - w + 1), I + 1)) | set(range(min(g, max(0, I - w + 1)))) | set(chosen)
        rows.append(sorted(row))
    return rows


@pytest.mark.parametrize("w,g,k", [(2, 1, 2), (4, 1, 16), (1, 0, 3), (3, 2, 5), (1, 0, 0)])
def test_topk_rows_brute_force_and_counts(w, g, k):
    rng = np.random.default_rng(w * 100 + g * 10 + k)
    nb = 40
    # few distinct values so ties are frequent
    ratios = rng.integers(30, 36, nb).astype(np.float32) / np.float32(32)
    rows = om.csr_topk_rows(ratios, w, g, k)
    assert rows == _topk_by_rank(ratios, w, g, k)
    for I, row in enumerate(rows):
        assert len(row) == om.topk_row_count(I, w, g, k)
        assert all(J <= I for J in row)


def test_topk_bytelm_8k_pair_and_edge_counts():
    cfg = workload("bytelm_topk_8k")
    nb = cfg["n_tokens"] // cfg["block"]
    counts = [om.topk_row_count(I, cfg["window_blocks"], cfg["global_blocks"], cfg["topk"]) for I in range(nb)]
    assert sum(counts) == 2478
    b = cfg["block"]
    edges = sum((c - 1) * b * b + b * (b + 1) // 2 for c in counts) * cfg["batch"] * cfg["heads"]
    assert edges == 474_808_320          # 4.748e8 edge pairs
    assert 4 * edges * cfg["head_dim"] == 121_550_929_920


def test_topk_special_cases():
    nb, b = 12, 4
    r = np.linspace(0.5, 1.5, nb).astype(np.float32)
    diag = om.csr_topk_rows(r, 1, 0, 0)
    assert diag == [[I] for I in range(nb)]
    dense = om.csr_topk_rows(r, nb, 0, 5)
    assert dense == [list(range(I + 1)) for I in range(nb)]
    rp, ci = om.build_csr(om.MaskParams("topk", b, nb * b, 1, nb, 0, 5), r[None, :], 1)
    tok = om.block_mask_to_token_mask(om.csr_to_block_mask(rp, ci, nb), b, 1)
    assert (tok == np.tril(np.ones((nb * b, nb * b), dtype=bool))).all()


# ------------------------------------------------------------------ literal_mean (Alg. 1)

def _algorithm1_token_mask(ratios, b, w):
    """Appendix B Algorithm 1 written with numpy outer products."""
    B = len(ratios)
    r = np.asarray(ratios, dtype=np.float64)
    lit = r > r.mean()
    i = np.arange(B)[:, None]
    j = np.arange(B)[None, :]
    M = np.eye(B, dtype=bool) | (np.abs(i - j) <= w) | (lit[:, None] & lit[None, :] & (np.abs(i - j) > w))
    tok = np.kron(M, np.ones((b, b), dtype=bool))
    return tok & ~np.triu(np.ones_like(tok), 1)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_literal_mean_matches_algorithm1(seed):
    data = bytes_zipf_text(seed, 2048)
    b, w = 64, 1
    r = oracle.block_ratios(data, b)
    p = om.MaskParams("literal_mean", b, 2048, 1, w)
    rp, ci = om.build_csr(p, r[None, :], 1)
    tok = om.block_mask_to_token_mask(om.csr_to_block_mask(rp, ci, p.nb), b, 1)
    assert (tok == _algorithm1_token_mask(r, b, w)).all()


# ------------------------------------------------------------------ bigbird

def test_bigbird_counts_against_page_formula():
    g_ = _golden("bigbird_defaults.txt")
    w, g, r = (int(g_[k][0]) for k in ("w", "g", "r"))
    for n in (4096, 16384, 1024):
        b = 32
        wb, gb, rb = w // b, g // b, r // b
        nb = n // b
        rows = om.csr_bigbird_rows(nb, wb, gb, rb, seed=45)
        G = set(range(gb))
        n_global = n_random = n_window = overlap = 0
        for I, row in enumerate(rows):
            W = set(om.bigbird_window(I, wb, nb))
            if I < gb:
                n_global += nb
                continue
            assert set(row) >= W | G
            R = set(row) - W - G
            assert len(R) == rb
            n_global += gb
            n_random += len(R)
            n_window += len(W)
            overlap += len(W & G)
        bb2 = b * b
        # |G_G| = 2gN - g^2 exactly (global rows see all keys, all rows see globals)
        assert n_global * bb2 == 2 * g * n - g * g
        # |G_R| = (N - g) r: every non-global query gets r random key tokens
        assert n_random * bb2 == (n - g) * r
        # the page's |G_BB| counts window and random edges of every row; the union
        # differs only by the global rows' window+random and by boundary/overlap terms
        deficit = sum(wb - len(om.bigbird_window(I, wb, nb)) for I in range(gb, nb))
        union = sum(len(row) for row in rows) * bb2
        assert union == n * (w + r) + 2 * g * n - g * g - g * (w + r) - (deficit + overlap) * bb2
        assert n_window * bb2 == (n - g) * w - deficit * bb2
    # interior key slots per query and the page's printed 13x reduction at N = 4096
    assert round(4096 / (w + g + r)) == int(g_["reduction_at_4096"][0])


def test_bigbird_random_draws_distinct_and_valid():
    nb, wb, gb, rb = 64, 4, 2, 3
    rows = om.csr_bigbird_rows(nb, wb, gb, rb, seed=7)
    for I, row in enumerate(rows):
        assert row == sorted(set(row))
        if I >= gb:
            assert len(row) == len(set(om.bigbird_window(I, wb, nb)) | set(range(gb))) + rb


def _chi2_sf(stat: float, dof: int) -> float:
    scipy_stats = pytest.importorskip("scipy.stats")
    return float(scipy_stats.chi2.sf(stat, dof))


@pytest.mark.parametrize("seed,rb", [(45, 1), (7, 1), (45, 3)])
def test_bigbird_random_draws_are_uniform(seed, rb):
    """[BB] section 2: the random blocks are drawn uniformly among the blocks outside the
    window and the globals. Over 4096 rows the position of every drawn block within its
    row's candidate list A(I), scaled to [0, 1), must be uniform (a chi-square test on 20
    bins), and so must the drawn block indices themselves, against the expected count
    sum_I |A(I) n bin| / |A(I)| of each of 16 index bins. A biased index map (a shift too
    many, a modulo of the low word, the draw taken from the full row) fails one of them."""
    nb, wb, gb = 4096, 8, 1
    rows = om.csr_bigbird_rows(nb, wb, gb, rb, seed)
    pos_bins = np.zeros(20)
    idx_obs = np.zeros(16)
    idx_exp = np.zeros(16)
    edges = np.linspace(0, nb, 17)
    for I in range(gb, nb):
        W = set(om.bigbird_window(I, wb, nb))
        A = [J for J in range(nb) if J not in W and J >= gb]
        drawn = [J for J in rows[I] if J not in W and J >= gb]
        assert len(drawn) == rb
        for J in drawn:
            u = A.index(J) / len(A)
            pos_bins[min(19, int(u * 20))] += 1
            idx_obs[min(15, int(J * 16 // nb))] += 1
        counts, _ = np.histogram(A, bins=edges)
        idx_exp += rb * counts / len(A)
    exp_pos = pos_bins.sum() / 20
    stat_pos = float(((pos_bins - exp_pos) ** 2 / exp_pos).sum())
    stat_idx = float(((idx_obs - idx_exp) ** 2 / idx_exp).sum())
    assert _chi2_sf(stat_pos, 19) > 1e-3, (stat_pos, pos_bins)
    assert _chi2_sf(stat_idx, 15) > 1e-3, (stat_idx, idx_obs, idx_exp)


def test_bigbird_uniformity_test_rejects_a_biased_draw(monkeypatch):
    """The chi-square statistic above does detect a plausible mistake: an index map that
    drops one bit (draws only from the first half of A) is rejected."""
    nb, wb, gb = 4096, 8, 1
    real = om.philox_word
    monkeypatch.setattr(om, "philox_word", lambda seed, p: real(seed, p) >> 1)
    rows = om.csr_bigbird_rows(nb, wb, gb, 1, 45)
    pos_bins = np.zeros(20)
    for I in range(gb, nb):
        W = set(om.bigbird_window(I, wb, nb))
        A = [J for J in range(nb) if J not in W and J >= gb]
        J = [J for J in rows[I] if J not in W and J >= gb][0]
        pos_bins[min(19, int(A.index(J) / len(A) * 20))] += 1
    exp_pos = pos_bins.sum() / 20
    assert _chi2_sf(float(((pos_bins - exp_pos) ** 2 / exp_pos).sum()), 19) < 1e-6


def test_bigbird_dense_special_case():
    nb = 10
    rows = om.csr_bigbird_rows(nb, 2 * nb, 1, 2, seed=1)
    assert rows == [list(range(nb))] * nb


# ------------------------------------------------------------------ fibonacci

def test_fib_rungs_and_alpha_schedule_match_page():
    g_ = _golden("fib_rungs.txt")
    assert oracle.fib_rungs(int(g_["K"][0])) == [int(x) for x in g_["rungs"]]
    al = oracle.alpha_schedule(int(g_["layers"][0]), lo=(1, 2), hi=(3, 2))
    assert al[0] == Fraction(g_["alpha_first"][0]) and al[-1] == Fraction(g_["alpha_last"][0])
    assert all(al[l + 1] - al[l] == Fraction(1, 15) for l in range(15))
    # workload ramp 0.5 -> 2.0 is (5 + l) / 10
    assert oracle.alpha_schedule(16, (1, 2), (2, 1)) == [Fraction(5 + l, 10) for l in range(16)]


def test_fib_offsets_integer_closed_form():
    rungs = oracle.fib_rungs(15)
    for alpha in oracle.alpha_schedule(16, (1, 2), (2, 1)) + oracle.alpha_schedule(16, (1, 2), (3, 2)):
        num, den = alpha.numerator, alpha.denominator
        want = set()
        for f in rungs:
            q, rem = divmod(2 * num * f + den, 2 * den)   # floor(x + 1/2)
            if rem == 0 and q % 2 == 1:                   # exact tie: go to even
                q -= 1
            want.add(q)
        assert oracle.fib_offsets(alpha, rungs) == sorted(want)
    # the half-even reading changes layer 0 (alpha = 1/2): 1/2 -> 0, 3/2 -> 2, 5/2 -> 2
    assert oracle.fib_offsets(Fraction(1, 2), [1, 3, 5]) == [0, 2]


def test_coprime_stagger_is_a_permutation_of_the_ramp():
    """[FIB] section 2: the same multiset of alphas, layer l -> (7 l mod 16); adjacent
    layers land at least 7 ramp steps apart, and 7 is its own inverse mod 16 (so both
    directions of the map give the same schedule)."""
    lin = oracle.alpha_schedule(16, (1, 2), (3, 2))
    cop = oracle.alpha_schedule(16, (1, 2), (3, 2), stride=7)
    assert sorted(cop) == sorted(lin) and cop != lin
    idx = [lin.index(a) for a in cop]
    assert idx == [0, 7, 14, 5, 12, 3, 10, 1, 8, 15, 6, 13, 4, 11, 2, 9]
    assert min(abs(idx[l + 1] - idx[l]) for l in range(15)) == 7
    assert (7 * 7) % 16 == 1 and [idx.index(l) for l in range(16)] == idx
    with pytest.raises(ValueError):
        oracle.alpha_schedule(16, (1, 2), (3, 2), stride=4)


def test_pow2_rungs_reach_and_offsets():
    """[FIB] "Control base": powers of two reaching the Fibonacci base's 987 ~ 1024 with
    fewer rungs; integer offsets follow the same rounding as the Fibonacci ones."""
    r = oracle.pow2_rungs()
    assert r == [1 << k for k in range(11)] and len(r) < len(oracle.fib_rungs(15))
    assert r[-1] == 1024 and r[-2] < 987 < r[-1]
    assert oracle.pow2_rungs_upto(8192) == [1 << k for k in range(14)]
    # alpha = 3/4: 3/4 -> 1, 3/2 -> 2, 3 -> 3, 6, 12, ..., 768
    assert oracle.fib_offsets(Fraction(3, 4), r) == [1, 2, 3, 6, 12, 24, 48, 96, 192, 384, 768]


def test_offset_key_set_count_closed_form():
    D = oracle.fib_offsets(Fraction(7, 10), oracle.fib_rungs(15))
    W = 8
    for i in range(0, 1500, 7):
        ks = oracle.offset_key_set(i, W, D)
        assert len(ks) == min(W, i) + 1 + sum(1 for d in D if W < d <= i)


# ------------------------------------------------------------------ attention

def _tiny_qkv(n=64, h=2, hkv=2, d=16, seed=0, qmul=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((2, n, h, d)) * qmul
    k = rng.standard_normal((2, n, hkv, d))
    v = rng.standard_normal((2, n, hkv, d))
    return q, k, v


def _brute_attention(q, k, v, allowed, scale):
    """Per-query pure-Python loops with math.exp (no vectorised softmax)."""
    bt, n, h, d = q.shape
    hkv = k.shape[2]
    o = np.zeros_like(q)
    lse = np.full((bt, h, n), -np.inf)
    for s in range(bt):
        for hh in range(h):
            hk = hh // (h // hkv)
            for i in range(n):
                keys = [j for j in range(n) if allowed(s, i, j)]
                if not keys:
                    continue
                sc = [scale * sum(q[s, i, hh, c] * k[s, j, hk, c] for c in range(d)) for j in keys]
                m = max(sc)
                z = sum(math.exp(x - m) for x in sc)
                lse[s, hh, i] = m + math.log(z)
                for j, x in zip(keys, sc):
                    o[s, i, hh, :] += math.exp(x - lse[s, hh, i]) * v[s, j, hk, :]
    return o, lse


def test_attention_csr_brute_force_topk_gqa():
    n, b = 48, 8
    q, k, v = _tiny_qkv(n=n, h=4, hkv=2, d=8, qmul=3.0)
    rng = np.random.default_rng(5)
    ratios = rng.integers(6, 12, (2, n // b)).astype(np.float32) / np.float32(8)
    p = om.MaskParams("topk", b, n, 1, 2, 1, 1)
    rp, ci = om.build_csr(p, ratios, 2)
    o, lse = oracle.attention_csr(q, k, v, rp, ci, b, 1)
    masks = [om.block_mask_to_token_mask(om.csr_to_block_mask(rp, ci, n // b, s), b, 1) for s in range(2)]
    ob, lb = _brute_attention(q, k, v, lambda s, i, j: masks[s][i, j], 1 / math.sqrt(8))
    assert np.allclose(o, ob, atol=1e-12) and np.allclose(lse, lb, atol=1e-12)


def test_full_mode_equals_dense_causal_and_bidirectional():
    n, b = 64, 16
    q, k, v = _tiny_qkv(n=n, d=16, qmul=4.0, seed=2)
    for causal in (1, 0):
        rp, ci = om.build_csr(om.MaskParams("full", b, n, causal), None, 1)
        o, lse = oracle.attention_csr(q, k, v, rp, ci, b, causal)
        tm = np.tril(np.ones((n, n), dtype=bool)) if causal else np.ones((n, n), dtype=bool)
        od, ld = oracle.dense_masked_attention(q, k, v, tm)
        assert np.max(np.abs(o - od)) < 1e-12 and np.max(np.abs(lse - ld)) < 1e-12


def test_rows_sum_to_one_and_lse_counts_keys():
    """V = 1 gives O = sum_j P_ij = 1; K = 0 gives LSE = ln |S(i)|."""
    cfg = workload("tiny_topk")
    n, b = cfg["n_tokens"], cfg["block"]
    data = bytes_phrase_random(cfg["seed"], n)
    r = oracle.block_ratios(data, b)[None, :]
    p = om.MaskParams("topk", b, n, 1, cfg["window_blocks"], cfg["global_blocks"], cfg["topk"])
    rp, ci = om.build_csr(p, r, 1)
    qb, kb, vb = qkv_bits(cfg, q_scale_pow2=3)
    q, k = bf16_bits_to_f64(qb), bf16_bits_to_f64(kb)
    o, lse = oracle.attention_csr(q, k, np.ones_like(k), rp, ci, b, 1)
    assert np.max(np.abs(o - 1.0)) < 1e-12
    _, lse0 = oracle.attention_csr(q, np.zeros_like(k), np.ones_like(k), rp, ci, b, 1)
    counts = np.zeros(n)
    for i in range(n):
        I = i // b
        counts[i] = sum(min(b, i - J * b + 1) for J in ci[rp[0, I]:rp[0, I + 1]])
    assert np.max(np.abs(lse0[0] - np.log(counts)[None, :])) < 1e-12


def test_offset_attention_equals_dense_route_and_counts():
    n, W = 64, 3
    q, k, v = _tiny_qkv(n=n, h=2, hkv=1, d=8, qmul=3.0, seed=4)
    D = oracle.fib_offsets(Fraction(3, 5), oracle.fib_rungs(15))
    o, lse = oracle.attention_offsets(q, k, v, W, D)
    tm = np.zeros((n, n), dtype=bool)
    for i in range(n):
        tm[i, oracle.offset_key_set(i, W, D)] = True
    od, ld = oracle.dense_masked_attention(q, k, v, tm)
    assert np.max(np.abs(o - od)) < 1e-12 and np.max(np.abs(lse - ld)) < 1e-12
    _, l0 = oracle.attention_offsets(q, np.zeros_like(k), v, W, D)
    cnt = np.array([len(oracle.offset_key_set(i, W, D)) for i in range(n)])
    assert np.max(np.abs(l0[0, 0] - np.log(cnt))) < 1e-12
    samples = [(1, 63, 1), (0, 0, 0), (0, 17, 1)]
    os_, ls_ = oracle.attention_offsets(q, k, v, W, D, samples=samples)
    for t, (s, i, hh) in enumerate(samples):
        assert np.allclose(os_[t], o[s, i, hh]) and np.isclose(ls_[t], lse[s, hh, i])


def test_sampled_rows_match_full_csr_attention():
    n, b = 64, 8
    q, k, v = _tiny_qkv(n=n, d=8, seed=9, qmul=2.0)
    rp, ci = om.build_csr(om.MaskParams("bigbird", b, n, 0, 2, 1, 0, 1, 3), None, 1)
    o, lse = oracle.attention_csr(q, k, v, rp, ci, b, 0)
    samples = [(0, 0, 0), (1, 33, 1), (0, 63, 0)]
    os_, ls_ = oracle.attention_rows_csr(q, k, v, rp, ci, b, 0, samples)
    for t, (s, i, hh) in enumerate(samples):
        assert np.allclose(os_[t], o[s, i, hh], atol=1e-13) and np.isclose(ls_[t], lse[s, hh, i])


def test_empty_row_gives_zero_and_minus_inf():
    n, b = 32, 8
    q, k, v = _tiny_qkv(n=n, d=8)
    rp = np.array([[0, 1, 1, 2, 3]], dtype=np.int32)      # row 1 is empty
    ci = np.array([0, 2, 3], dtype=np.int32)
    o, lse = oracle.attention_csr(q, k, v, rp, ci, b, 1)
    assert np.all(o[:, 8:16] == 0) and np.all(np.isneginf(lse[:, :, 8:16]))


# ------------------------------------------------------------------ head groups ([CAS] App. B)

def _algorithm1_parts(ratios, w):
    """Algorithm 1's three block-mask components as separate numpy outer products."""
    B = len(ratios)
    r = np.asarray(ratios, dtype=np.float64)
    lit = r > r.mean()
    i = np.arange(B)[:, None]
    j = np.arange(B)[None, :]
    eye = np.eye(B, dtype=bool)
    local = np.abs(i - j) <= w
    literal = lit[:, None] & lit[None, :] & (np.abs(i - j) > w)
    return eye, local, literal


@pytest.mark.parametrize("seed,causal,w", [(0, 1, 1), (1, 0, 2), (2, 1, 0)])
def test_literal_mean_components_match_algorithm1_parts(seed, causal, w):
    """LOCAL = M_local u I, LITERAL = M_lit u I, both = M, each intersected with the
    causal triangle at token level ([CAS] Appendix B, Algorithm 1 step 3 and the head
    distribution paragraph)."""
    data = bytes_zipf_text(seed, 2048)
    b = 64
    r = oracle.block_ratios(data, b)
    eye, local, literal = _algorithm1_parts(r, w)
    want = {oracle.LOCAL: eye | local, oracle.LITERAL: eye | literal, 0: eye | local | literal}
    for comp, M in want.items():
        p = om.MaskParams("literal_mean", b, 2048, causal, w, components=comp)
        rp, ci = om.build_csr(p, r[None, :], 1)
        tok = om.block_mask_to_token_mask(om.csr_to_block_mask(rp, ci, p.nb), b, causal)
        ref = np.kron(M, np.ones((b, b), dtype=bool))
        if causal:
            ref &= ~np.triu(np.ones_like(ref), 1)
        assert (tok == ref).all()


def test_literal_mean_components_partition_rows():
    """Every row of the full mask is the union of its LOCAL and LITERAL rows, and the two
    share only the diagonal block (local edges have |I-J| <= w, literal ones > w)."""
    rng = np.random.default_rng(5)
    for trial in range(6):
        nb = int(rng.integers(4, 40))
        ratios = rng.choice([0.5, 0.75, 1.0, 1.25], size=nb)
        w = int(rng.integers(0, 4))
        causal = trial % 2
        full = om.csr_literal_mean_rows(ratios, w, causal, 0)
        loc = om.csr_literal_mean_rows(ratios, w, causal, oracle.LOCAL)
        lit = om.csr_literal_mean_rows(ratios, w, causal, oracle.LITERAL)
        for I in range(nb):
            assert set(full[I]) == set(loc[I]) | set(lit[I])
            assert set(loc[I]) & set(lit[I]) == {I}


def test_local_component_is_topk_band_without_literals():
    """Causal LOCAL (|I-J| <= w, J <= I) is the TOPK mode's window of w+1 blocks with no
    globals and k = 0; the ratios must not matter."""
    rng = np.random.default_rng(9)
    for w in range(0, 5):
        nb = 37
        ratios = rng.random(nb)
        loc = om.csr_literal_mean_rows(ratios, w, 1, oracle.LOCAL)
        assert loc == om.csr_topk_rows(ratios, w + 1, 0, 0)


def test_literal_component_uniform_ratios_is_identity():
    """Equal ratios: no block exceeds the mean, so LITERAL leaves only the diagonal."""
    rows = om.csr_literal_mean_rows([0.7] * 20, 2, 0, oracle.LITERAL)
    assert rows == [[I] for I in range(20)]


def test_cas_head_groups_page_split():
    """12 heads: 0-5 local, 6-8 long-range (literal), 9-11 hybrid (full M)."""
    comp = oracle.cas_head_components(12)
    assert comp == [oracle.LOCAL] * 6 + [oracle.LITERAL] * 3 + [oracle.LOCAL | oracle.LITERAL] * 3


def test_attention_heads_reduces_to_single_csr_per_head():
    """Per-head CSR attention equals, head by head, the dense masked route with that
    head's token mask."""
    rng = np.random.default_rng(3)
    bt, n, h, d, b, w = 1, 256, 4, 16, 32, 1
    q, k, v = (rng.standard_normal((bt, n, h, d)) for _ in range(3))
    ratios = rng.choice([0.5, 1.0, 1.5], size=(1, n // b))
    csrs = []
    for comp in (oracle.LOCAL, oracle.LITERAL, 0):
        csrs.append(om.build_csr(om.MaskParams("literal_mean", b, n, 1, w, components=comp), ratios, 1))
    head_mask = [0, 1, 2, 1]
    o, lse = oracle.attention_csr_heads(q, k, v, csrs, head_mask, b, 1)
    for hh in range(h):
        rp, ci = csrs[head_mask[hh]]
        tok = om.block_mask_to_token_mask(om.csr_to_block_mask(rp, ci, n // b), b, 1)
        od, ld = oracle.dense_masked_attention(q[:, :, hh:hh + 1], k[:, :, hh:hh + 1], v[:, :, hh:hh + 1], tok)
        assert np.abs(o[:, :, hh] - od[:, :, 0]).max() < 1e-12
        assert np.abs(lse[:, hh] - ld[:, 0]).max() < 1e-12


def test_cas_workload_uses_page_head_split():
    from workloads import workload as _wl
    cfg = _wl("cas_heads_8k")
    assert list(cfg["head_components"]) == oracle.cas_head_components(cfg["heads"])
    assert cfg["block"] == 128 and cfg["window_blocks"] == 1 and cfg["zlib_level"] == 1   # [CAS] Table 8


# ------------------------------------------------------------------ backward

def _tiny_backward_case(seed, causal, hkv=1):
    rng = np.random.default_rng(seed)
    bt, n, h, d, b = 1, 48, 2, 4, 8
    q, k, v, do = (rng.standard_normal((bt, n, hh, d)) for hh in (h, hkv, hkv, h))
    rows = [[0], [0, 1], [1, 2], [0, 3], [2, 4], [0, 4, 5]] if causal else \
        [[0, 3], [1, 5], [0, 1, 2], [4], [2, 4, 5], [0, 5]]
    rp = np.zeros((1, len(rows) + 1), dtype=np.int32)
    cols = []
    for I, r in enumerate(rows):
        cols += r
        rp[0, I + 1] = len(cols)
    return q, k, v, do, rp, np.array(cols, dtype=np.int32), b


@pytest.mark.parametrize("causal,hkv", [(1, 1), (0, 2), (1, 2)])
def test_backward_matches_central_differences(causal, hkv):
    """dQ, dK, dV of L = sum(dO * O) against central differences of the forward oracle."""
    q, k, v, do, rp, ci, b = _tiny_backward_case(11 + causal + hkv, causal, hkv)
    dq, dk, dv = oracle.attention_csr_backward(q, k, v, do, rp, ci, b, causal)

    def loss(qq, kk, vv):
        o, _ = oracle.attention_csr(qq, kk, vv, rp, ci, b, causal)
        return float(np.sum(o * do))

    eps = 1e-6
    rng = np.random.default_rng(0)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        flat = x.reshape(-1)
        for idx in rng.choice(flat.size, size=40, replace=False):
            old = flat[idx]
            flat[idx] = old + eps
            lp = loss(q, k, v)
            flat[idx] = old - eps
            lm = loss(q, k, v)
            flat[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - g.reshape(-1)[idx]) < 1e-7 * max(1.0, abs(fd)), (name, idx)


def test_backward_matches_torch_autograd_dense_route():
    """The same gradients from torch autograd through a dense N x N masked softmax."""
    torch = pytest.importorskip("torch")
    q, k, v, do, rp, ci, b = _tiny_backward_case(5, 1, 1)
    n, g = q.shape[1], q.shape[2] // k.shape[2]
    tok = om.block_mask_to_token_mask(om.csr_to_block_mask(rp, ci, n // b), b, 1)
    dq, dk, dv = oracle.attention_csr_backward(q, k, v, do, rp, ci, b, 1)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    kk = tk.repeat_interleave(g, dim=2)
    vv = tv.repeat_interleave(g, dim=2)
    s = torch.einsum("bihd,bjhd->bhij", tq, kk) / np.sqrt(q.shape[3])
    s = s.masked_fill(~torch.tensor(tok), float("-inf"))
    o = torch.einsum("bhij,bjhd->bihd", torch.softmax(s, dim=-1), vv)
    o.backward(torch.tensor(do))
    assert np.abs(tq.grad.numpy() - dq).max() < 1e-12
    assert np.abs(tk.grad.numpy() - dk).max() < 1e-12
    assert np.abs(tv.grad.numpy() - dv).max() < 1e-12


def test_backward_invariants_and_sampled_forms():
    """Softmax rows of dS sum to zero, so dK sums to zero over the keys of each
    (sequence, kv head); dV sums to the sum of dO over queries with a key. The sampled
    evaluators agree with the full backward."""
    rng = np.random.default_rng(21)
    bt, n, h, hkv, d, b = 2, 256, 4, 2, 8, 32
    q, k, v, do = (rng.standard_normal((bt, n, hh, d)) for hh in (h, hkv, hkv, h))
    ratios = rng.integers(20, 60, (bt, n // b)) / np.float32(b)
    p = om.MaskParams("topk", b, n, 1, 2, 1, 2)
    rp, ci = om.build_csr(p, ratios, bt)
    dq, dk, dv = oracle.attention_csr_backward(q, k, v, do, rp, ci, b, 1)
    assert np.abs(dk.sum(axis=1)).max() < 1e-11
    want_dv = do.reshape(bt, n, hkv, h // hkv, d).sum(axis=(1, 3))
    assert np.abs(dv.sum(axis=1) - want_dv).max() < 1e-11
    smp = [(0, 0, 0), (1, 255, 3), (0, 100, 2), (1, 33, 1)]
    got = oracle.attention_rows_dq(q, k, v, do, rp, ci, b, 1, smp)
    assert np.abs(got - np.stack([dq[s, i, hh] for s, i, hh in smp])).max() < 1e-12
    smp_kv = [(0, 0, 0), (1, 255, 1), (0, 70, 1), (1, 31, 0)]
    gk, gv = oracle.attention_rows_dkdv(q, k, v, do, rp, ci, b, 1, smp_kv)
    assert np.abs(gk - np.stack([dk[s, j, hk] for s, j, hk in smp_kv])).max() < 1e-12
    assert np.abs(gv - np.stack([dv[s, j, hk] for s, j, hk in smp_kv])).max() < 1e-12


# ------------------------------------------------------------------ interpolated gather

@pytest.mark.parametrize("alpha", [1, 2, 3])
def test_interp_integer_alpha_is_the_integer_offset_set(alpha):
    """Integer alpha: every rung is an exact row; the result is the integer-offset
    attention of the same rungs (window duplicates removed)."""
    rng = np.random.default_rng(alpha)
    q, k, v = (rng.standard_normal((1, 300, 2, 8)) for _ in range(3))
    W = 6
    rungs = oracle.fib_rungs(15)
    lt = oracle.interp_rungs(alpha, rungs, W)
    assert all(t == 0.0 for _, t in lt)
    o1, l1 = oracle.attention_offsets_interp(q, k, v, W, lt)
    o2, l2 = oracle.attention_offsets(q, k, v, W, oracle.fib_offsets(Fraction(alpha), rungs))
    assert np.abs(o1 - o2).max() < 1e-12 and np.abs(l1 - l2).max() < 1e-12


def test_interp_linear_rows_give_keys_at_continuous_positions():
    """Keys and values linear in the position, K[j] = A + j B: the interpolated rung of
    query i is exactly the key at the continuous position i - alpha f_k, so attention
    equals a softmax over the closed-form keys A + (i - d) B."""
    rng = np.random.default_rng(3)
    n, d, W = 400, 8, 4
    A, B, C, E = (rng.standard_normal(d) for _ in range(4))
    pos = np.arange(n, dtype=np.float64)
    k = (A[None, :] + pos[:, None] * B[None, :] / n)[None, :, None, :]
    v = (C[None, :] + pos[:, None] * E[None, :] / n)[None, :, None, :]
    q = rng.standard_normal((1, n, 1, d))
    alpha = 0.8317
    lt = oracle.interp_rungs(alpha, oracle.fib_rungs(15), W)
    assert any(t > 0 for _, t in lt)
    smp = [(0, i, 0) for i in (0, 5, 37, 120, 399)]
    o, lse = oracle.attention_offsets_interp(q, k, v, W, lt, samples=smp)
    scale = 1.0 / np.sqrt(d)
    for t_idx, (_, i, _) in enumerate(smp):
        ps = [i - dl for dl in range(W + 1) if i - dl >= 0]
        ps += [i - alpha * f for f in oracle.fib_rungs(15)
               if i - alpha * f >= 0 and not (float(alpha * f).is_integer() and alpha * f <= W)]
        ps = np.array(ps)
        keys = A[None, :] + ps[:, None] * B[None, :] / n
        vals = C[None, :] + ps[:, None] * E[None, :] / n
        sc = keys @ q[0, i, 0] * scale
        m = sc.max()
        p = np.exp(sc - m)
        assert abs(lse[t_idx] - (m + np.log(p.sum()))) < 1e-12
        assert np.abs(o[t_idx] - (p / p.sum()) @ vals).max() < 1e-12


def test_backward_heads_matches_central_differences():
    """Per-head CSRs with a KV group shared by heads of different groups: the per-head
    backward against central differences of the per-head forward oracle."""
    rng = np.random.default_rng(17)
    bt, n, h, hkv, d, b = 1, 64, 4, 2, 4, 8
    q, k, v, do = (rng.standard_normal((bt, n, hh, d)) for hh in (h, hkv, hkv, h))
    ratios = rng.choice([0.5, 1.0, 1.5], size=(1, n // b))
    csrs = [om.build_csr(om.MaskParams("literal_mean", b, n, 1, 1, components=c), ratios, 1) for c in (1, 2, 3)]
    head_mask = [0, 2, 1, 0]                      # KV head 0: local + full; KV head 1: literal + local
    dq, dk, dv = oracle.attention_csr_backward_heads(q, k, v, do, csrs, head_mask, b, 1)

    def loss(qq, kk, vv):
        o, _ = oracle.attention_csr_heads(qq, kk, vv, csrs, head_mask, b, 1)
        return float(np.sum(o * do))

    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        flat = x.reshape(-1)
        for idx in rng.choice(flat.size, size=30, replace=False):
            old = flat[idx]
            flat[idx] = old + eps
            lp = loss(q, k, v)
            flat[idx] = old - eps
            lm = loss(q, k, v)
            flat[idx] = old
            assert abs((lp - lm) / (2 * eps) - g.reshape(-1)[idx]) < 1e-7 * max(1.0, abs(g.reshape(-1)[idx]))
