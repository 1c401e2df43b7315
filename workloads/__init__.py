"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds no arithmetic of the attention method: it only draws bytes and
bf16 bit patterns from seeded generators and names the workload shapes. Both the
oracle (``oracle/``) and the GPU tests / bench consume exactly these arrays, so
parity is always checked on identical bits.

Workloads (shapes and pattern parameters as the pages and the workload statement give them):

* ``tiny_topk``      - 1 x 512 byte tokens, block 32, 2 heads, d_h 32, top-2
                       compression-guided causal mask (correctness size).
* ``bytelm_topk_8k`` - 4 x 8192 byte tokens, block 64, 12 heads, d_h 64, 4-block
                       window, 1 global block, top-16 literal blocks (the
                       Parameter-free Adaptive Sparse Attention page, section 4.1 /
                       Table 6 model shape: 12 heads of 64 at 8K bytes).
* ``bigbird_4k`` / ``bigbird_16k`` - 8 sequences, 12 heads, d_h 64, block 32,
                       window 256 tokens, 32 global tokens, 32 random tokens (the
                       BigBird page, section 2 defaults w=256, g=32, r=32).
* ``fib_2k`` / ``fib_8k`` - 16 layers, 8 sequences, 8 heads of 64, token-granular
                       window plus alpha-scaled Fibonacci offsets (Depth-Staggered
                       Fibonacci Spacing page, sections 2-3).
* ``cas_heads_8k``   - 4 x 8192 byte tokens, block 128, 12 heads, d_h 64, the mean-threshold
                       mask with a +-1-block window and zlib level 1, split over head
                       groups: 6 local, 3 long-range (literal pairs), 3 hybrid (the
                       Parameter-free Adaptive Sparse Attention page, section 4.1,
                       Table 8 and Appendix B "Head-specific mask distribution").
* ``fib_8k_coprime`` / ``pow2_8k`` - ``fib_8k`` with the coprime stagger of the alpha
                       ramp, and with the power-of-2 control base (same page, section 2).
* ``fib_interp_8k``  - ``fib_8k`` through the interpolated gather of a continuous alpha
                       (the same page, section 2 "Attended set").
* ``long_topk_64k``  - 1 x 65536 byte tokens, block 128, 16 heads, d_h 128, top-64
                       (top-k swept over 16/64/256), plus ``full_16k``.
* ``full_32k_one_head`` - the full causal mask over 32768 tokens for one sequence and one
                       head of 128: few work items with long key lists.

Stand-in data: the pages measure on PG-19 and FineWeb-Edu style corpora, which are
not available here. The byte generators below reproduce the properties the mask
depends on - a mix of repetitive (compressible) and random (incompressible)
segments - and nothing else.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "WORKLOADS", "workload", "bytes_phrase_random", "bytes_zipf_text",
    "bf16_normal_bits", "qkv_bits", "byte_stream", "bf16_bits_to_f64",
]


# --------------------------------------------------------------------------
# workload table (pure parameters)
# --------------------------------------------------------------------------

WORKLOADS = {
    "tiny_topk": dict(kind="topk", batch=1, n_tokens=512, block=32, heads=2, kv_heads=2,
                      head_dim=32, window_blocks=2, global_blocks=1, topk=2, causal=1,
                      std=1.0 / np.sqrt(32.0), bytes="phrase_random", seed=43),
    "bytelm_topk_8k": dict(kind="topk", batch=4, n_tokens=8192, block=64, heads=12, kv_heads=12,
                           head_dim=64, window_blocks=4, global_blocks=1, topk=16, causal=1,
                           std=1.0 / 8.0, bytes="zipf_text", seed=44),
    "bigbird_4k": dict(kind="bigbird", batch=8, n_tokens=4096, block=32, heads=12, kv_heads=12,
                       head_dim=64, window_tokens=256, global_tokens=32, random_tokens=32,
                       causal=0, std=1.0 / 8.0, seed=45),
    "bigbird_16k": dict(kind="bigbird", batch=8, n_tokens=16384, block=32, heads=12, kv_heads=12,
                        head_dim=64, window_tokens=256, global_tokens=32, random_tokens=32,
                        causal=0, std=1.0 / 8.0, seed=45),
    "fib_2k": dict(kind="fib", layers=16, batch=8, n_tokens=2048, heads=8, kv_heads=8, head_dim=64,
                   window=8, alpha_lo=(1, 2), alpha_hi=(2, 1), n_rungs=15, std=1.0 / 8.0, seed=46),
    "fib_8k": dict(kind="fib", layers=16, batch=8, n_tokens=8192, heads=8, kv_heads=8, head_dim=64,
                   window=8, alpha_lo=(1, 2), alpha_hi=(2, 1), n_rungs=15, std=1.0 / 8.0, seed=46),
    # head_components: per head, the mask part it reads (1 local, 2 literal pairs, 3 both)
    "cas_heads_8k": dict(kind="literal_heads", batch=4, n_tokens=8192, block=128, heads=12, kv_heads=12,
                         head_dim=64, window_blocks=1, causal=1, zlib_level=1,
                         head_components=(1, 1, 1, 1, 1, 1, 2, 2, 2, 3, 3, 3),
                         std=1.0 / 8.0, bytes="zipf_text", seed=48),
    # schedule variants of fib_8k: coprime alpha stagger (layer l takes ramp index 7l mod 16)
    # and the power-of-2 control base (11 rungs up to 1024)
    "fib_8k_coprime": dict(kind="fib", layers=16, batch=8, n_tokens=8192, heads=8, kv_heads=8, head_dim=64,
                           window=8, alpha_lo=(1, 2), alpha_hi=(2, 1), n_rungs=15, stride=7, std=1.0 / 8.0,
                           seed=46),
    "pow2_8k": dict(kind="fib", layers=16, batch=8, n_tokens=8192, heads=8, kv_heads=8, head_dim=64, window=8,
                    alpha_lo=(1, 2), alpha_hi=(2, 1), n_rungs=11, ladder="pow2", std=1.0 / 8.0, seed=46),
    # interpolated gather: the page's ramp alpha_l = 0.5 + l / 15 taken as real numbers
    # (continuous distances alpha f_k, interpolated between neighbouring rows)
    "fib_interp_8k": dict(kind="fib", layers=16, batch=8, n_tokens=8192, heads=8, kv_heads=8, head_dim=64,
                          window=8, alpha_lo=(1, 2), alpha_hi=(3, 2), n_rungs=15, interp=True, std=1.0 / 8.0,
                          seed=46),
    "long_topk_64k": dict(kind="topk", batch=1, n_tokens=65536, block=128, heads=16, kv_heads=16,
                          head_dim=128, window_blocks=4, global_blocks=1, topk=64, causal=1,
                          std=1.0 / np.sqrt(128.0), bytes="phrase_random", seed=47),
    "full_16k": dict(kind="full", batch=1, n_tokens=16384, block=128, heads=16, kv_heads=16,
                     head_dim=128, causal=1, std=1.0 / np.sqrt(128.0), seed=47),
    # few work items with long key lists (one sequence, one head): the forward's split path
    "full_32k_one_head": dict(kind="full", batch=1, n_tokens=32768, block=128, heads=1, kv_heads=1,
                              head_dim=128, causal=1, std=1.0 / np.sqrt(128.0), seed=49),
}


def workload(name: str, **overrides) -> dict:
    """Return a copy of a named workload with optional parameter overrides."""
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    cfg["name"] = name
    return cfg


# --------------------------------------------------------------------------
# byte streams
# --------------------------------------------------------------------------

def bytes_phrase_random(seed: int, n: int) -> np.ndarray:
    """Alternate a repeated random 16-byte phrase with a uniform-random byte run.

    Segment lengths are uniform in [32, 128]; the stream starts with a phrase
    segment. Returns ``uint8[n]``.
    """
    rng = np.random.default_rng(seed)
    out = np.empty(n, dtype=np.uint8)
    pos = 0
    phrase_turn = True
    while pos < n:
        seg = int(rng.integers(32, 129))
        seg = min(seg, n - pos)
        if phrase_turn:
            phrase = rng.integers(0, 256, size=16, dtype=np.uint8)
            reps = -(-seg // 16)
            out[pos:pos + seg] = np.tile(phrase, reps)[:seg]
        else:
            out[pos:pos + seg] = rng.integers(0, 256, size=seg, dtype=np.uint8)
        pos += seg
        phrase_turn = not phrase_turn
    return out


def _vocabulary(rng: np.random.Generator, size: int = 256) -> list[bytes]:
    words = []
    letters = np.frombuffer(b"abcdefghijklmnopqrstuvwxyz", dtype=np.uint8)
    for _ in range(size):
        length = int(rng.integers(2, 11))
        words.append(bytes(letters[rng.integers(0, 26, size=length)].tolist()))
    return words


def bytes_zipf_text(seed: int, n: int, p_text: float = 0.6, zipf_s: float = 1.1) -> np.ndarray:
    """Mix of text-like segments and uniform-random byte segments.

    Each segment has a length uniform in [32, 128]. With probability ``p_text`` it is
    text: space-separated words from a 256-entry random lowercase vocabulary (word
    length 2-10), drawn with truncated Zipf frequencies p(k) ~ k^-1.1; otherwise it
    is uniform-random bytes. Returns ``uint8[n]``.
    """
    rng = np.random.default_rng(seed)
    vocab = _vocabulary(rng)
    ranks = np.arange(1, len(vocab) + 1, dtype=np.float64)
    probs = ranks ** (-zipf_s)
    probs /= probs.sum()
    out = np.empty(n, dtype=np.uint8)
    pos = 0
    while pos < n:
        seg = min(int(rng.integers(32, 129)), n - pos)
        if rng.random() < p_text:
            buf = bytearray()
            while len(buf) < seg:
                buf += vocab[int(rng.choice(len(vocab), p=probs))] + b" "
            out[pos:pos + seg] = np.frombuffer(bytes(buf[:seg]), dtype=np.uint8)
        else:
            out[pos:pos + seg] = rng.integers(0, 256, size=seg, dtype=np.uint8)
        pos += seg
    return out


def byte_stream(cfg: dict, seq_offset: int = 0) -> np.ndarray:
    """``uint8[batch, n_tokens]`` byte tokens for a compression-guided workload.

    Sequence ``b`` of the result is global sequence ``seq_offset + b``: shards of a larger
    global batch (one per rank) are generated independently and agree with the whole."""
    gen = {"phrase_random": bytes_phrase_random, "zipf_text": bytes_zipf_text}[cfg["bytes"]]
    rows = [gen(cfg["seed"] * 1000 + seq_offset + b, cfg["n_tokens"]) for b in range(cfg["batch"])]
    return np.stack(rows)


# --------------------------------------------------------------------------
# bf16 tensors
# --------------------------------------------------------------------------

def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_normal_bits(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    """Draw N(0, std^2) in float32 and round to bf16; returns uint16 bit patterns."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    x *= np.float32(std)
    return _f32_to_bf16_bits(x)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def qkv_bits(cfg: dict, seed_offset: int = 0, n_tokens: int | None = None,
             batch: int | None = None, q_scale_pow2: int = 0):
    """Q, K, V bf16 bit patterns with layout [batch, n_tokens, heads(kv), head_dim].

    ``q_scale_pow2`` multiplies Q by 2**q_scale_pow2 exactly (a stress input that
    makes the softmax far from uniform).
    """
    n = cfg["n_tokens"] if n_tokens is None else n_tokens
    bt = cfg["batch"] if batch is None else batch
    rng = np.random.default_rng(cfg["seed"] + 7919 * seed_offset)
    d = cfg["head_dim"]
    q = bf16_normal_bits(rng, (bt, n, cfg["heads"], d), cfg["std"] * (2.0 ** q_scale_pow2))
    k = bf16_normal_bits(rng, (bt, n, cfg["kv_heads"], d), cfg["std"])
    v = bf16_normal_bits(rng, (bt, n, cfg["kv_heads"], d), cfg["std"])
    return q, k, v
