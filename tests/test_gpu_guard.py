"""Guard bands around every output: no kernel writes outside its output views.

Each output (O, LSE, dQ, dK, dV) lives inside a larger device buffer filled with a poison
byte: 4 KB of margin before and after, and, for the bf16 tensors, unused interleaved slots
between the rows of a strided view (the output is one slot of a [batch, tokens, slots,
heads, d] buffer). After each call the margins and the unused slots must still hold the
poison, bit for bit, and the outputs must match the oracle. The cases cover a tiny
sequence, a ragged last query tile (13 blocks of 32), rows without any key block, and the
32-token block with every head dimension. The checks run on the host after the kernels
finished; nothing here writes out of bounds on purpose.
"""
import numpy as np
import pytest

import content_adaptive_sparse_gb300 as sa
import oracle
from oracle import masks as om
from workloads import bf16_bits_to_f64, bf16_normal_bits
from gpu_helpers import assert_attention_close, assert_grad_close, bf16_to_f64, torch_cuda

pytestmark = pytest.mark.gpu

MARGIN = 4096
POISON = 0xA5


class Guarded:
    """A tensor of ``shape`` and ``dtype`` at byte offset MARGIN inside a poisoned buffer."""

    def __init__(self, shape, dtype):
        torch = torch_cuda()
        self.torch = torch
        n_el = int(np.prod(shape))
        esz = torch.tensor([], dtype=dtype).element_size()
        self.nbytes = n_el * esz
        self.raw = torch.full((MARGIN + self.nbytes + MARGIN,), POISON, dtype=torch.uint8, device="cuda")
        self.full = self.raw[MARGIN:MARGIN + self.nbytes].view(dtype).view(shape)

    def margins_intact(self) -> bool:
        h = self.raw.cpu().numpy()
        return bool(np.all(h[:MARGIN] == POISON) and np.all(h[MARGIN + self.nbytes:] == POISON))


def _poisoned_slots_intact(g: Guarded, used_slots) -> bool:
    """Every slot of dim 2 not in used_slots still holds the poison bytes."""
    torch = g.torch
    full = g.full
    for sl in range(full.shape[2]):
        if sl in used_slots:
            continue
        b = full[:, :, sl].contiguous().view(torch.uint8).cpu().numpy()
        if not np.all(b == POISON):
            return False
    return True


def _upload(bits, slots, slot, g: Guarded):
    """Write bf16 bits into slot ``slot`` of a guarded [bt, n, slots, h, d] buffer."""
    torch = g.torch
    g.full[:, :, slot] = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _case(bt, n, h, hkv, d, b, rows=None, causal=1, seed=0):
    """Forward and backward with every output guarded; returns nothing, asserts all."""
    torch = torch_cuda()
    rng = np.random.default_rng(seed)
    qb = bf16_normal_bits(rng, (bt, n, h, d), 0.4)
    kb = bf16_normal_bits(rng, (bt, n, hkv, d), 0.4)
    vb = bf16_normal_bits(rng, (bt, n, hkv, d), 0.4)
    dob = bf16_normal_bits(rng, (bt, n, h, d), 0.4)
    nb = n // b
    if rows is None:
        p = om.MaskParams("full", b, n, causal)
        rp, ci = om.build_csr(p, None, bt)
    else:
        rp = np.zeros((bt, nb + 1), dtype=np.int32)
        cols = []
        for s in range(bt):
            rp[s, 0] = len(cols)
            for I, row in enumerate(rows):
                cols += row
                rp[s, I + 1] = len(cols)
        ci = np.array(cols, dtype=np.int32)
    rp_d, ci_d = torch.from_numpy(rp).cuda(), torch.from_numpy(ci).cuda()

    # inputs: q in slot 0 of a 2-slot buffer, k / v in slots 0 / 1 of a 3-slot buffer
    qbuf = Guarded((bt, n, 2, h, d), torch.bfloat16)
    kvbuf = Guarded((bt, n, 3, hkv, d), torch.bfloat16)
    _upload(qb, 2, 0, qbuf)
    _upload(kb, 3, 0, kvbuf)
    _upload(vb, 3, 1, kvbuf)
    q, k, v = qbuf.full[:, :, 0], kvbuf.full[:, :, 0], kvbuf.full[:, :, 1]
    # outputs: O in slot 0 of a 2-slot buffer, LSE contiguous, both inside poison
    obuf = Guarded((bt, n, 2, h, d), torch.bfloat16)
    lbuf = Guarded((bt, h, n), torch.float32)
    o, lse = obuf.full[:, :, 0], lbuf.full
    sa.sa_attn_fwd(q, k, v, rp_d, ci_d, b, causal, o, lse)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    assert obuf.margins_intact() and _poisoned_slots_intact(obuf, {0}), "O written outside its view"
    assert lbuf.margins_intact(), "LSE written outside its buffer"
    f = bf16_bits_to_f64
    o_ref, lse_ref = oracle.attention_csr(f(qb), f(kb), f(vb), rp, ci, b, causal)
    assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, "guarded fwd")

    # backward: dO with O's strides; dQ with q's, dK / dV with k's (slots 0 / 1 of 3)
    dobuf = Guarded((bt, n, 2, h, d), torch.bfloat16)
    _upload(dob, 2, 0, dobuf)
    d_o = dobuf.full[:, :, 0]
    dqbuf = Guarded((bt, n, 2, h, d), torch.bfloat16)
    dkvbuf = Guarded((bt, n, 3, hkv, d), torch.bfloat16)
    dq, dk, dv = dqbuf.full[:, :, 0], dkvbuf.full[:, :, 0], dkvbuf.full[:, :, 1]
    cap = max(int(ci.size), 1)
    ws_bytes = sa.sa_attn_bwd_workspace_size(bt, n, h, b, bt, cap)
    wsbuf = Guarded((ws_bytes,), torch.uint8)
    sa.sa_attn_bwd(q, k, v, o, d_o, lse, rp_d, ci_d, b, causal, dq, dk, dv, wsbuf.full)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    assert dqbuf.margins_intact() and _poisoned_slots_intact(dqbuf, {0}), "dQ written outside its view"
    assert dkvbuf.margins_intact() and _poisoned_slots_intact(dkvbuf, {0, 1}), "dK / dV written outside"
    assert wsbuf.margins_intact(), "workspace written outside its size"
    rq, rk, rv = oracle.attention_csr_backward(f(qb), f(kb), f(vb), f(dob), rp, ci, b, causal)
    assert_grad_close(bf16_to_f64(dq), rq, "guarded dQ")
    assert_grad_close(bf16_to_f64(dk), rk, "guarded dK")
    assert_grad_close(bf16_to_f64(dv), rv, "guarded dV")


@pytest.mark.parametrize("d", [32, 64, 128])
def test_guard_tiny(d):
    _case(1, 256, 2, 2, d, 64, seed=d)


@pytest.mark.parametrize("d", [32, 64, 128])
def test_guard_ragged_tail_block32(d):
    # 13 blocks of 32: the last 128-row query tile holds one block
    _case(2, 416, 2, 1, d, 32, seed=100 + d)


def test_guard_empty_rows_bidirectional_gqa():
    rows = [[0], [], [0, 1], [2, 7], [], [1, 3, 5], [6], [0, 7]]
    _case(2, 256, 4, 2, 64, 32, rows=rows, causal=0, seed=7)


def test_guard_empty_rows_causal():
    rows = [[0], [], [0, 1], [2], [], [1, 3, 5], [6], [0, 7]]
    _case(1, 256, 2, 2, 64, 32, rows=rows, causal=1, seed=8)


@pytest.mark.parametrize("d", [64, 128])
def test_guard_keyless_query_tile(d):
    """The second 128-row query tile of every (sequence, head) has no key block at all (its
    four 32-token query blocks have empty rows): those items write zeros and -inf without key
    tiles, next to items that do have some (at d = 128 through the epilogue warps)."""
    rows = [[0], [0, 1], [], [2, 3], [], [], [], []]
    _case(2, 256, 4, 2, d, 32, rows=rows, causal=1, seed=11 + d)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("interp", [False, True])
def test_guard_offset_kernels(interp, d):
    """The window-plus-offset kernels (integer and interpolated) at every head dimension: O
    and LSE guarded, a length that is not a multiple of the 64- or 128-query tile."""
    torch = torch_cuda()
    rng = np.random.default_rng(5 + d)
    bt, n, h, hkv, W = 2, 1000, 2, 1, 8
    qb = bf16_normal_bits(rng, (bt, n, h, d), 0.4)
    kb = bf16_normal_bits(rng, (bt, n, hkv, d), 0.4)
    vb = bf16_normal_bits(rng, (bt, n, hkv, d), 0.4)
    dev = [torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.bfloat16) for x in (qb, kb, vb)]
    obuf = Guarded((bt, n, 2, h, d), torch.bfloat16)
    lbuf = Guarded((bt, h, n), torch.float32)
    o, lse = obuf.full[:, :, 0], lbuf.full
    f = bf16_bits_to_f64
    if interp:
        sa.sa_offset_attn_interp_fwd(dev[0], dev[1], dev[2], W, 0.8317, o, lse)
        o_ref, lse_ref = oracle.attention_offsets_interp(f(qb), f(kb), f(vb), W,
                                                         oracle.interp_rungs(0.8317, oracle.fib_rungs(15), W))
    else:
        sa.sa_offset_attn_fwd(dev[0], dev[1], dev[2], W, 7, 10, 15, o, lse)
        from fractions import Fraction
        o_ref, lse_ref = oracle.attention_offsets(f(qb), f(kb), f(vb), W,
                                                  oracle.fib_offsets(Fraction(7, 10), oracle.fib_rungs(15)))
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    assert obuf.margins_intact() and _poisoned_slots_intact(obuf, {0}), "O written outside its view"
    assert lbuf.margins_intact(), "LSE written outside its buffer"
    assert_attention_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                           f"guarded offsets d={d}")
