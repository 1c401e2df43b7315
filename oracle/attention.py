"""Attention restricted to a key set, in float64.

For query i with allowed key set S(i) (from a CSR row or an offset set) and scale c
(default 1/sqrt(d), as in the [BB] section 3 sketch which divides scores by d**0.5):

    s_ij   = c * sum_t q_it k_jt                       (j in S(i))
    LSE_i  = m_i + ln sum_{j in S(i)} exp(s_ij - m_i),  m_i = max_j s_ij
    O_i    = sum_{j in S(i)} exp(s_ij - LSE_i) v_j

An empty key set gives O_i = 0 and LSE_i = -inf. Inputs are float64 arrays with layout
[batch, tokens, heads, d]; query head h reads key/value head h // (H / H_kv).
Outputs: O [batch, tokens, heads, d] and LSE [batch, heads, tokens] (natural log).
"""
from __future__ import annotations

import numpy as np


def _softmax_rows(s: np.ndarray):
    """Row-wise exact softmax of a score matrix whose masked entries are -inf."""
    m = np.max(s, axis=1, keepdims=True) if s.shape[1] else np.full((s.shape[0], 1), -np.inf)
    empty = ~np.isfinite(m[:, 0])
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe)
    tot = e.sum(axis=1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(tot > 0, e / np.where(tot > 0, tot, 1.0), 0.0)
        lse = np.where(empty, -np.inf, m_safe[:, 0] + np.log(np.where(tot[:, 0] > 0, tot[:, 0], 1.0)))
    return p, lse


def _csr_batch(row_ptr, s):
    return s if row_ptr.shape[0] > 1 else 0


def attention_csr_block(q, k, v, row_ptr, col_idx, block: int, causal: int, s: int, I: int, hh: int,
                        scale: float | None = None, convert=None):
    """One query block I of sequence s and head hh: returns O [block, d] and LSE [block].

    ``convert`` (optional) widens gathered rows to float64 (e.g. from bf16 bit patterns).
    """
    cv = convert if convert is not None else (lambda x: x)
    d = q.shape[3]
    h, hkv = q.shape[2], k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    cs = _csr_batch(row_ptr, s)
    row = col_idx[row_ptr[cs, I]:row_ptr[cs, I + 1]]
    if len(row) == 0:
        return np.zeros((block, d)), np.full(block, -np.inf)
    keys = np.concatenate([np.arange(J * block, (J + 1) * block) for J in row])
    qi = np.arange(I * block, (I + 1) * block)
    allowed = keys[None, :] <= qi[:, None] if causal else np.ones((block, len(keys)), dtype=bool)
    hk = hh // (h // hkv)
    sc = (cv(q[s, qi, hh, :]) @ cv(k[s, keys, hk, :]).T) * scale
    sc = np.where(allowed, sc, -np.inf)
    p, l = _softmax_rows(sc)
    return p @ cv(v[s, keys, hk, :]), l


def attention_csr(q, k, v, row_ptr, col_idx, block: int, causal: int, scale: float | None = None):
    """Block-CSR attention for every query; see module docstring."""
    bt, n, h, d = q.shape
    nb = n // block
    o = np.zeros((bt, n, h, d), dtype=np.float64)
    lse = np.full((bt, h, n), -np.inf, dtype=np.float64)
    for s in range(bt):
        for I in range(nb):
            for hh in range(h):
                ob, lb = attention_csr_block(q, k, v, row_ptr, col_idx, block, causal, s, I, hh, scale)
                o[s, I * block:(I + 1) * block, hh, :] = ob
                lse[s, hh, I * block:(I + 1) * block] = lb
    return o, lse


def attention_csr_heads(q, k, v, csrs, head_mask, block: int, causal: int, scale: float | None = None):
    """Block-CSR attention where query head h uses CSR ``csrs[head_mask[h]]`` (a list of
    (row_ptr, col_idx) pairs), as in [CAS] Appendix B "Head-specific mask distribution"
    (head groups with different parts of the block mask)."""
    bt, n, h, d = q.shape
    nb = n // block
    o = np.zeros((bt, n, h, d), dtype=np.float64)
    lse = np.full((bt, h, n), -np.inf, dtype=np.float64)
    for s in range(bt):
        for I in range(nb):
            for hh in range(h):
                row_ptr, col_idx = csrs[head_mask[hh]]
                ob, lb = attention_csr_block(q, k, v, row_ptr, col_idx, block, causal, s, I, hh, scale)
                o[s, I * block:(I + 1) * block, hh, :] = ob
                lse[s, hh, I * block:(I + 1) * block] = lb
    return o, lse


def attention_rows_csr(q, k, v, row_ptr, col_idx, block: int, causal: int, samples,
                       scale: float | None = None, convert=None):
    """The same definition evaluated only at sampled (batch, token, head) triples.

    ``convert`` (optional) widens gathered rows to float64 (e.g. from bf16 bit
    patterns), so that large inputs need not be converted as a whole.
    Returns ``o [len(samples), d]`` and ``lse [len(samples)]``.
    """
    cv = convert if convert is not None else (lambda x: x)
    d = q.shape[3]
    h = q.shape[2]
    hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.zeros((len(samples), d))
    lse = np.full(len(samples), -np.inf)
    for t, (s, i, hh) in enumerate(samples):
        cs = _csr_batch(row_ptr, s)
        I = i // block
        row = col_idx[row_ptr[cs, I]:row_ptr[cs, I + 1]]
        keys = [j for J in row for j in range(J * block, (J + 1) * block) if not causal or j <= i]
        if not keys:
            continue
        hk = hh // (h // hkv)
        sc = (cv(k[s, keys, hk, :]) @ cv(q[s, i, hh, :])) * scale
        p, l = _softmax_rows(sc[None, :])
        o[t] = p[0] @ cv(v[s, keys, hk, :])
        lse[t] = l[0]
    return o, lse


def attention_offsets(q, k, v, window: int, offsets, scale: float | None = None,
                      samples=None, convert=None):
    """Token-granular window-plus-offset attention ([FIB] section 2 "Attended set").

    Key set of query i: {i - delta : delta in {0..window} u offsets, i - delta >= 0},
    deduplicated. If ``samples`` (list of (batch, token, head)) is given, only those
    queries are evaluated and ``o [len, d]``, ``lse [len]`` are returned.
    """
    bt, n, h, d = q.shape
    hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    deltas = np.array(sorted(set(range(window + 1)) | {int(x) for x in offsets}), dtype=np.int64)
    cv = convert if convert is not None else (lambda x: x)
    if samples is not None:
        o = np.zeros((len(samples), d))
        lse = np.full(len(samples), -np.inf)
        for t, (s, i, hh) in enumerate(samples):
            keys = i - deltas[deltas <= i]
            hk = hh // (h // hkv)
            sc = (cv(k[s, keys, hk, :]) @ cv(q[s, i, hh, :])) * scale
            p, l = _softmax_rows(sc[None, :])
            o[t] = p[0] @ cv(v[s, keys, hk, :])
            lse[t] = l[0]
        return o, lse
    o = np.zeros((bt, n, h, d))
    lse = np.full((bt, h, n), -np.inf)
    idx = np.arange(n)[:, None] - deltas[None, :]          # [n, n_delta] key index
    valid = idx >= 0
    idx_c = np.where(valid, idx, 0)
    for s in range(bt):
        for hh in range(h):
            hk = hh // (h // hkv)
            kk = k[s, :, hk, :][idx_c]                       # [n, n_delta, d]
            sc = np.einsum("nd,nkd->nk", q[s, :, hh, :], kk) * scale
            sc = np.where(valid, sc, -np.inf)
            p, l = _softmax_rows(sc)
            o[s, :, hh, :] = np.einsum("nk,nkd->nd", p, v[s, :, hk, :][idx_c])
            lse[s, hh, :] = l
    return o, lse


def dense_masked_attention(q, k, v, token_mask: np.ndarray, scale: float | None = None):
    """Second route: full N x N scores, masked fill with -inf, softmax, times V.

    This is the dense formulation both [CAS] (section 5 "Limitations": the mask is
    applied to the materialised N x N matrix) and the [BB] section 3 sketch use.
    ``token_mask`` is bool [N, N] (shared over batch and heads).
    """
    bt, n, h, d = q.shape
    hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.zeros((bt, n, h, d))
    lse = np.full((bt, h, n), -np.inf)
    for s in range(bt):
        for hh in range(h):
            hk = hh // (h // hkv)
            sc = (q[s, :, hh, :] @ k[s, :, hk, :].T) * scale
            sc = np.where(token_mask, sc, -np.inf)
            p, l = _softmax_rows(sc)
            o[s, :, hh, :] = p @ v[s, :, hk, :]
            lse[s, hh, :] = l
    return o, lse


def attention_csr_backward(q, k, v, d_o, row_ptr, col_idx, block: int, causal: int, scale: float | None = None,
                           convert=None):
    """Gradients of L = sum(dO * O) for block-CSR attention, from the definitions.

    For query i with allowed keys S(i) (same token rule as ``attention_csr``):
        P_ij   = exp(s_ij - LSE_i)
        dV_j  += sum_i P_ij dO_i
        dP_ij  = <dO_i, v_j>
        dS_ij  = P_ij (dP_ij - sum_{l in S(i)} P_il dP_il)
        dQ_i   = scale * sum_j dS_ij k_j
        dK_j  += scale * sum_i dS_ij q_i
    With grouped-query attention, dK / dV of a key/value head sum over the query heads
    that read it. Returns dq [batch, tokens, heads, d], dk and dv [batch, tokens,
    kv_heads, d], float64.
    """
    cv = convert if convert is not None else (lambda x: x)
    bt, n, h, d = q.shape
    hkv = k.shape[2]
    nb = n // block
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.zeros((bt, n, h, d))
    dk = np.zeros((bt, n, hkv, d))
    dv = np.zeros((bt, n, hkv, d))
    for s in range(bt):
        cs = _csr_batch(row_ptr, s)
        for I in range(nb):
            row = col_idx[row_ptr[cs, I]:row_ptr[cs, I + 1]]
            if len(row) == 0:
                continue
            keys = np.concatenate([np.arange(J * block, (J + 1) * block) for J in row])
            qi = np.arange(I * block, (I + 1) * block)
            allowed = keys[None, :] <= qi[:, None] if causal else np.ones((block, len(keys)), dtype=bool)
            for hh in range(h):
                hk = hh // (h // hkv)
                Q = cv(q[s, qi, hh, :])
                K = cv(k[s, keys, hk, :])
                V = cv(v[s, keys, hk, :])
                dO = cv(d_o[s, qi, hh, :])
                sc = np.where(allowed, (Q @ K.T) * scale, -np.inf)
                P, _ = _softmax_rows(sc)
                dP = dO @ V.T
                dS = P * (dP - np.sum(P * dP, axis=1, keepdims=True))
                dq[s, qi, hh, :] += scale * (dS @ K)
                np.add.at(dk[s, :, hk, :], keys, scale * (dS.T @ Q))
                np.add.at(dv[s, :, hk, :], keys, P.T @ dO)
    return dq, dk, dv


def attention_rows_dq(q, k, v, d_o, row_ptr, col_idx, block: int, causal: int, samples,
                      scale: float | None = None, convert=None):
    """dQ_i of the backward above at sampled (batch, token, head) triples."""
    cv = convert if convert is not None else (lambda x: x)
    d = q.shape[3]
    h, hkv = q.shape[2], k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((len(samples), d))
    for t, (s, i, hh) in enumerate(samples):
        cs = _csr_batch(row_ptr, s)
        I = i // block
        row = col_idx[row_ptr[cs, I]:row_ptr[cs, I + 1]]
        keys = [j for J in row for j in range(J * block, (J + 1) * block) if not causal or j <= i]
        if not keys:
            continue
        hk = hh // (h // hkv)
        K = cv(k[s, keys, hk, :])
        V = cv(v[s, keys, hk, :])
        P, _ = _softmax_rows(((K @ cv(q[s, i, hh, :])) * scale)[None, :])
        dP = V @ cv(d_o[s, i, hh, :])
        dS = P[0] * (dP - np.sum(P[0] * dP))
        out[t] = scale * (dS @ K)
    return out


def attention_rows_dkdv(q, k, v, d_o, row_ptr, col_idx, block: int, causal: int, samples,
                        scale: float | None = None, convert=None):
    """dK_j and dV_j of the backward above at sampled (batch, token, kv head) triples:
    sums over every query (of every query head of the group) whose key set holds j."""
    cv = convert if convert is not None else (lambda x: x)
    n, h, d = q.shape[1], q.shape[2], q.shape[3]
    hkv = k.shape[2]
    nb = n // block
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dk = np.zeros((len(samples), d))
    dv = np.zeros((len(samples), d))
    for t, (s, j, hk) in enumerate(samples):
        cs = _csr_batch(row_ptr, s)
        J = j // block
        q_blocks = [I for I in range(nb) if J in set(col_idx[row_ptr[cs, I]:row_ptr[cs, I + 1]].tolist())]
        for I in q_blocks:
            row = col_idx[row_ptr[cs, I]:row_ptr[cs, I + 1]]
            for i in range(I * block, (I + 1) * block):
                if causal and j > i:
                    continue
                keys = [x for Jr in row for x in range(Jr * block, (Jr + 1) * block) if not causal or x <= i]
                pos = keys.index(j)
                for hh in range(hk * (h // hkv), (hk + 1) * (h // hkv)):
                    K = cv(k[s, keys, hk, :])
                    V = cv(v[s, keys, hk, :])
                    qv = cv(q[s, i, hh, :])
                    dov = cv(d_o[s, i, hh, :])
                    P, _ = _softmax_rows(((K @ qv) * scale)[None, :])
                    dP = V @ dov
                    dS = P[0] * (dP - np.sum(P[0] * dP))
                    dk[t] += scale * dS[pos] * qv
                    dv[t] += P[0][pos] * dov
    return dk, dv


def attention_offsets_interp(q, k, v, window: int, rungs_lo_t, scale: float | None = None, samples=None,
                             convert=None):
    """Window plus interpolated-rung attention ([FIB] section 2, the interpolated gather).

    Entries of query i: the window rows i - delta (delta = 0..W, i - delta >= 0) and, for
    every rung (lo, t) with i - lo - t >= 0, the interpolated key and value
        k~ = (1 - t) k[i - lo] + t k[i - lo - 1],   v~ likewise (t = 0: row i - lo).
    Softmax over all entries with s = scale <q_i, k~>. ``rungs_lo_t`` as returned by
    ``fib.interp_rungs``. If ``samples`` (list of (batch, token, head)) is given only those
    queries are evaluated; returns o [len, d], lse [len]; else o [B, N, H, d], lse [B, H, N].
    """
    cv = convert if convert is not None else (lambda x: x)
    bt, n, h, d = q.shape
    hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if samples is None:
        samples = [(s, i, hh) for s in range(bt) for i in range(n) for hh in range(h)]
        full = True
    else:
        full = False
    o = np.zeros((len(samples), d))
    lse = np.full(len(samples), -np.inf)
    for t_idx, (s, i, hh) in enumerate(samples):
        hk = hh // (h // hkv)
        keys, vals = [], []
        for delta in range(window + 1):
            if i - delta >= 0:
                keys.append(cv(k[s, i - delta, hk, :]))
                vals.append(cv(v[s, i - delta, hk, :]))
        for lo, t in rungs_lo_t:
            if i - lo - t < 0:
                continue
            if t == 0.0:
                keys.append(cv(k[s, i - lo, hk, :]))
                vals.append(cv(v[s, i - lo, hk, :]))
            else:
                keys.append((1.0 - t) * cv(k[s, i - lo, hk, :]) + t * cv(k[s, i - lo - 1, hk, :]))
                vals.append((1.0 - t) * cv(v[s, i - lo, hk, :]) + t * cv(v[s, i - lo - 1, hk, :]))
        K = np.stack(keys)
        V = np.stack(vals)
        sc = (K @ cv(q[s, i, hh, :])) * scale
        p, l = _softmax_rows(sc[None, :])
        o[t_idx] = p[0] @ V
        lse[t_idx] = l[0]
    if not full:
        return o, lse
    return o.reshape(bt, n, h, d), lse.reshape(bt, n, h).transpose(0, 2, 1)


def attention_csr_backward_heads(q, k, v, d_o, csrs, head_mask, block: int, causal: int,
                                 scale: float | None = None):
    """Backward of ``attention_csr_heads``: query head h uses CSR ``csrs[head_mask[h]]``;
    dK / dV of a key/value head sum over its query heads (each with its own CSR)."""
    bt, n, h, d = q.shape
    hkv = k.shape[2]
    g = h // hkv
    dq = np.zeros((bt, n, h, d))
    dk = np.zeros((bt, n, hkv, d))
    dv = np.zeros((bt, n, hkv, d))
    for hh in range(h):
        hk = hh // g
        rp, ci = csrs[head_mask[hh]]
        a, b_, c = attention_csr_backward(q[:, :, hh:hh + 1], k[:, :, hk:hk + 1], v[:, :, hk:hk + 1],
                                          d_o[:, :, hh:hh + 1], rp, ci, block, causal, scale)
        dq[:, :, hh] = a[:, :, 0]
        dk[:, :, hk] += b_[:, :, 0]
        dv[:, :, hk] += c[:, :, 0]
    return dq, dk, dv
