"""Block-sparse key graphs as CSR lists of key blocks per query block.

Notation: block size b, nb = N / b blocks, I = query block, J = key block. A row is
the ascending list of key blocks that query block I may attend to; a token pair
(i, j) is an edge iff blk(j) is in row(blk(i)) and, when causal, j <= i ([CAS]
section 3.2 last paragraph and section 3.4 "Block-to-token expansion").

Modes
-----
* ``topk``  compression-guided, causal. For query block I with window w (counting the
  diagonal block), g global key blocks and k literal blocks:
      W(I) = {J : max(0, I-w+1) <= J <= I}
      G(I) = {J < g : J <= I} minus W(I)
      C(I) = {J : 0 <= J <= I} minus (W(I) u G(I))
      L(I) = the first min(k, |C(I)|) of C(I) ordered by ratio descending, then J
             ascending
      row(I) = W u G u L
  Readings (the top-k rule comes from the workload statement; [CAS] itself uses the
  mean threshold of ``literal_mean``): the window counts the diagonal block, literal
  candidates exclude window and global blocks ([CAS] Eq. 3 keeps literal edges at
  |i-j| > w), ties go to the smaller block index, global blocks are key columns only
  under causality.
* ``literal_mean``  [CAS] section 3.1 Eq. 2 and section 3.2 Eq. 3 / Algorithm 1:
  l_i = [r_i > mean(r)], M = M_lit u M_local u I with M_lit(i,j) = l_i l_j [|i-j| > w]
  and M_local(i,j) = [|i-j| <= w]; causal keeps J <= I. ``components`` selects the
  parts [CAS] Appendix B "Head-specific mask distribution" hands to head groups:
  LOCAL (M_local u I), LITERAL (M_lit u I) or both (the full M; 0 means both).
* ``bigbird``  [BB] section 2: window of w_b consecutive blocks placed as
  [I - w_b//2, I - w_b//2 + w_b - 1] (reading: an even window cannot be centred, this
  placement gives exactly w tokens), g global blocks (global rows attend to every
  block, every row attends to the global blocks) and r_b random blocks per
  non-global row drawn without replacement from the blocks outside window and
  globals. Draw t of row I uses Philox word I*r_b + t and picks index
  ((x >> 32) * |A|) >> 32 of the remaining ascending candidate list A.
  Bidirectional only ([BB] section 4: the construction is encoder-only).
* ``full``  every block J <= I (causal) or every block (bidirectional).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from .philox import philox_word


@dataclass(frozen=True)
class MaskParams:
    mode: str                 # "topk" | "bigbird" | "full" | "literal_mean"
    block: int
    n_tokens: int
    causal: int = 1
    window_blocks: int = 0
    global_blocks: int = 0
    topk: int = 0
    random_blocks: int = 0
    seed: int = 0
    components: int = 0       # literal_mean only: LOCAL | LITERAL, 0 = both


    @property
    def nb(self) -> int:
        return self.n_tokens // self.block


# ---------------------------------------------------------------- topk (causal)

def csr_topk_rows(ratios, w: int, g: int, k: int) -> list[list[int]]:
    nb = len(ratios)
    rows = []
    for I in range(nb):
        W = set(range(max(0, I - w + 1), I + 1))
        G = {J for J in range(min(g, nb)) if J <= I} - W
        C = [J for J in range(I + 1) if J not in W and J not in G]
        C.sort(key=lambda J: (-float(ratios[J]), J))
        L = set(C[:min(k, len(C))])
        rows.append(sorted(W | G | L))
    return rows


def topk_row_count(I: int, w: int, g: int, k: int) -> int:
    """Closed form |W(I)| + |G(I)| + min(k, |C(I)|) (independent of the ratios)."""
    n_w = min(w, I + 1)
    n_g = max(0, min(g, I - w + 1))
    n_c = max(0, I - w + 1 - g)
    return n_w + n_g + min(k, n_c)


# ---------------------------------------------------------------- literal_mean

LOCAL, LITERAL = 1, 2          # components of the [CAS] block mask besides the identity

def literal_flags(ratios) -> list[bool]:
    """[CAS] Eq. 2: l_i = 1 iff r_i > mean(r) (mean over all B blocks)."""
    r = [float(x) for x in ratios]
    mean = math.fsum(r) / len(r)
    return [x > mean for x in r]


def csr_literal_mean_rows(ratios, w: int, causal: int, components: int = 0) -> list[list[int]]:
    nb = len(ratios)
    lit = literal_flags(ratios)
    comp = components or (LOCAL | LITERAL)
    rows = []
    for I in range(nb):
        row = []
        for J in range(nb):
            if causal and J > I:
                continue
            local = bool(comp & LOCAL) and abs(I - J) <= w
            ident = I == J
            literal = bool(comp & LITERAL) and lit[I] and lit[J] and abs(I - J) > w
            if local or ident or literal:
                row.append(J)
        rows.append(row)
    return rows


# ---------------------------------------------------------------- bigbird

def bigbird_window(I: int, wb: int, nb: int) -> list[int]:
    lo = I - wb // 2
    return [J for J in range(lo, lo + wb) if 0 <= J < nb]


def csr_bigbird_rows(nb: int, wb: int, g: int, rb: int, seed: int) -> list[list[int]]:
    rows = []
    for I in range(nb):
        if I < g:
            rows.append(list(range(nb)))
            continue
        W = set(bigbird_window(I, wb, nb))
        G = set(range(min(g, nb)))
        A = [J for J in range(nb) if J not in W and J not in G]
        R = []
        for t in range(min(rb, len(A))):
            x = philox_word(seed, I * rb + t)
            idx = ((x >> 32) * len(A)) >> 32
            R.append(A.pop(idx))
        rows.append(sorted(W | G | set(R)))
    return rows


# ---------------------------------------------------------------- full

def csr_full_rows(nb: int, causal: int) -> list[list[int]]:
    return [list(range(I + 1)) if causal else list(range(nb)) for I in range(nb)]


# ---------------------------------------------------------------- CSR assembly

def _rows_for(p: MaskParams, ratios_row):
    nb = p.nb
    if p.mode == "topk":
        if not p.causal:
            raise ValueError("topk mode is causal only")
        return csr_topk_rows(ratios_row, p.window_blocks, p.global_blocks, p.topk)
    if p.mode == "literal_mean":
        return csr_literal_mean_rows(ratios_row, p.window_blocks, p.causal, p.components)
    if p.mode == "bigbird":
        if p.causal:
            raise ValueError("bigbird mode is bidirectional only")
        return csr_bigbird_rows(nb, p.window_blocks, p.global_blocks, p.random_blocks, p.seed)
    if p.mode == "full":
        return csr_full_rows(nb, p.causal)
    raise ValueError(p.mode)


def build_csr(p: MaskParams, ratios=None, batch: int = 1):
    """CSR for ``batch`` sequences.

    Returns ``row_ptr int32[batch, nb+1]`` (absolute offsets into ``col_idx``; batch
    s starts where batch s-1 ends) and ``col_idx int32[nnz]``.
    """
    nb = p.nb
    row_ptr = np.zeros((batch, nb + 1), dtype=np.int64)
    cols = []
    base = 0
    for s in range(batch):
        rr = None if ratios is None else np.asarray(ratios)[s]
        rows = _rows_for(p, rr)
        row_ptr[s, 0] = base
        for I, row in enumerate(rows):
            cols.extend(row)
            base += len(row)
            row_ptr[s, I + 1] = base
    return row_ptr.astype(np.int32), np.asarray(cols, dtype=np.int32)


def csr_to_block_mask(row_ptr, col_idx, nb: int, s: int = 0) -> np.ndarray:
    m = np.zeros((nb, nb), dtype=bool)
    for I in range(nb):
        for t in range(row_ptr[s, I], row_ptr[s, I + 1]):
            m[I, col_idx[t]] = True
    return m


def block_mask_to_token_mask(block_mask: np.ndarray, block: int, causal: int) -> np.ndarray:
    """[CAS] section 3.4: M'[i, j] = M[i // b, j // b], intersected with j <= i if causal."""
    tok = np.repeat(np.repeat(block_mask, block, axis=0), block, axis=1)
    if causal:
        n = tok.shape[0]
        tok &= np.tril(np.ones((n, n), dtype=bool))
    return tok


# ---------------------------------------------------------------- head groups

def cas_head_components(heads: int) -> list[int]:
    """[CAS] Appendix B "Head-specific mask distribution": of 12 heads, heads 0-5 get
    the local part, heads 6-8 the literal (long-range) part and heads 9-11 the full
    mask. Reading for other head counts: the same proportions, first half local, next
    quarter literal, the rest full (12 heads give exactly the page's split)."""
    n_local = heads // 2
    n_lit = heads // 4
    return [LOCAL if h < n_local else LITERAL if h < n_local + n_lit else LOCAL | LITERAL
            for h in range(heads)]
