"""Float64 oracle of the full-sum loss over a generic FSA (test infrastructure only).

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU baseline leg of ``bench.py`` may import this module; it shares no
code with the CUDA library.

Page "feat(asr): native CTC loss kernel over sequence-packed log
probabilities", ctc_loss.py, module docstring: the packed CTC loss descends
from RETURNN's packed full-sum loss over a generic FSA edge list (scores
addressed in the token-flat buffer through per-sequence start offsets, the
gradient ``exp(log_probs) - posterior`` masked per frame); the CTC topology
is the special case built into the recursion.  This module states that
generic form plainly.

Sequence b has ``S_b`` states (local ids ``0 .. S_b - 1``), a log start
weight and a log final weight per state (``-inf``: not a start / final
state), and edges ``(from, to, label, weight)``; every edge consumes exactly
one frame (no epsilon edges).  With ``lp`` the rows of sequence b:

    alpha_0(s)       = start(s)
    alpha_{t+1}(s')  = logsumexp over edges e = (s, s', c, w) of alpha_t(s) + w + lp[t, c]
    Z_b              = logsumexp_s alpha_{T_b}(s) + final(s)
    loss_b           = -Z_b                       (+inf when no path exists)

    beta_{T_b}(s)    = final(s)
    beta_t(s)        = logsumexp over edges e = (s, s', c, w) of w + lp[t, c] + beta_{t+1}(s')
    occupancy_t(e)   = exp(alpha_t(s) + w + lp[t, c] + beta_{t+1}(s') - Z_b)
    grad[t, c]       = scale_b * (exp(lp[t, c]) - sum over edges e with label c of occupancy_t(e))

The gradient follows the page's convention: ``exp(lp) - posterior``, the
gradient with respect to the logits of a log_softmax.  ``scale_b`` is the
upstream gradient of sequence b, 0 when ``zero_infinity`` meets an
infinite loss (which is then reported as 0).  Rows outside every sequence
get 0.
"""

from __future__ import annotations

from typing import Sequence

import numpy as np


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        return np.ascontiguousarray(x.detach().cpu().double().numpy())
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _logsumexp(v: np.ndarray) -> float:
    if v.size == 0:
        return -np.inf
    m = np.max(v)
    if m == -np.inf:
        return -np.inf
    return float(m + np.log(np.sum(np.exp(v - m))))


def fsa_sequence(lp: np.ndarray, start: np.ndarray, final: np.ndarray, edges: np.ndarray, weights: np.ndarray,
                 scale: float, zero_infinity: bool):
    """Loss and gradient rows of one sequence.  ``lp`` (T, D) float64,
    ``start`` / ``final`` (S,), ``edges`` (E, 3) int (from, to, label),
    ``weights`` (E,).  Returns ``(loss, grad (T, D))``."""
    T, D = lp.shape
    S = start.shape[0]
    fr, to, lab = (edges[:, 0], edges[:, 1], edges[:, 2]) if edges.size else (np.zeros(0, int),) * 3
    alpha = np.full((T + 1, S), -np.inf)
    alpha[0] = start
    for t in range(T):
        v = alpha[t][fr] + weights + lp[t, lab]
        nxt = np.full(S, -np.inf)
        np.logaddexp.at(nxt, to, v)
        alpha[t + 1] = nxt
    Z = _logsumexp(alpha[T] + final)
    grad = np.zeros((T, D))
    if np.isnan(Z):  # a NaN score anywhere on the lattice (as a NaN log probability gives torch's CTC loss)
        return np.nan, np.full((T, D), np.nan)
    if not np.isfinite(Z):
        if zero_infinity:
            return 0.0, grad
        return np.inf, None  # no path: the loss is +inf and the gradient is undefined
    beta = np.full((T + 1, S), -np.inf)
    beta[T] = final
    for t in range(T - 1, -1, -1):
        v = weights + lp[t, lab] + beta[t + 1][to]
        cur = np.full(S, -np.inf)
        np.logaddexp.at(cur, fr, v)
        beta[t] = cur
    for t in range(T):
        occ = np.exp(alpha[t][fr] + weights + lp[t, lab] + beta[t + 1][to] - Z)
        post = np.zeros(D)
        np.add.at(post, lab, occ)
        grad[t] = scale * (np.exp(lp[t]) - post)
    return -Z, grad


def fsa_loss_packed(log_probs, cu_seqlens, lengths, state_offsets, start_weight, final_weight, edge_offsets,
                    edges, edge_weight, grad_loss=None, zero_infinity: bool = False):
    """Per-sequence losses ``(B,)`` and the gradient ``(T_total, D)`` of the
    packed FSA full-sum (see the module docstring).  ``edges`` holds
    ``(from, to, label)`` rows with state ids local to their sequence;
    sequence b owns states ``state_offsets[b] .. state_offsets[b+1]`` of the
    weight arrays and edges ``edge_offsets[b] .. edge_offsets[b+1]``.
    Gradient rows of a sequence with an infinite loss and no
    ``zero_infinity`` are left NaN (undefined)."""
    lp = _f64(log_probs)
    cu, ln = _i64(cu_seqlens), _i64(lengths)
    so, eo = _i64(state_offsets), _i64(edge_offsets)
    sw, fw = _f64(start_weight), _f64(final_weight)
    ed = _i64(edges).reshape(-1, 3)
    ew = _f64(edge_weight).reshape(-1)
    B = ln.shape[0]
    g = np.ones(B) if grad_loss is None else _f64(grad_loss).reshape(B)
    loss = np.zeros(B)
    grad = np.zeros_like(lp)
    for b in range(B):
        rows = slice(int(cu[b]), int(cu[b]) + int(ln[b]))
        st = slice(int(so[b]), int(so[b + 1]))
        es = slice(int(eo[b]), int(eo[b + 1]))
        l, gr = fsa_sequence(lp[rows], sw[st], fw[st], ed[es], ew[es], float(g[b]), zero_infinity)
        loss[b] = l
        if gr is None:
            grad[rows] = np.nan
        else:
            grad[rows] = gr
    return loss, grad


def ctc_topology(targets: Sequence[int], blank: int):
    """The CTC lattice of one target sequence as an FSA: states
    ``0 .. 2U`` of the extended labels ``blank, l_1, blank, ..., l_U,
    blank``; a state's edge into itself, into the next state, and a skip over
    a blank between two different labels, each edge carrying the class of the
    state it enters; start in the virtual state before frame 0 (a state
    ``2U + 1`` with edges into states 0 and 1), final in the last two states.
    Returns ``(start, final, edges, weights)``."""
    U = len(targets)
    S = 2 * U + 1
    ext = [blank if s % 2 == 0 else int(targets[(s - 1) // 2]) for s in range(S)]
    pre = S  # the state before the first frame
    edges = []
    for s in range(S):
        edges.append((s, s, ext[s]))
        if s + 1 < S:
            edges.append((s, s + 1, ext[s + 1]))
        if s + 2 < S and s % 2 == 1 and ext[s + 2] != ext[s]:
            edges.append((s, s + 2, ext[s + 2]))
    edges.append((pre, 0, ext[0]))
    if S > 1:
        edges.append((pre, 1, ext[1]))
    start = np.full(S + 1, -np.inf)
    start[pre] = 0.0
    final = np.full(S + 1, -np.inf)
    final[S - 1] = 0.0
    if S > 1:
        final[S - 2] = 0.0
    # with no frames the path ends where it starts: only an empty target has one
    if U == 0:
        final[pre] = 0.0
    return start, final, np.array(edges, dtype=np.int64), np.zeros(len(edges))
