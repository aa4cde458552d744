"""Seeded synthetic inputs for the packed CTC loss.

This module only draws inputs: utterance lengths, target sequences and
log-softmax log probabilities laid out token-flat.  It holds none of the
CTC arithmetic, so both the fp64 oracle and the CUDA path can be fed the
very same batch.

The five named workloads follow the shapes, sizes and value distributions
of the packed-CTC benchmark configurations:

* ``tiny``      -- 4 utterances, T=[50,37,64,20], D=32, U=[10,8,12,4], fp32
* ``conformer`` -- 32 utterances, T~U[200,400], D=1025, U~U[T/6,T/4],
                   10% forced adjacent repeats, N(0,3^2) logits, bf16, mean
* ``longform``  -- 8 utterances, T~U[1500,2000], D=1025, U~U[T/4,T/3], fp32,
                   plus one infeasible all-repeat utterance, zero_infinity, sum
* ``char``      -- 256 utterances, T~U[100,1000], D=29, U~U[T/8,T/3],
                   20% forced adjacent repeats, fp16, mean
* ``largevocab``-- 64 utterances, T~U[400,800], D=8193, U~U[T/8,T/4],
                   N(0,3^2) logits, bf16, none

Readings of the distribution wording (the same for every workload):
"uniform in [a, b]" draws integers with both ends included; ``U ~ U[T/k, T/m]``
draws from ``[ceil(T/k), floor(T/m)]``; "x% forced adjacent repeats" lets each
target position i >= 1 copy position i-1 with probability x, and a sequence
that this makes infeasible (T < U + repeats) is drawn again.  Logits are
float32 N(0, sigma^2), the log-softmax is taken in float32 and then cast.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch

__all__ = ["Batch", "WORKLOADS", "make_batch", "workload", "padded_targets", "select_utterances"]


@dataclasses.dataclass
class Batch:
    """One packed batch: metadata on the CPU, log probabilities on the device
    they were drawn on.

    ``log_probs`` is ``(T_total, D)``; utterance ``b`` owns rows
    ``[cu_seqlens[b], cu_seqlens[b] + lengths[b])``.  ``targets`` holds the
    target sequences concatenated (``sum(target_lengths)`` int32 entries).
    """

    name: str
    log_probs: torch.Tensor
    cu_seqlens: torch.Tensor
    lengths: torch.Tensor
    targets: torch.Tensor
    target_lengths: torch.Tensor
    blank: int
    zero_infinity: bool
    reduction: str
    max_target_len: int

    @property
    def B(self) -> int:
        return int(self.lengths.numel())

    @property
    def D(self) -> int:
        return int(self.log_probs.shape[1])

    @property
    def T_total(self) -> int:
        return int(self.log_probs.shape[0])

    @property
    def frames(self) -> int:
        return int(self.lengths.sum())


def _uniform_int(gen: torch.Generator, lo: int, hi: int) -> int:
    """Integer uniform on [lo, hi], both ends included."""
    return int(torch.randint(lo, hi + 1, (1,), generator=gen).item())


def _draw_targets(gen, length, lo, hi, repeat_prob):
    labels = torch.randint(lo, hi + 1, (length,), generator=gen)
    if repeat_prob > 0 and length > 1:
        copy = torch.rand(length, generator=gen) < repeat_prob
        for i in range(1, length):
            if copy[i]:
                labels[i] = labels[i - 1]
    return labels


def _adjacent_repeats(labels: torch.Tensor) -> int:
    if labels.numel() < 2:
        return 0
    return int((labels[1:] == labels[:-1]).sum())


def make_batch(
    lengths: Sequence[int],
    target_lengths: Sequence[int],
    num_classes: int,
    *,
    dtype: torch.dtype = torch.float32,
    seed: int = 0,
    sigma: float = 2.0,
    label_low: int = 1,
    label_high: Optional[int] = None,
    repeat_prob: float = 0.0,
    blank: int = 0,
    zero_infinity: bool = False,
    reduction: str = "none",
    targets: Optional[Sequence[Sequence[int]]] = None,
    max_target_len: Optional[int] = None,
    gaps: Optional[Sequence[int]] = None,
    redraw_infeasible: bool = False,
    name: str = "custom",
    device="cpu",
) -> Batch:
    """Build a packed batch with the given per-utterance frame and target counts.

    ``gaps[b]`` extra rows may follow utterance ``b`` inside its cu_seqlens
    span (a gapped layout); those rows hold log probabilities too but belong
    to no utterance.

    The logits are drawn on ``device`` (a CUDA device draws the 300M-element
    large-vocabulary batch in milliseconds; the CPU takes about a minute);
    ``log_probs`` stays there.  The same seed gives the same batch on the same
    kind of device.
    """
    gen = torch.Generator().manual_seed(seed)
    B = len(lengths)
    label_high = num_classes - 1 if label_high is None else label_high
    gaps = [0] * B if gaps is None else list(gaps)
    seqs: List[torch.Tensor] = []
    for b in range(B):
        if targets is not None:
            seq = torch.as_tensor(list(targets[b])[: target_lengths[b]], dtype=torch.int64)
        else:
            for _ in range(1000):
                seq = _draw_targets(gen, int(target_lengths[b]), label_low, label_high, repeat_prob)
                if not redraw_infeasible or lengths[b] >= seq.numel() + _adjacent_repeats(seq):
                    break
        seqs.append(seq)
    spans = [int(lengths[b]) + int(gaps[b]) for b in range(B)]
    cu = [0]
    for s in spans:
        cu.append(cu[-1] + s)
    T_total = cu[-1]
    dev = torch.device(device)
    dgen = torch.Generator(device=dev).manual_seed(seed + 7919)
    logits = torch.randn(T_total, num_classes, generator=dgen, dtype=torch.float32, device=dev)
    logits.mul_(sigma)
    log_probs = torch.log_softmax(logits, dim=-1).to(dtype)
    del logits
    flat = torch.cat(seqs) if seqs else torch.zeros(0, dtype=torch.int64)
    mtl = max([int(t) for t in target_lengths] + [0]) if max_target_len is None else max_target_len
    return Batch(
        name=name,
        log_probs=log_probs,
        cu_seqlens=torch.tensor(cu, dtype=torch.int32),
        lengths=torch.tensor(list(lengths), dtype=torch.int32),
        targets=flat.to(torch.int32),
        target_lengths=torch.tensor(list(target_lengths), dtype=torch.int32),
        blank=blank,
        zero_infinity=zero_infinity,
        reduction=reduction,
        max_target_len=mtl,
    )


def _tiny(device="cpu"):
    return make_batch([50, 37, 64, 20], [10, 8, 12, 4], 32, dtype=torch.float32, seed=0, sigma=2.0,
                      label_low=1, label_high=31, reduction="none", zero_infinity=False, name="tiny", device=device)


def _lengths(gen, B, t_lo, t_hi, u_num_lo, u_den_lo, u_num_hi, u_den_hi):
    Ts, Us = [], []
    for _ in range(B):
        T = _uniform_int(gen, t_lo, t_hi)
        lo = math.ceil(T * u_num_lo / u_den_lo)
        hi = (T * u_num_hi) // u_den_hi
        Ts.append(T)
        Us.append(_uniform_int(gen, lo, hi))
    return Ts, Us


def _conformer(device="cpu"):
    gen = torch.Generator().manual_seed(0)
    Ts, Us = _lengths(gen, 32, 200, 400, 1, 6, 1, 4)
    return make_batch(Ts, Us, 1025, dtype=torch.bfloat16, seed=1, sigma=3.0, label_low=1, label_high=1024,
                      repeat_prob=0.10, redraw_infeasible=True, reduction="mean", name="conformer",
                      device=device)


def _longform(device="cpu"):
    gen = torch.Generator().manual_seed(0)
    Ts, Us = _lengths(gen, 8, 1500, 2000, 1, 4, 1, 3)
    T_bad = _uniform_int(gen, 1500, 2000)
    U_bad = (T_bad + 1) // 2 + 1  # all one id: aligning needs 2U - 1 > T frames
    bad_label = _uniform_int(gen, 1, 1024)
    lab_gen = torch.Generator().manual_seed(2)
    seqs = [torch.randint(1, 1025, (u,), generator=lab_gen).tolist() for u in Us]
    seqs.append([bad_label] * U_bad)
    return make_batch(Ts + [T_bad], Us + [U_bad], 1025, dtype=torch.float32, seed=1, sigma=2.0, targets=seqs,
                      zero_infinity=True, reduction="sum", name="longform", device=device)


def _char(device="cpu"):
    gen = torch.Generator().manual_seed(0)
    Ts, Us = _lengths(gen, 256, 100, 1000, 1, 8, 1, 3)
    return make_batch(Ts, Us, 29, dtype=torch.float16, seed=1, sigma=2.0, label_low=1, label_high=28,
                      repeat_prob=0.20, redraw_infeasible=True, reduction="mean", name="char", device=device)


def _largevocab(device="cpu"):
    gen = torch.Generator().manual_seed(0)
    Ts, Us = _lengths(gen, 64, 400, 800, 1, 8, 1, 4)
    return make_batch(Ts, Us, 8193, dtype=torch.bfloat16, seed=1, sigma=3.0, label_low=1, label_high=8192,
                      reduction="none", name="largevocab", device=device)


WORKLOADS = {
    "tiny": _tiny,
    "conformer": _conformer,
    "longform": _longform,
    "char": _char,
    "largevocab": _largevocab,
}


def workload(name: str, device="cpu") -> Batch:
    """One of the five named benchmark workloads, generated from seed 0."""
    return WORKLOADS[name](device=device)


def unnormalised_logits(batch: Batch, seed: int = 0, offset: float = 8.0) -> torch.Tensor:
    """Logits for the logits input form: the batch's log probabilities plus a
    seeded per-row offset drawn uniformly from [-offset, offset] (in float32,
    then cast to the batch's dtype), so that each row's log_softmax is the
    batch's row up to that cast."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    T_total = batch.log_probs.shape[0]
    shift = (torch.rand(T_total, 1, generator=gen, dtype=torch.float32) * 2.0 - 1.0) * offset
    z = batch.log_probs.detach().cpu().float() + shift
    return z.to(batch.log_probs.dtype)


def pack_fsas(fsas):
    """Concatenate per-sequence FSAs ``(start, final, edges (E, 3), weights)``
    into the packed arrays of the FSA entry points: ``(state_offsets,
    start_weight, final_weight, edge_offsets, edges, edge_weight)`` as
    int32 / float32 CPU tensors."""
    so, eo = [0], [0]
    sw, fw, ed, ew = [], [], [], []
    for start, final, edges, weights in fsas:
        sw += list(start)
        fw += list(final)
        ed += [list(e) for e in edges]
        ew += list(weights)
        so.append(so[-1] + len(start))
        eo.append(eo[-1] + len(edges))
    return (torch.tensor(so, dtype=torch.int32), torch.tensor(sw, dtype=torch.float32),
            torch.tensor(fw, dtype=torch.float32), torch.tensor(eo, dtype=torch.int32),
            torch.tensor(ed, dtype=torch.int32).reshape(-1, 3), torch.tensor(ew, dtype=torch.float32))


def ctc_lattice_fsa(targets: Sequence[int], blank: int):
    """The CTC lattice of one target sequence as FSA data: states 0 .. 2U of
    ``blank, l_1, blank, ..., l_U, blank`` plus an entry state 2U + 1; each
    state's edges into itself, into the next state and (from a label over a
    blank to a different label) two states on, each labelled with the class
    of the state it enters; the entry state starts, the last two states end
    (and the entry state too for an empty target)."""
    U = len(targets)
    S = 2 * U + 1
    ext = [blank if s % 2 == 0 else int(targets[(s - 1) // 2]) for s in range(S)]
    edges = []
    for s in range(S):
        edges.append((s, s, ext[s]))
        if s + 1 < S:
            edges.append((s, s + 1, ext[s + 1]))
        if s + 2 < S and s % 2 == 1 and ext[s + 2] != ext[s]:
            edges.append((s, s + 2, ext[s + 2]))
    edges.append((S, 0, ext[0]))
    if S > 1:
        edges.append((S, 1, ext[1]))
    inf = float("-inf")
    start = [inf] * (S + 1)
    start[S] = 0.0
    final = [inf] * (S + 1)
    final[S - 1] = 0.0
    if S > 1:
        final[S - 2] = 0.0
    if U == 0:
        final[S] = 0.0
    return start, final, edges, [0.0] * len(edges)


def random_fsa(num_states: int, num_edges: int, num_classes: int, seed: int):
    """A seeded random FSA: a left-to-right chain (so that paths exist) plus
    random extra edges, N(0, 0.5^2) edge weights, state 0 starting and the
    last state ending with weight 0, a few more start and final states."""
    gen = torch.Generator().manual_seed(seed)
    S = num_states
    edges = [(s, s + 1, int(torch.randint(0, num_classes, (1,), generator=gen))) for s in range(S - 1)]
    edges += [(s, s, int(torch.randint(0, num_classes, (1,), generator=gen))) for s in range(S)]
    while len(edges) < num_edges:
        a, b, c = (int(torch.randint(0, n, (1,), generator=gen)) for n in (S, S, num_classes))
        edges.append((a, b, c))
    weights = (torch.randn(len(edges), generator=gen) * 0.5).tolist()
    inf = float("-inf")
    start = [0.0] + [(float(torch.randn(1, generator=gen)) * 0.3 if float(torch.rand(1, generator=gen)) < 0.2
                      else inf) for _ in range(S - 1)]
    final = [(float(torch.randn(1, generator=gen)) * 0.3 if float(torch.rand(1, generator=gen)) < 0.2 else inf)
             for _ in range(S - 1)] + [0.0]
    return start, final, edges, weights


def padded_targets(batch: Batch, width: Optional[int] = None, fill: int = 0) -> torch.Tensor:
    """The concatenated targets as a padded ``(B, width)`` int64 tensor."""
    width = batch.max_target_len if width is None else width
    out = torch.full((batch.B, max(width, 0)), fill, dtype=torch.int64)
    off = 0
    for b in range(batch.B):
        u = int(batch.target_lengths[b])
        out[b, :u] = batch.targets[off: off + u].to(torch.int64)
        off += u
    return out


def select_utterances(batch: Batch, index: Sequence[int]) -> Batch:
    """A new tight batch made of the chosen utterances (rows copied out)."""
    toff = [0]
    for u in batch.target_lengths.tolist():
        toff.append(toff[-1] + int(u))
    rows, seqs, Ts, Us, cu = [], [], [], [], [0]
    for b in index:
        s = int(batch.cu_seqlens[b])
        T = int(batch.lengths[b])
        rows.append(batch.log_probs[s: s + T].cpu())
        seqs.append(batch.targets[toff[b]: toff[b + 1]])
        Ts.append(T)
        Us.append(int(batch.target_lengths[b]))
        cu.append(cu[-1] + T)
    return Batch(
        name=f"{batch.name}[{len(index)}]",
        log_probs=torch.cat(rows) if rows else batch.log_probs[:0].cpu(),
        cu_seqlens=torch.tensor(cu, dtype=torch.int32),
        lengths=torch.tensor(Ts, dtype=torch.int32),
        targets=torch.cat(seqs) if seqs else batch.targets[:0],
        target_lengths=torch.tensor(Us, dtype=torch.int32),
        blank=batch.blank,
        zero_infinity=batch.zero_infinity,
        reduction=batch.reduction,
        max_target_len=max(Us + [0]),
    )
