"""Seeded synthetic inputs for the row-wise softmax cross-entropy path.

This module only draws inputs. It holds none of the arithmetic of the method
(no max, no exp, no sum, no argmax): the tests and the bench hand the same
arrays to the CUDA path and to the CPU oracle.

Five workloads mirror the sizes and value structure of a language model's
output head (f32 logits ``[rows, vocab]`` row-major, int64 labels):

=============================  =====  =======  =======  ========================================
name                           rows   vocab    stride   values / structure
=============================  =====  =======  =======  ========================================
ce_64x1000                        64     1000     1000  N(0, 1); labels uniform; scale 1/64
ce_4096x32000                   4096    32000    32000  N(0, 2^2); labels uniform; scale 1/4096
ce_8192x128256                  8192   128256   128256  N(0, 3^2) (4.2 GB); scale 1/8192
argmax_256x151936_s152064        256   151936   152064  N(0, 1); padding -1e30; 10% of rows
                                                        with an exact tie at two random columns
ce_16384x50257_x30             16384    50257    50257  N(0, 30^2); 5% of rows one constant;
                                                        1% of rows with the label at the row max;
                                                        scale 1.0
=============================  =====  =======  =======  ========================================

"N(0, s^2)" means ``s * randn``: the second number of each spec is a standard
deviation.

Recipe (the same on any device; the bulk draw uses that device's torch
generator, so a CPU copy and a CUDA copy of one seed hold different numbers):

1. ``logits[:, :vocab] = sigma * randn`` from ``torch.Generator(device)``
   seeded with the workload's seed; columns ``vocab..stride`` hold the
   padding value.
2. ``labels = randint(0, vocab)`` from the same generator.
3. Row structure comes from a CPU generator seeded with ``seed + 7919``:
   a random permutation of the rows picks, in this order and disjoint,
   the constant rows, the label-at-max rows and the tie rows.
   - constant row: every column holds one value ``sigma * randn``;
   - label-at-max row: a label column L is drawn; the row is a draw of
     ``vocab`` iid normals conditioned on column L holding the largest:
     ``g = ndtri(u0 ** (1 / vocab))`` (the maximum of ``vocab`` normals) at L
     and ``ndtri(u_j * ndtr(g))`` (a normal truncated below g) elsewhere,
     all times sigma. No maximum of drawn values is ever taken;
   - tie row: two distinct columns c1 < c2 both get ``12 * sigma``, a value
     that ``sigma * randn`` does not reach (P < 1e-32 per draw), so both
     hold the row max and the expected token is c1.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    rows: int
    vocab: int
    stride: int
    sigma: float
    seed: int
    scale: float | None = None        # gradient scale; None for argmax-only
    pad_value: float | None = None    # value of columns vocab..stride
    tie_frac: float = 0.0             # rows with a planted exact tie
    const_frac: float = 0.0           # rows holding one constant value
    label_at_max_frac: float = 0.0    # rows whose label holds the row max
    ops: tuple = ("rows", "loss", "grad", "argmax")

    @property
    def elements(self) -> int:
        return self.rows * self.vocab

    def with_rows(self, rows: int) -> "Workload":
        """The same recipe over fewer (or more) rows."""
        return dataclasses.replace(self, name=f"{self.name}[rows={rows}]", rows=rows)


WORKLOADS: dict[str, Workload] = {
    w.name: w for w in [
        Workload("ce_64x1000", 64, 1000, 1000, 1.0, seed=0, scale=1.0 / 64),
        Workload("ce_4096x32000", 4096, 32000, 32000, 2.0, seed=1, scale=1.0 / 4096,
                 ops=("loss", "grad", "argmax")),
        Workload("ce_8192x128256", 8192, 128256, 128256, 3.0, seed=2, scale=1.0 / 8192,
                 ops=("rows", "loss", "grad", "argmax")),
        Workload("argmax_256x151936_s152064", 256, 151936, 152064, 1.0, seed=3,
                 pad_value=-1e30, tie_frac=0.10, ops=("argmax",)),
        Workload("ce_16384x50257_x30", 16384, 50257, 50257, 30.0, seed=4, scale=1.0,
                 const_frac=0.05, label_at_max_frac=0.01, ops=("loss", "grad", "argmax")),
    ]
}

# The training-step workload the bench times, and the decode-argmax workload.
HEADLINE = "ce_8192x128256"
DECODE = "argmax_256x151936_s152064"


@dataclass
class Batch:
    workload: Workload
    logits: torch.Tensor          # [rows, stride] f32
    labels: torch.Tensor          # [rows] int64
    const_rows: torch.Tensor      # row indices (int64, CPU)
    label_at_max_rows: torch.Tensor
    tie_rows: torch.Tensor        # row indices
    tie_cols: torch.Tensor        # [n, 2] (c1 < c2)

    @property
    def scale(self) -> float:
        return 1.0 if self.workload.scale is None else self.workload.scale

    def special_rows(self) -> torch.Tensor:
        return torch.cat([self.const_rows, self.label_at_max_rows, self.tie_rows])


def _count(frac: float, rows: int) -> int:
    return int(round(frac * rows))


def generate(w: Workload, device: str | torch.device = "cpu") -> Batch:
    """Draw one batch of ``w`` on ``device`` (see the module docstring)."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    logits = torch.empty((w.rows, w.stride), dtype=torch.float32, device=device)
    if w.rows:
        body = logits[:, : w.vocab]
        body.normal_(0.0, 1.0, generator=g)
        body.mul_(w.sigma)
        if w.stride > w.vocab:
            logits[:, w.vocab:].fill_(0.0 if w.pad_value is None else w.pad_value)
    labels = torch.randint(0, w.vocab, (w.rows,), generator=g, device=device, dtype=torch.int64)

    cg = torch.Generator(device="cpu")
    cg.manual_seed(w.seed + 7919)
    perm = torch.randperm(w.rows, generator=cg)
    n_const = _count(w.const_frac, w.rows)
    n_lam = _count(w.label_at_max_frac, w.rows)
    n_tie = _count(w.tie_frac, w.rows)
    const_rows = perm[:n_const].clone()
    lam_rows = perm[n_const:n_const + n_lam].clone()
    tie_rows = perm[n_const + n_lam:n_const + n_lam + n_tie].clone()

    if n_const:
        vals = (w.sigma * torch.randn(n_const, generator=cg, dtype=torch.float64)).float()
        logits[const_rows.to(device), : w.vocab] = vals.to(device)[:, None]

    if n_lam:
        lam_labels = torch.randint(0, w.vocab, (n_lam,), generator=cg, dtype=torch.int64)
        for k in range(n_lam):
            u0 = torch.rand((), generator=cg, dtype=torch.float64)
            top = torch.special.ndtri(u0 ** (1.0 / w.vocab))
            u = torch.rand(w.vocab, generator=cg, dtype=torch.float64)
            row = torch.special.ndtri(u * torch.special.ndtr(top))
            row[lam_labels[k]] = top
            logits[int(lam_rows[k]), : w.vocab] = (w.sigma * row).float().to(device)
        labels[lam_rows.to(device)] = lam_labels.to(device)

    tie_cols = torch.empty((n_tie, 2), dtype=torch.int64)
    if n_tie:
        for k in range(n_tie):
            c = torch.randperm(w.vocab, generator=cg)[:2]
            tie_cols[k, 0] = int(c.min())
            tie_cols[k, 1] = int(c.max())
        r = tie_rows.to(device)
        v = torch.full((n_tie,), 12.0 * w.sigma, dtype=torch.float32, device=device)
        logits[r, tie_cols[:, 0].to(device)] = v
        logits[r, tie_cols[:, 1].to(device)] = v

    return Batch(w, logits, labels, const_rows, lam_rows, tie_rows, tie_cols)


def random_logits(rows: int, vocab: int, stride: int | None = None, sigma: float = 1.0,
                  seed: int = 0, pad_value: float = float("nan"), device="cpu"):
    """A plain seeded ``[rows, stride]`` f32 batch (``sigma * randn``; padding
    columns hold ``pad_value``) and uniform int64 labels, for small cases."""
    stride = vocab if stride is None else stride
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.empty((rows, stride), dtype=torch.float32)
    x[:, :vocab] = sigma * torch.randn((rows, vocab), generator=g)
    if stride > vocab:
        x[:, vocab:] = pad_value
    labels = torch.randint(0, vocab, (rows,), generator=g, dtype=torch.int64)
    return x.to(device), labels.to(device)
