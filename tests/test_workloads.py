"""The seeded input generators: shapes, determinism and the planted row
structure (checked with the oracle on reduced-row copies). CPU only."""
import math

import numpy as np
import torch

import oracle
import workloads as W


def test_catalogue_sizes():
    w = W.WORKLOADS
    assert (w["ce_64x1000"].rows, w["ce_64x1000"].vocab) == (64, 1000)
    assert w["ce_64x1000"].seed == 0 and w["ce_64x1000"].scale == 1 / 64
    assert (w["ce_8192x128256"].rows, w["ce_8192x128256"].vocab) == (8192, 128256)
    d = w["argmax_256x151936_s152064"]
    assert (d.rows, d.vocab, d.stride, d.pad_value) == (256, 151936, 152064, -1e30)
    s = w["ce_16384x50257_x30"]
    assert (s.rows, s.vocab, s.sigma, s.scale) == (16384, 50257, 30.0, 1.0)
    assert W.HEADLINE in w and W.DECODE in w


def test_deterministic_and_shaped():
    w = W.WORKLOADS["ce_64x1000"]
    a, b = W.generate(w), W.generate(w)
    assert a.logits.shape == (64, 1000) and a.logits.dtype == torch.float32
    assert a.labels.dtype == torch.int64
    assert torch.equal(a.logits, b.logits) and torch.equal(a.labels, b.labels)
    assert 0.9 < float(a.logits.std()) < 1.1


def test_decode_padding_and_ties():
    w = W.WORKLOADS["argmax_256x151936_s152064"].with_rows(64)
    b = W.generate(w)
    x = b.logits.numpy()
    assert (x[:, w.vocab:] == np.float32(-1e30)).all()
    assert len(b.tie_rows) == round(0.1 * 64)
    top = oracle.load().argmax(x, w.vocab)
    for r, (c1, c2) in zip(b.tie_rows.tolist(), b.tie_cols.tolist()):
        assert c1 < c2 and x[r, c1] == x[r, c2]
        assert top[r] == c1, "the planted tie must hold the row max, lowest index first"


def test_stability_rows():
    w = W.WORKLOADS["ce_16384x50257_x30"].with_rows(300)
    b = W.generate(w)
    x = b.logits.numpy()
    orc = oracle.load()
    assert len(b.const_rows) == 15 and len(b.label_at_max_rows) == 3
    assert not set(b.const_rows.tolist()) & set(b.label_at_max_rows.tolist())
    for r in b.const_rows.tolist():
        assert (x[r, :w.vocab] == x[r, 0]).all()
    loss = orc.ce_rows(x, w.vocab, b.labels.numpy())
    for r in b.const_rows.tolist():
        assert abs(loss[r] - math.log(w.vocab)) < 1e-12
    top = orc.argmax(x, w.vocab)
    for r in b.label_at_max_rows.tolist():
        assert top[r] == int(b.labels[r])
        assert loss[r] < math.log(2)   # label holds the unique max
    assert 25 < float(np.std(x[:, :w.vocab])) < 35
