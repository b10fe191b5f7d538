"""Shared test helpers: tolerances, conversions, seeded routing for GPU tests."""
import numpy as np
import torch

# Floating-point parity bar for bf16 outputs with fp32 accumulation, normwise
# per tensor: max|got-ref| / max|ref| <= 1e-2 and sum|got-ref| / sum|ref| <= 1e-3.
MAX_REL = 1e-2
MEAN_REL = 1e-3


def f64(t):
    """A torch tensor (any device/dtype) as a float64 numpy array."""
    return t.detach().to("cpu", torch.float64).numpy()


def bits(t):
    """A bf16 torch tensor as numpy uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def rel_errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = np.abs(got - ref)
    mx = float(diff.max() / max(np.abs(ref).max(), 1e-30)) if ref.size else 0.0
    mean = float(diff.sum() / max(np.abs(ref).sum(), 1e-30)) if ref.size else 0.0
    return mx, mean


def assert_close(got, ref, name, max_rel=MAX_REL, mean_rel=MEAN_REL):
    mx, mean = rel_errors(got, ref)
    assert np.isfinite(np.asarray(got, np.float64)).all(), f"{name}: non-finite values"
    assert mx <= max_rel and mean <= mean_rel, f"{name}: max_rel={mx:.3e} mean_rel={mean:.3e}"
    return mx, mean


def near_tie_tokens(logits, R, rel=6e-5):
    """Tokens whose routing may differ between two logit computations that each
    stay within the logits' max bar (3e-5 * max|logit|): two of the token's R + 1
    largest logits lie within twice that, rel * max|logit|.  The R-th / (R+1)-th
    pair decides which experts are chosen; the pairs above it decide the slot
    order (slot order = selection order)."""
    l = np.asarray(logits, np.float64)
    T, E = l.shape
    k = min(R + 1, E)
    s = -np.sort(-l, axis=1)[:, :k]
    gaps = s[:, :-1] - s[:, 1:]
    return (gaps <= rel * np.abs(l).max()).any(axis=1)


def random_routing(T, E, R, seed, skew=0.0):
    """Seeded distinct-expert routing (host), weights positive and summing to 1."""
    g = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** (-skew)
    p /= p.sum()
    keys = np.log(p)[None, :] - np.log(-np.log(g.random((T, E)).clip(1e-300, 1.0)))
    idx = np.argsort(-keys, axis=1)[:, :R].astype(np.int32)
    u = g.random((T, R)) + 0.5
    w = (u / u.sum(1, keepdims=True)).astype(np.float32)
    return idx, w


class LazyExperts:
    """[E, ...] device weight tensor read one expert at a time as bf16 bits."""

    def __init__(self, t):
        self.t, self.shape = t, tuple(t.shape)

    def __getitem__(self, e):
        return bits(self.t[e])
