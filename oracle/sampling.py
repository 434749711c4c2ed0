"""Next-token sampling from the LM head's logits, written out plainly.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Float64 NumPy.

[Next] "How Llama 3.1 Generates the Next Token", Temperature, Softmax and
"Top-k and top-p sampling":

  1. divide the logits by the temperature T;
  2. softmax over the whole vocabulary, P(i) = e^{z_i/T} / sum_j e^{z_j/T};
  3. top-k keeps the k most probable tokens; top-p keeps the smallest set of the
     most probable tokens whose probability adds up to at least p; with both,
     both restrictions apply;
  4. the kept probabilities are renormalised to sum to one and one token is drawn
     from them.

Readings where the pages leave a step open:
  * the draw is the inverse of the cumulative distribution: with the kept tokens
    in order of decreasing probability, the token whose cumulative renormalised
    probability first exceeds a uniform u in [0, 1) is chosen (the random number
    is an input, so both implementations can be given the same one);
  * equal logits are ordered by increasing token index (the same tie rule as
    the greedy choice);
  * "both restrictions apply" is the intersection of the two kept sets; both are
    prefixes of the same order, so the shorter prefix is kept: n = min(k, n_p);
  * T = 0 is the limit T -> 0: the greedy choice; top_k = 0 means no top-k
    restriction and top_p = 1 no top-p restriction.
"""
from __future__ import annotations

import numpy as np


def softmax_temperature(z: np.ndarray, temperature: float) -> np.ndarray:
    """P(i) = e^{z_i/T} / sum_j e^{z_j/T} over the last axis, max-subtracted ([Next]
    Softmax, with the temperature of [Next] Temperature)."""
    s = np.asarray(z, dtype=np.float64) / temperature
    s = s - np.max(s, axis=-1, keepdims=True)
    e = np.exp(s)
    return e / np.sum(e, axis=-1, keepdims=True)


def descending_order(z: np.ndarray) -> np.ndarray:
    """Token indices by decreasing logit, equal logits by increasing index."""
    return np.argsort(-np.asarray(z, dtype=np.float64), kind="stable")


def kept_count(p_sorted: np.ndarray, top_k: int, top_p: float) -> int:
    """How many of the most probable tokens survive top-k and top-p ([Next] Top-k and
    top-p sampling): the smallest prefix with probability >= top_p, cut to top_k."""
    V = p_sorted.shape[-1]
    n = V
    if 0 < top_k < V:
        n = top_k
    if top_p < 1.0:
        cum = np.cumsum(p_sorted)
        n_p = int(np.argmax(cum >= top_p)) + 1 if np.any(cum >= top_p) else V
        n = min(n, n_p)
    return n


def sample_row(z: np.ndarray, temperature: float, top_k: int, top_p: float, u: float) -> int:
    """One token id from one row of logits, given the uniform u in [0, 1)."""
    if temperature == 0.0 or top_k == 1:
        return int(np.argmax(z))                       # greedy: the first maximum
    order = descending_order(z)
    p_sorted = softmax_temperature(z, temperature)[order]
    n = kept_count(p_sorted, top_k, top_p)
    q = p_sorted[:n] / np.sum(p_sorted[:n])            # renormalised
    cum = np.cumsum(q)
    j = int(np.searchsorted(cum, u, side="right"))     # first cumulative value > u
    return int(order[min(j, n - 1)])


def sample(logits: np.ndarray, temperature: float, top_k: int, top_p: float, uniforms: np.ndarray) -> np.ndarray:
    """Token ids [B] for logits [B, V] and one uniform per row."""
    return np.array([sample_row(logits[b], temperature, top_k, top_p, float(uniforms[b]))
                     for b in range(logits.shape[0])], dtype=np.int64)


__all__ = ["softmax_temperature", "descending_order", "kept_count", "sample_row", "sample"]
