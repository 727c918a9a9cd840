"""fp64 oracle of the counter-causal surprise refresh, fast single-layer variant. TEST
INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import it; the library's CUDA path shares no code with it.

Counter-causal page ("Back from the Future: KV Cache Management by Counter-Causal Surprise"):
* Section 3.1, Eq. 1: the surprise of cached token i is 1 - P(x_i | x_{i+1:t});
* Section 3.2: a pass over the cached keys and values with a strictly upper-triangular mask and
  fresh queries at the original positions (step 1, step 3); the logit of the true token x_i stands
  in for the probability, lower logit = higher surprise (step 4); the last token has no future and
  gets the maximum surprise (step 5);
* Section 3.3: the fast variant runs only the last layer, from its stored input activations;
* Algorithm 3 (memory refresh): keep the J highest-surprise entries of the J + h candidates;
* Algorithm 1 (driver): a refresh after every h-th token, the recent chunk cleared after it;
* Design choice 4: system-prompt sink slots are never scored or evicted.

Readings (the page leaves them open): the fresh queries, the last layer's input residual stream
h_i, its output projection W_O ([d_model][H_q * d], the PyTorch o_proj layout) and the unembedding
W_U ([vocab][d_model]) are inputs; the layer's output is the residual stream plus the attention
update, h_i + W_O [o_i^0; ...; o_i^{H_q-1}], without the MLP or final norm (weights the page does not
give); query head h reads KV head h // (H_q / H_kv); the attention scale is 1/sqrt(d); equal
surprise keeps the lower position; kept tokens stay in ascending position order.
"""
from __future__ import annotations

import math

import numpy as np


def _d(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().float().cpu().numpy()
    return np.asarray(a, dtype=np.float64)


def cc_attention_rows(K, V, Qf, rows) -> np.ndarray:
    """Counter-causal attention of one sequence at the listed positions (Section 3.2, step 1).

    K, V [H_kv][n][d]; Qf [H_q][n][d] fresh queries. Position i attends to positions j > i only:
    o_i^h = sum_{j>i} softmax_j(q_i^h . k_j / sqrt d) v_j; query head h reads KV head
    h // (H_q / H_kv). The last position sees nothing (o = 0). Returns o [len(rows)][H_q][d]."""
    K, V, Qf = _d(K), _d(V), _d(Qf)
    hkv, n, d = K.shape
    hq = Qf.shape[0]
    g = hq // hkv
    o = np.zeros((len(rows), hq, d))
    for r, i in enumerate(rows):
        if i >= n - 1:
            continue
        for h in range(hq):
            kh = h // g
            s = K[kh, i + 1:] @ Qf[h, i] / math.sqrt(d)
            a = np.exp(s - s.max())
            o[r, h] = (a / a.sum()) @ V[kh, i + 1:]
    return o


def cc_attention(K, V, Qf) -> np.ndarray:
    """Counter-causal attention at every position of one sequence: o [n][H_q][d]."""
    return cc_attention_rows(K, V, Qf, range(_d(K).shape[1]))


def cc_logits(o, Hres, W_O, W_U, X) -> np.ndarray:
    """logit_i = W_U[x_i] . (h_i + W_O [o_i^0; ...; o_i^{H_q-1}]) (Section 3.2 step 4, Section 3.3).

    o [n][H_q][d]; Hres [n][d_model]; W_O [d_model][H_q*d]; W_U [vocab][d_model]; X [n] token ids."""
    o, Hres, W_O, W_U = _d(o), _d(Hres), _d(W_O), _d(W_U)
    X = np.asarray(X, dtype=np.int64)
    n = o.shape[0]
    r = Hres + o.reshape(n, -1) @ W_O.T
    return np.einsum("nm,nm->n", W_U[X], r)


def cc_surprise(K, V, Qf, Hres, W_O, W_U, X, sink: int) -> np.ndarray:
    """Surprise of every cached token of one sequence: -logit_i; +inf for the sink slots (never
    scored, design choice 4) and for the last token (no future, step 5)."""
    s = -cc_logits(cc_attention(K, V, Qf), Hres, W_O, W_U, X)
    s[:sink] = np.inf
    s[-1] = np.inf
    return s


def cc_select(s, J: int) -> np.ndarray:
    """Algorithm 3: keep the J highest-surprise tokens (equal surprise: the lower position first),
    returned in ascending position order; all tokens when J >= n."""
    n = len(s)
    if J >= n:
        return np.arange(n, dtype=np.int32)
    order = sorted(range(n), key=lambda i: (-s[i], i))
    return np.sort(np.asarray(order[:J], dtype=np.int32))


def cc_refresh(K, V, Qf, Hres, W_O, W_U, X, cand, J: int, sink: int) -> np.ndarray:
    """Algorithm 3 over the candidate positions `cand` (ascending: the memory, then the recent
    chunk): score the candidates as one sequence (cc_surprise; the candidates with position < sink
    are the system-prompt slots) and keep the J most surprising, ascending. All are kept when there
    are J or fewer. K, V [H_kv][T][d], Qf [H_q][T][d], Hres [T][d_model], X [T] hold every token
    seen so far, indexed by position."""
    cand = np.asarray(cand, dtype=np.int64)
    if len(cand) <= J:
        return cand
    K, V, Qf, Hres = _d(K), _d(V), _d(Qf), _d(Hres)
    X = np.asarray(X, dtype=np.int64)
    s = cc_surprise(K[:, cand], V[:, cand], Qf[:, cand], Hres[cand], W_O, W_U, X[cand],
                    int(np.sum(cand < sink)))
    return cand[cc_select(s, J)]


def cc_cycle(K, V, Qf, Hres, W_O, W_U, X, J: int, h: int, sink: int, chunks) -> list:
    """Algorithm 1 without the model: tokens 0, 1, ... arrive in appends of the given sizes (each
    at most the free rows of the current chunk); after every h-th token the memory plus the chunk
    is refreshed (cc_refresh) and the chunk is cleared. Returns the memory after each refresh."""
    mem, recent, t, out = [], [], 0, []
    for c in chunks:
        assert 1 <= c <= h - len(recent)
        recent.extend(range(t, t + c))
        t += c
        if len(recent) == h:
            mem = list(cc_refresh(K, V, Qf, Hres, W_O, W_U, X, mem + recent, J, sink))
            recent = []
            out.append(np.asarray(mem))
    return out
