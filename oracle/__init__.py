"""fp64 CPU oracle of the eviction pass. TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this
package. The library's CUDA path never calls it and shares no code with it; the only thing both
sides use is the seeded input generator (``kv_cache_eviction_02_gb300.synth``), which holds none of
the method's arithmetic.

The arithmetic lives in ``oracle.c`` (plain C, double precision, written step by step from the
pages); this module builds it with gcc, loads it with ctypes and converts arrays. The H2O decode
loop (append, attend, accumulate, evict) is driven from Python in :class:`H2OUnit` on top of the
C routines.

Citations: LORE-KV project page ("LORE-KV: Monte Carlo Estimation for KV-Cache Eviction"), Method:
Eqs. 1-4, 10 (reliability), Eqs. 5-7 (projected deletion score), Eq. 8 (evict); Hyperparameters
table. H2O summary ("H2O: Heavy-Hitter Oracle ..."): Section 2.1, Definitions 2.1/2.2, Section 4.1
(Algorithm 1), Appendix A.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, ENOTPD = 0, 1, 4


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp,
                        "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            D = ctypes.POINTER(ctypes.c_double)
            I = ctypes.POINTER(ctypes.c_int)
            C = ctypes.POINTER(ctypes.c_char)
            i, l, d = ctypes.c_int, ctypes.c_long, ctypes.c_double
            lib.kvo_row_stats.argtypes = [l, D, l, D, D, D]
            lib.kvo_row_stats.restype = None
            lib.kvo_reliability.argtypes = [i, i, l, D, I, i, i, D, d, d, d, D, D, D, D, D]
            lib.kvo_gram_cholesky.argtypes = [i, i, i, D, i, D, D]
            lib.kvo_lorekv_unit.argtypes = [i, i, i, i, i, i, i, i, D, D, D, D, D, D, d, d, D, D, D, D]
            lib.kvo_lorekv_units.argtypes = [i, i, i, i, i, i, i, i, i, D, D, D, D, D, D, d, d, D]
            lib.kvo_select.argtypes = [i, i, i, i, i, D, I, I, D]
            lib.kvo_h2o_prefill_acc.argtypes = [i, i, D, D, D]
            lib.kvo_h2o_attend.argtypes = [i, i, D, D, D, D, D]
            lib.kvo_h2o_evict.argtypes = [i, I, D, i, d, C]
            lib.kvo_threads.argtypes = []
            _lib = lib
    return _lib


def _d(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _pd(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _pi(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def threads() -> int:
    return _load().kvo_threads()


# ---------------------------------------------------------------------------------------------
# LORE-KV
# ---------------------------------------------------------------------------------------------
def row_stats(z, y: int):
    """(lse, H, log q(y)) of one logits row (Eqs. 2-4)."""
    z = _d(z)
    out = [ctypes.c_double() for _ in range(3)]
    _load().kvo_row_stats(z.size, _pd(z), int(y), *[ctypes.byref(o) for o in out])
    return tuple(o.value for o in out)


def reliability(logits, sampled, qlook, M: int, T: int, beta: float, gamma: float,
                lambda_D: float) -> dict:
    """Reliability weights of one sequence (Eqs. 2-4, 10).

    logits [M*T][V], sampled [M*T], qlook [L][Hq][M*T][d] (or [LH][M*T][d])."""
    z = _d(logits)
    y = np.ascontiguousarray(np.asarray(sampled.cpu() if hasattr(sampled, "cpu") else sampled),
                             dtype=np.int32)
    q = _d(qlook)
    d = q.shape[-1]
    LH = q.size // (M * T * d)
    c = np.zeros(M * T)
    H = np.zeros(M * T)
    Dh = np.zeros(M)
    R = np.zeros(M)
    om = np.zeros(M)
    st = _load().kvo_reliability(M, T, z.shape[-1], _pd(z), _pi(y), LH, d, _pd(q), beta, gamma,
                                 lambda_D, _pd(c), _pd(H), _pd(Dh), _pd(R), _pd(om))
    if st != OK:
        raise ValueError(f"oracle reliability: status {st}")
    return {"c": c, "H": H, "Dhat": Dh, "R": R, "omega": om}


def gram_cholesky(W, d: int, h: int):
    """(G_h, L_h, status) for head h of the o_proj weight W [d_model][Hq*d]."""
    W = _d(W)
    G = np.zeros((d, d))
    L = np.zeros((d, d))
    st = _load().kvo_gram_cholesky(W.shape[0], W.shape[1], d, _pd(W), h, _pd(G), _pd(L))
    return G, L, st


def lorekv_unit(K, V, QW, QL, Lf, omega, *, M, T, sink, lambda_L, eps, window_causal=1,
                want=()):
    """Score one unit. K,V [n][d]; QW [g][w][d]; QL [g][M*T][d]; Lf [g][d][d]; omega [M].

    Returns S [n]; with ``want`` containing "lse", "o" or "E" also those arrays."""
    K, V, QW, QL, Lf, om = map(_d, (K, V, QW, QL, Lf, omega))
    n, d = K.shape
    g, w = QW.shape[0], QW.shape[1]
    nq = w + M * T
    S = np.zeros(n)
    lse = np.zeros((g, nq)) if "lse" in want else None
    o = np.zeros((g, nq, d)) if "o" in want else None
    E = np.zeros((g, nq, n)) if "E" in want else None
    nul = ctypes.POINTER(ctypes.c_double)()
    st = _load().kvo_lorekv_unit(n, d, g, w, M, T, int(window_causal), sink, _pd(K), _pd(V),
                                 _pd(QW), _pd(QL), _pd(Lf), _pd(om), lambda_L, eps, _pd(S),
                                 _pd(lse) if lse is not None else nul,
                                 _pd(o) if o is not None else nul,
                                 _pd(E) if E is not None else nul)
    if st != OK:
        raise ValueError(f"oracle lorekv_unit: status {st}")
    if not want:
        return S
    out = {"S": S}
    for k, v in (("lse", lse), ("o", o), ("E", E)):
        if v is not None:
            out[k] = v
    return out


def lorekv_units(K, V, QW, QL, Lf, omega, *, M, T, sink, lambda_L, eps, window_causal=1):
    """Score a stack of units in parallel (OpenMP over units). Leading axis = unit."""
    K, V, QW, QL, Lf, om = map(_d, (K, V, QW, QL, Lf, omega))
    units, n, d = K.shape
    g, w = QW.shape[1], QW.shape[2]
    S = np.zeros((units, n))
    st = _load().kvo_lorekv_units(units, n, d, g, w, M, T, int(window_causal), sink, _pd(K),
                                  _pd(V), _pd(QW), _pd(QL), _pd(Lf), _pd(om), lambda_L, eps,
                                  _pd(S))
    if st != OK:
        raise ValueError(f"oracle lorekv_units: status {st}")
    return S


def select(S, *, sink: int, w: int, chunk: int, B: int, want_chunks: bool = False):
    """Kept positions (ascending) of one unit (Eq. 8, chunked top-B)."""
    S = _d(S)
    n = S.size
    kept = np.zeros(n, dtype=np.int32)
    ln = ctypes.c_int()
    nch = max((n - sink - w) // chunk, 0)
    cs = np.zeros(max(nch, 1))
    st = _load().kvo_select(n, sink, w, chunk, B, _pd(S), _pi(kept), ctypes.byref(ln), _pd(cs))
    if st != OK:
        raise ValueError(f"oracle select: status {st}")
    kept = kept[: ln.value].copy()
    return (kept, cs[:nch].copy()) if want_chunks else kept


def compact(X, kept):
    """Dense compressed rows X[kept] (gather)."""
    return X[np.asarray(kept, dtype=np.int64)]


def lorekv_config_units(cfg, inputs, units, *, want_kept=True):
    """Oracle outputs for selected units of a full config.

    ``units`` is a list of (s, l, kh). Returns {unit: {"S", "kept", "omega"}}. omega uses every
    layer and head of the sequence (Eq. 10 with the disagreement term); the Cholesky factors come
    from the layer's W_O. The units are scored in parallel (OpenMP over units)."""
    from kv_cache_eviction_02_gb300.synth import unit_slice  # input slicing only

    g, d = cfg.g, cfg.d
    omegas = {}
    for (s, _, _) in units:
        if s not in omegas:
            omegas[s] = reliability(inputs["logits"][s], inputs["sampled"][s],
                                    inputs["Q_look"][s], cfg.M, cfg.T, cfg.beta, cfg.gamma,
                                    cfg.lambda_D)["omega"]
    Ks, Vs, QWs, QLs, Lfs, oms = [], [], [], [], [], []
    chol = {}
    for (s, l, kh) in units:
        u = unit_slice(cfg, inputs, s, l, kh)
        Lf = np.zeros((g, d, d))
        for j in range(g):
            key = (l, kh * g + j)
            if key not in chol:
                _, Lj, st = gram_cholesky(u["W_O"], d, kh * g + j)
                if st != OK:
                    raise ValueError("W_O^T W_O not positive definite")
                chol[key] = Lj
            Lf[j] = chol[key]
        Ks.append(_d(u["K"]))
        Vs.append(_d(u["V"]))
        QWs.append(_d(u["Q_W"]))
        QLs.append(_d(u["Q_look"]))
        Lfs.append(Lf)
        oms.append(omegas[s])
    S_all = lorekv_units(np.stack(Ks), np.stack(Vs), np.stack(QWs), np.stack(QLs),
                         np.stack(Lfs), np.stack(oms), M=cfg.M, T=cfg.T, sink=cfg.sink,
                         lambda_L=cfg.lambda_L, eps=cfg.eps, window_causal=cfg.window_causal)
    res = {}
    for i, (s, l, kh) in enumerate(units):
        r = {"S": S_all[i], "omega": omegas[s]}
        if want_kept:
            r["kept"] = select(S_all[i], sink=cfg.sink, w=cfg.w, chunk=cfg.chunk, B=cfg.B)
        res[(s, l, kh)] = r
    return res


# ---------------------------------------------------------------------------------------------
# H2O
# ---------------------------------------------------------------------------------------------
def h2o_prefill_acc(K, Q):
    """acc_j = sum_{i>=j} softmax_i(q_i . K_{<=i} / sqrt d)_j over a causal prompt."""
    K, Q = _d(K), _d(Q)
    P, d = K.shape
    acc = np.zeros(P)
    _load().kvo_h2o_prefill_acc(P, d, _pd(K), _pd(Q), _pd(acc))
    return acc


def h2o_attend(Kc, Vc, q):
    """(p, out) of one query over the retained rows (Section 2.1 restricted to S_i, Def. 2.2)."""
    Kc, Vc, q = _d(Kc), _d(Vc), _d(q)
    cnt, d = Kc.shape
    p = np.zeros(cnt)
    out = np.zeros(d)
    _load().kvo_h2o_attend(cnt, d, _pd(Kc), _pd(Vc), _pd(q), _pd(p), _pd(out))
    return p, out


def h2o_evict(pos, acc, t: int, frac: float):
    """Boolean mask of the entries evicted at length t (greedy argmin, k_t/2 recent protected)."""
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    acc = _d(acc)
    ev = ctypes.create_string_buffer(max(pos.size, 1))
    ne = _load().kvo_h2o_evict(pos.size, _pi(pos), _pd(acc), t, frac, ev)
    if ne < 0:
        raise ValueError("no eviction candidate")
    return np.frombuffer(ev.raw[: pos.size], dtype=np.uint8).astype(bool)


class H2OUnit:
    """One (batch, layer, head) unit of H2O decode in fp64.

    State: retained positions, their K/V rows and accumulated scores. ``full_acc`` keeps the
    accumulated score of every token ever seen (evicted ones included) for the invariant that
    the accumulated scores over all tokens sum to the number of queries processed."""

    def __init__(self, K, V, Q, frac: float, max_len: int):
        K, V, Q = _d(K), _d(V), _d(Q)
        P = K.shape[0]
        self.frac = frac
        self.d = K.shape[1]
        self.full_acc = np.zeros(max_len)
        acc = h2o_prefill_acc(K, Q)
        self.full_acc[:P] = acc
        self.t = P
        self.pos = np.arange(P, dtype=np.int32)
        self.K, self.V, self.acc = K.copy(), V.copy(), acc.copy()
        self.prefill_acc = acc.copy()
        self.queries = P
        self._evict_now()

    def adopt_prefill(self, keep_positions, K, V):
        """Teacher forcing after the prefill compression: retain exactly ``keep_positions`` of the
        prompt (K, V are the prompt rows) with their prefill accumulated scores."""
        keep = np.asarray(sorted(keep_positions), dtype=np.int32)
        K, V = _d(K), _d(V)
        self.pos, self.K, self.V = keep, K[keep], V[keep]
        self.acc = self.prefill_acc[keep].copy()

    def _evict_now(self):
        ev = h2o_evict(self.pos, self.acc, self.t, self.frac)
        keep = ~ev
        evicted = self.pos[ev].tolist()
        self.pos, self.K, self.V, self.acc = self.pos[keep], self.K[keep], self.V[keep], self.acc[keep]
        return evicted

    def step(self, q, k, v, evict: bool = True):
        """append -> attend (the new token attends to itself) -> accumulate -> evict.

        With evict=False the step stops before the eviction (teacher forcing: the caller then
        adopts a retained set with :meth:`adopt`)."""
        q, k, v = _d(q), _d(k), _d(v)
        self.pos = np.append(self.pos, np.int32(self.t))
        self.K = np.vstack([self.K, k[None]])
        self.V = np.vstack([self.V, v[None]])
        self.acc = np.append(self.acc, 0.0)
        self.t += 1
        p, out = h2o_attend(self.K, self.V, q)
        self.acc += p
        self.full_acc[self.pos] += p
        self.queries += 1
        pre = {"pos": self.pos.copy(), "acc": self.acc.copy()}
        evicted = self._evict_now() if evict else []
        return out, evicted, pre

    def adopt(self, keep_positions):
        """Teacher forcing: replace the retained set by ``keep_positions`` (a subset of it)."""
        keep = np.isin(self.pos, np.asarray(keep_positions))
        self.pos, self.K, self.V, self.acc = self.pos[keep], self.K[keep], self.V[keep], self.acc[keep]


def h2o_budget(t: int, frac: float):
    """(k_t, r_t): tokens held at length t and how many of the most recent are protected."""
    k = int(math.floor(frac * t))
    return k, k // 2
