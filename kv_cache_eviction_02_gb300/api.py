"""Thin ctypes binding of libkvevict (include/kvevict.h), same names as the C-ABI.

Argument marshalling only: tensors go in as raw device pointers with their sizes, the stream is
the current torch CUDA stream unless one is given, and every non-zero status raises
:class:`KveError`. There is no fallback: if the library is missing or a tensor is not on a CUDA
device, the call fails.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvevict.so")

KVE_OK, KVE_EINVAL, KVE_EDTYPE, KVE_EWORKSPACE, KVE_ENOTPD, KVE_ECUDA, KVE_ETIMEOUT = range(7)
KVE_F32, KVE_BF16, KVE_F16 = 0, 1, 2
_DT = {torch.float32: KVE_F32, torch.bfloat16: KVE_BF16, torch.float16: KVE_F16}

EXPORTED = ("lorekv_prepare_wo", "lorekv_workspace_size", "lorekv_score",
            "lorekv_attention_stats", "lorekv_kept_capacity", "lorekv_select_compact",
            "lorekv_output_fidelity",
            "h2o_state_create", "h2o_prefill", "h2o_decode_step", "h2o_export", "h2o_capacity",
            "h2o_length", "h2o_state_destroy", "kve_last_error", "kve_check_device",
            "kve_inject_failure", "kve_profile_enable", "kve_profile_report", "kve_version",
            "kve_selftest_wait_timeout", "lorekv_score_noalloc",
            "cc_workspace_size", "cc_surprise", "cc_select_compact", "cc_cache_create",
            "cc_cache_append", "cc_cache_refresh", "cc_cache_step", "cc_cache_export",
            "cc_cache_length", "cc_cache_seen", "cc_cache_destroy")


class KveError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"kvevict status {status}: {msg}")
        self.status = status


class KveShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_seq", "n_layers", "n_q_heads", "n_kv_heads",
                                             "d_head", "d_model", "n_tokens", "vocab", "dtype")]


class KveLorekvParams(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_int) for n in ("w", "M", "T", "chunk", "sink", "budget_B",
                                              "window_causal")] +
                [(n, ctypes.c_float) for n in ("lambda_L", "beta", "gamma", "lambda_D", "eps")])


class KveCcShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_seq", "n_q_heads", "n_kv_heads", "d_head",
                                             "d_model", "n_tokens", "vocab", "dtype", "sink",
                                             "keep_J")]


_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, Z, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
        SP, PP = ctypes.POINTER(KveShape), ctypes.POINTER(KveLorekvParams)
        L.lorekv_prepare_wo.argtypes = [SP, P, P, P, P]
        L.lorekv_workspace_size.argtypes = [SP, PP]
        L.lorekv_workspace_size.restype = Z
        L.lorekv_score.argtypes = [SP, PP, P, P, P, P, P, P, P, P, P, P, P, Z, P]
        L.lorekv_score_noalloc.argtypes = [SP, PP, P, P, P, P, P, P, P, P, P, P, P]
        L.lorekv_attention_stats.argtypes = [SP, PP, P, P, P, P, P, P, P, Z, P]
        L.lorekv_output_fidelity.argtypes = [P, P, I, I, P, P, P]
        L.lorekv_kept_capacity.argtypes = [SP, PP]
        L.lorekv_select_compact.argtypes = [SP, PP, P, P, P, P, P, P, P, P, Z, P]
        L.h2o_state_create.argtypes = [ctypes.POINTER(P), I, I, I, I, I, F, I]
        L.h2o_prefill.argtypes = [P, P, P, P, I, P]
        L.h2o_decode_step.argtypes = [P, P, P, P, P, P]
        L.h2o_export.argtypes = [P, P, P, P, P, P, P]
        L.h2o_capacity.argtypes = [P]
        L.h2o_length.argtypes = [P]
        L.h2o_state_destroy.argtypes = [P]
        L.h2o_state_destroy.restype = None
        L.kve_last_error.restype = ctypes.c_char_p
        L.kve_check_device.argtypes = [P]
        L.kve_inject_failure.argtypes = [I, I]
        L.kve_profile_enable.argtypes = [I]
        L.kve_selftest_wait_timeout.argtypes = [I, P]
        L.kve_profile_report.argtypes = [ctypes.c_char_p, Z]
        CS = ctypes.POINTER(KveCcShape)
        L.cc_workspace_size.argtypes = [CS]
        L.cc_workspace_size.restype = Z
        L.cc_surprise.argtypes = [CS, P, P, P, P, P, P, P, P, P, Z, P]
        L.cc_select_compact.argtypes = [CS, P, P, P, P, P, P, P, P, P]
        L.cc_cache_create.argtypes = [ctypes.POINTER(P), CS]
        L.cc_cache_append.argtypes = [P, P, P, P, P, P, I, P]
        L.cc_cache_refresh.argtypes = [P, P, P, P]
        L.cc_cache_step.argtypes = [P, P, P, P, P, P, I, P, P, ctypes.POINTER(I), P]
        L.cc_cache_export.argtypes = [P, P, P, P, P, P, P, P]
        L.cc_cache_length.argtypes = [P]
        L.cc_cache_seen.argtypes = [P]
        L.cc_cache_destroy.argtypes = [P]
        L.cc_cache_destroy.restype = None
        _lib = L
    return _lib


def _check(status: int):
    if status != KVE_OK:
        raise KveError(status, lib().kve_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensor arguments must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return t.data_ptr()


_TORCH_DTYPE = {KVE_F32: torch.float32, KVE_BF16: torch.bfloat16, KVE_F16: torch.float16}


def _sized(t, name, dtype, numel):
    """_ptr of a tensor argument after checking it against the declared shape: its element type
    and at least the number of elements the call reads or writes through it (a short buffer
    would otherwise be read or written past its end on the device). Integer addresses pass
    unchecked."""
    if t is None or isinstance(t, int):
        return _ptr(t)
    if isinstance(dtype, int):
        dtype = _TORCH_DTYPE[dtype]
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, the shape declares {dtype}")
    if t.numel() < numel:
        raise ValueError(f"{name}: {t.numel()} elements, the shape needs {numel}")
    return _ptr(t)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class LorekvProblem:
    """Shape + parameters of one LORE-KV pass (the two C structs)."""
    n_seq: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    d_head: int
    d_model: int
    n_tokens: int
    vocab: int
    dtype: int
    w: int = 32
    M: int = 4
    T: int = 8
    chunk: int = 4
    sink: int = 4
    budget_B: int = 128
    window_causal: int = 1
    lambda_L: float = 1.0
    beta: float = 1.0
    gamma: float = 1.3
    lambda_D: float = 0.0
    eps: float = 1e-6

    @classmethod
    def from_config(cls, cfg) -> "LorekvProblem":
        return cls(cfg.S, cfg.L, cfg.Hq, cfg.Hkv, cfg.d, cfg.d_model, cfg.n, cfg.vocab,
                   {"f32": KVE_F32, "bf16": KVE_BF16}[cfg.dtype], cfg.w, cfg.M, cfg.T,
                   cfg.chunk, cfg.sink, cfg.B, cfg.window_causal, cfg.lambda_L, cfg.beta,
                   cfg.gamma, cfg.lambda_D, cfg.eps)

    def shape(self) -> KveShape:
        return KveShape(self.n_seq, self.n_layers, self.n_q_heads, self.n_kv_heads, self.d_head,
                        self.d_model, self.n_tokens, self.vocab, self.dtype)

    def params(self) -> KveLorekvParams:
        return KveLorekvParams(self.w, self.M, self.T, self.chunk, self.sink, self.budget_B,
                               self.window_causal, self.lambda_L, self.beta, self.gamma,
                               self.lambda_D, self.eps)

    @property
    def units(self) -> int:
        return self.n_seq * self.n_layers * self.n_kv_heads

    def _inputs(self, K, V, Q_W, Q_look):
        """Checked pointers of the cache and query tensors (layouts of lorekv_score)."""
        rows = self.n_seq * self.n_layers
        return (_sized(K, "K", self.dtype, self.units * self.n_tokens * self.d_head),
                _sized(V, "V", self.dtype, self.units * self.n_tokens * self.d_head),
                _sized(Q_W, "Q_W", self.dtype, rows * self.n_q_heads * self.w * self.d_head),
                _sized(Q_look, "Q_look", self.dtype,
                       rows * self.n_q_heads * self.M * self.T * self.d_head))

    def _factors(self, L, G):
        f = self.n_layers * self.n_q_heads * self.d_head * self.d_head
        return _sized(L, "L", torch.float32, f), _sized(G, "G", torch.float32, f)

    def _outputs(self, logits, sampled, scores_out, omega_out):
        mt = self.n_seq * self.M * self.T
        return (_sized(logits, "logits", torch.float32, mt * self.vocab),
                _sized(sampled, "sampled", torch.int32, mt),
                _sized(scores_out, "scores_out", torch.float32, self.units * self.n_tokens),
                _sized(omega_out, "omega_out", torch.float32, self.n_seq * self.M))


def lorekv_prepare_wo(pb: LorekvProblem, W_O, L_out, G_out, stream=None):
    sh = pb.shape()
    f = pb.n_layers * pb.n_q_heads * pb.d_head * pb.d_head
    _check(lib().lorekv_prepare_wo(
        ctypes.byref(sh), _sized(W_O, "W_O", pb.dtype, f // pb.d_head * pb.d_model),
        _sized(L_out, "L_out", torch.float32, f), _sized(G_out, "G_out", torch.float32, f),
        _stream(stream)))


def lorekv_workspace_size(pb: LorekvProblem) -> int:
    sh, pr = pb.shape(), pb.params()
    return int(lib().lorekv_workspace_size(ctypes.byref(sh), ctypes.byref(pr)))


def lorekv_kept_capacity(pb: LorekvProblem) -> int:
    sh, pr = pb.shape(), pb.params()
    c = lib().lorekv_kept_capacity(ctypes.byref(sh), ctypes.byref(pr))
    if c < 0:
        _check(-c)
    return c


def lorekv_score(pb, K, V, Q_W, Q_look, L, G, logits, sampled, scores_out, omega_out, workspace,
                 stream=None):
    sh, pr = pb.shape(), pb.params()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().lorekv_score(ctypes.byref(sh), ctypes.byref(pr), *pb._inputs(K, V, Q_W, Q_look),
                              *pb._factors(L, G), *pb._outputs(logits, sampled, scores_out,
                                                               omega_out),
                              _ptr(workspace), ws_bytes, _stream(stream)))


def lorekv_score_noalloc(pb, K, V, Q_W, Q_look, L, G, logits, sampled, scores_out, omega_out,
                         stream=None):
    """lorekv_score with the library's fixed scratch array instead of a workspace (allocates
    nothing; shapes needing more than 64 MiB of scratch are rejected)."""
    sh, pr = pb.shape(), pb.params()
    _check(lib().lorekv_score_noalloc(ctypes.byref(sh), ctypes.byref(pr),
                                      *pb._inputs(K, V, Q_W, Q_look), *pb._factors(L, G),
                                      *pb._outputs(logits, sampled, scores_out, omega_out),
                                      _stream(stream)))


def lorekv_attention_stats(pb, K, V, Q_W, Q_look, lse_out, o_out, workspace, stream=None):
    sh, pr = pb.shape(), pb.params()
    ws_bytes = workspace.numel() * workspace.element_size()
    rows = pb.units * (pb.n_q_heads // pb.n_kv_heads) * (pb.w + pb.M * pb.T)
    _check(lib().lorekv_attention_stats(ctypes.byref(sh), ctypes.byref(pr),
                                        *pb._inputs(K, V, Q_W, Q_look),
                                        _sized(lse_out, "lse_out", torch.float32, rows),
                                        _sized(o_out, "o_out", torch.float32, rows * pb.d_head),
                                        _ptr(workspace), ws_bytes, _stream(stream)))


def lorekv_output_fidelity(o_full, o_comp, cos_out, mean_out=None, stream=None):
    rows, d = o_full.shape[0], o_full.shape[-1]
    _check(lib().lorekv_output_fidelity(_ptr(o_full), _ptr(o_comp), int(rows), int(d),
                                        _ptr(cos_out), _ptr(mean_out), _stream(stream)))


def lorekv_select_compact(pb, scores, K, V, kept_idx, kept_len, K_out, V_out, workspace=None,
                          stream=None):
    sh, pr = pb.shape(), pb.params()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    cap = lorekv_kept_capacity(pb)
    kv = pb.units * pb.n_tokens * pb.d_head
    _check(lib().lorekv_select_compact(
        ctypes.byref(sh), ctypes.byref(pr),
        _sized(scores, "scores", torch.float32, pb.units * pb.n_tokens),
        _sized(K, "K", pb.dtype, kv), _sized(V, "V", pb.dtype, kv),
        _sized(kept_idx, "kept_idx", torch.int32, pb.units * cap),
        _sized(kept_len, "kept_len", torch.int32, pb.units),
        _sized(K_out, "K_out", pb.dtype, pb.units * cap * pb.d_head),
        _sized(V_out, "V_out", pb.dtype, pb.units * cap * pb.d_head),
        _ptr(workspace), ws_bytes, _stream(stream)))


@dataclass
class CcProblem:
    """Shape of one counter-causal refresh (the C struct KveCcShape)."""
    n_seq: int
    n_q_heads: int
    n_kv_heads: int
    d_head: int
    d_model: int
    n_tokens: int
    vocab: int
    dtype: int
    sink: int
    keep_J: int

    def shape(self) -> KveCcShape:
        return KveCcShape(self.n_seq, self.n_q_heads, self.n_kv_heads, self.d_head, self.d_model,
                          self.n_tokens, self.vocab, self.dtype, self.sink, self.keep_J)

    def _rows(self, K, V, Q, H, tokens, m):
        """Checked pointers (K, V, Q, H, tokens) of m token rows per sequence: K, V
        [n_seq][n_kv_heads][m][d_head], Q [n_seq][n_q_heads][m][d_head], H [n_seq][m][d_model],
        tokens [n_seq][m] int32."""
        kv = self.n_seq * self.n_kv_heads * m * self.d_head
        return (_sized(K, "K", self.dtype, kv), _sized(V, "V", self.dtype, kv),
                _sized(Q, "Q", self.dtype, self.n_seq * self.n_q_heads * m * self.d_head),
                _sized(H, "H", self.dtype, self.n_seq * m * self.d_model),
                _sized(tokens, "tokens", torch.int32, self.n_seq * m))

    def _weights(self, W_O, W_U):
        return (_sized(W_O, "W_O", self.dtype, self.d_model * self.n_q_heads * self.d_head),
                _sized(W_U, "W_U", self.dtype, self.vocab * self.d_model))


def cc_workspace_size(pb: CcProblem) -> int:
    sh = pb.shape()
    return int(lib().cc_workspace_size(ctypes.byref(sh)))


def cc_surprise(pb: CcProblem, K, V, Q_fresh, H_last, W_O, W_U, tokens, surprise_out, workspace,
                stream=None):
    sh = pb.shape()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    k, v, q, h, t = pb._rows(K, V, Q_fresh, H_last, tokens, pb.n_tokens)
    _check(lib().cc_surprise(ctypes.byref(sh), k, v, q, h, *pb._weights(W_O, W_U), t,
                             _sized(surprise_out, "surprise_out", torch.float32,
                                    pb.n_seq * pb.n_tokens),
                             _ptr(workspace), ws_bytes, _stream(stream)))


def cc_select_compact(pb: CcProblem, surprise, K, V, tokens, kept_idx, K_out, V_out, tokens_out,
                      stream=None):
    sh = pb.shape()
    k, v, _, _, t = pb._rows(K, V, None, None, tokens, pb.n_tokens)
    ko, vo, _, _, to = pb._rows(K_out, V_out, None, None, tokens_out, pb.keep_J)
    _check(lib().cc_select_compact(ctypes.byref(sh),
                                   _sized(surprise, "surprise", torch.float32,
                                          pb.n_seq * pb.n_tokens), k, v, t,
                                   _sized(kept_idx, "kept_idx", torch.int32, pb.n_seq * pb.keep_J),
                                   ko, vo, to, _stream(stream)))


class CcCache:
    """Owns a KveCcCache handle (cc_cache_create / cc_cache_destroy): the counter-causal refresh
    cycle with memory keep_J and chunk h = n_tokens - keep_J."""

    def __init__(self, pb: CcProblem):
        h = ctypes.c_void_p()
        sh = pb.shape()
        _check(lib().cc_cache_create(ctypes.byref(h), ctypes.byref(sh)))
        self.h = h
        self.pb = pb

    @property
    def length(self) -> int:
        return lib().cc_cache_length(self.h)

    @property
    def seen(self) -> int:
        return lib().cc_cache_seen(self.h)

    def append(self, K_new, V_new, Q_new, H_new, tokens_new, stream=None):
        m = int(K_new.shape[-2])
        _check(lib().cc_cache_append(self.h, *self.pb._rows(K_new, V_new, Q_new, H_new,
                                                            tokens_new, m),
                                     m, _stream(stream)))

    def refresh(self, W_O, W_U, stream=None):
        _check(lib().cc_cache_refresh(self.h, *self.pb._weights(W_O, W_U), _stream(stream)))

    def step(self, K_new, V_new, Q_new, H_new, tokens_new, W_O, W_U, stream=None) -> bool:
        r = ctypes.c_int(0)
        m = int(K_new.shape[-2])
        _check(lib().cc_cache_step(self.h, *self.pb._rows(K_new, V_new, Q_new, H_new, tokens_new,
                                                          m),
                                   m, *self.pb._weights(W_O, W_U), ctypes.byref(r),
                                   _stream(stream)))
        return bool(r.value)

    def export(self, stream=None) -> dict:
        pb, n, dev = self.pb, self.length, torch.device("cuda")
        dt = {KVE_F32: torch.float32, KVE_BF16: torch.bfloat16}[pb.dtype]
        out = {"K": torch.empty(pb.n_seq, pb.n_kv_heads, n, pb.d_head, dtype=dt, device=dev),
               "Q": torch.empty(pb.n_seq, pb.n_q_heads, n, pb.d_head, dtype=dt, device=dev),
               "H": torch.empty(pb.n_seq, n, pb.d_model, dtype=dt, device=dev),
               "tokens": torch.empty(pb.n_seq, n, dtype=torch.int32, device=dev),
               "pos": torch.empty(pb.n_seq, n, dtype=torch.int32, device=dev)}
        out["V"] = torch.empty_like(out["K"])
        if n > 0:
            _check(lib().cc_cache_export(self.h, _ptr(out["K"]), _ptr(out["V"]), _ptr(out["Q"]),
                                         _ptr(out["H"]), _ptr(out["tokens"]), _ptr(out["pos"]),
                                         _stream(stream)))
        return out

    def close(self):
        if self.h:
            lib().cc_cache_destroy(self.h)
            self.h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def kve_check_device(stream=None):
    _check(lib().kve_check_device(_stream(stream)))


def kve_selftest_wait_timeout(limit_ms: int, stream=None):
    _check(lib().kve_selftest_wait_timeout(limit_ms, _stream(stream)))


def kve_inject_failure(status: int, count: int):
    lib().kve_inject_failure(status, count)


def kve_profile_enable(on: bool):
    lib().kve_profile_enable(1 if on else 0)


def kve_profile_report() -> dict:
    """{stage: {"groups", "kernels", "ms"}} of the launches recorded since the last report."""
    buf = ctypes.create_string_buffer(1 << 16)
    lib().kve_profile_report(buf, len(buf))
    out = {}
    for ln in buf.value.decode().splitlines():
        name, groups, kernels, ms = ln.split()
        out[name] = {"groups": int(groups), "kernels": int(kernels), "ms": float(ms)}
    return out


def kve_version() -> int:
    return lib().kve_version()


class H2OState:
    """Owns a KveH2O handle (h2o_state_create / h2o_state_destroy)."""

    def __init__(self, batch, n_layers, n_heads, d_head, max_len, budget_frac, dtype):
        h = ctypes.c_void_p()
        _check(lib().h2o_state_create(ctypes.byref(h), batch, n_layers, n_heads, d_head, max_len,
                                      float(budget_frac), _DT[dtype]))
        self.h = h
        self.units = batch * n_layers * n_heads
        self.d = d_head
        self.dtype = dtype

    @property
    def capacity(self) -> int:
        return lib().h2o_capacity(self.h)

    @property
    def length(self) -> int:
        return lib().h2o_length(self.h)

    def prefill(self, K, V, Q, stream=None):
        P = int(K.shape[-2])
        n = self.units * P * self.d  # [batch][n_layers][n_heads][P][d_head] each
        _check(lib().h2o_prefill(self.h, _sized(K, "K", self.dtype, n), _sized(V, "V", self.dtype, n),
                                 _sized(Q, "Q", self.dtype, n), P, _stream(stream)))

    def decode_step(self, q, k_new, v_new, attn_out, stream=None):
        n = self.units * self.d  # [batch][n_layers][n_heads][d_head] each
        _check(lib().h2o_decode_step(self.h, _sized(q, "q", self.dtype, n),
                                     _sized(k_new, "k_new", self.dtype, n),
                                     _sized(v_new, "v_new", self.dtype, n),
                                     _sized(attn_out, "attn_out", self.dtype, n), _stream(stream)))

    def export(self, stream=None):
        cap, dev = self.capacity, torch.device("cuda")
        K = torch.empty(self.units, cap, self.d, dtype=self.dtype, device=dev)
        V = torch.empty_like(K)
        pos = torch.empty(self.units, cap, dtype=torch.int32, device=dev)
        acc = torch.empty(self.units, cap, dtype=torch.float32, device=dev)
        cnt = torch.empty(self.units, dtype=torch.int32, device=dev)
        _check(lib().h2o_export(self.h, _ptr(K), _ptr(V), _ptr(pos), _ptr(acc), _ptr(cnt),
                                _stream(stream)))
        return {"K": K, "V": V, "pos": pos, "acc": acc, "count": cnt}

    def close(self):
        if self.h:
            lib().h2o_state_destroy(self.h)
            self.h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def h2o_state_create(batch, n_layers, n_heads, d_head, max_len, budget_frac, dtype) -> H2OState:
    return H2OState(batch, n_layers, n_heads, d_head, max_len, budget_frac, dtype)


def h2o_prefill(state: H2OState, K, V, Q, stream=None):
    state.prefill(K, V, Q, stream)


def h2o_decode_step(state: H2OState, q, k_new, v_new, attn_out, stream=None):
    state.decode_step(q, k_new, v_new, attn_out, stream)


def h2o_export(state: H2OState, stream=None):
    return state.export(stream)


# ---- convenience: one full eviction pass --------------------------------------------------------
class LorekvPass:
    """Owns the outputs and the workspace of LORE-KV passes of one shape (allocated once)."""

    def __init__(self, pb: LorekvProblem, device="cuda"):
        self.pb = pb
        dt = {KVE_F32: torch.float32, KVE_BF16: torch.bfloat16}[pb.dtype]
        dev = torch.device(device)
        u = pb.units
        self.cap = lorekv_kept_capacity(pb)
        self.scores = torch.empty(u, pb.n_tokens, dtype=torch.float32, device=dev)
        self.omega = torch.empty(pb.n_seq, pb.M, dtype=torch.float32, device=dev)
        self.workspace = torch.empty(lorekv_workspace_size(pb), dtype=torch.uint8, device=dev)
        self.kept_idx = torch.empty(u, self.cap, dtype=torch.int32, device=dev)
        self.kept_len = torch.empty(u, dtype=torch.int32, device=dev)
        self.K_out = torch.empty(u, self.cap, pb.d_head, dtype=dt, device=dev)
        self.V_out = torch.empty_like(self.K_out)

    def run(self, inp: dict, L, G, stream=None):
        lorekv_score(self.pb, inp["K"], inp["V"], inp["Q_W"], inp["Q_look"], L, G, inp["logits"],
                     inp["sampled"], self.scores, self.omega, self.workspace, stream)
        lorekv_select_compact(self.pb, self.scores, inp["K"], inp["V"], self.kept_idx,
                              self.kept_len, self.K_out, self.V_out, None, stream)
