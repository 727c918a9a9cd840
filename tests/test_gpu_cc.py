"""GPU parity of the counter-causal surprise refresh (fast single-layer variant) against the fp64
oracle (oracle/counter_causal.py), through the C-ABI.

Surprise: the GPU computes in fp32 from the same rounded inputs the oracle reads in fp64. The
error bound per token is relative to the sum of magnitudes of every term of its logit,
    scale_i = sum_m |W_U[x_i][m]| (|h_im| + sum_k |W_O[m][k]| |o_ik|),
because an fp32 sum of N terms carries at most about N * 2^-24 times that sum and in practice
about sqrt(N) * 2^-24 of it: 1e-5 * scale_i + 1e-6 is far above that and far below any
plausible mistake (a dropped head, a wrong KV head, one missing key), which moves the logit by
order |logit| ~ scale_i / sqrt(d_model).

On the tensor-core path (bf16, d_head 128) the softmax numerators p_j are rounded to bf16 before
the product with V, while their sum l stays fp32: o_h carries sum_j a_j eps_j v_j with a_j the
attention weights and eps_j the relative rounding errors (independent, zero mean, standard
deviation at most 2^-8 / sqrt 3). Through the logit weights c = W_O^T W_U[x_i] that gives a
standard deviation sigma_P = 2^-8/sqrt(3) * sqrt(sum_h sum_j a_j^2 (c_h . v_j)^2). The projection
W_O o then runs on the tensor cores from o rounded to bf16, which adds
sigma_O = 2^-8/sqrt(3) * sqrt(sum_k c_k^2 o_k^2). The bound there adds 6 sqrt(sigma_P^2 + sigma_O^2).

Selection: integer work, compared bit-exactly on the GPU's own surprise vector (the oracle selects
from the same fp32 values); the gathers are byte-exact.
"""
import math

import numpy as np
import pytest
import torch

from kv_cache_eviction_02_gb300 import api, synth
from oracle import counter_causal as cc

pytestmark = pytest.mark.gpu

SURPRISE_RTOL = 1e-5
BF16_REL_SD = 2.0 ** -8 / math.sqrt(3.0)  # relative sd of a round-to-nearest bf16 value (bound)


def _dev():
    return torch.device("cuda:0")


def _pb(cfg, **kw):
    p = api.CcProblem(cfg.batch, cfg.Hq, cfg.Hkv, cfg.d, cfg.d_model, cfg.n, cfg.vocab,
                      {"f32": api.KVE_F32, "bf16": api.KVE_BF16}[cfg.dtype], cfg.sink, cfg.J)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _run_surprise(cfg, inp):
    pb = _pb(cfg)
    ws = torch.empty(api.cc_workspace_size(pb), dtype=torch.uint8, device=_dev())
    s = torch.full((cfg.batch, cfg.n), float("nan"), dtype=torch.float32, device=_dev())
    api.cc_surprise(pb, inp["K"], inp["V"], inp["Q_fresh"], inp["H_last"], inp["W_O"],
                    inp["W_U"], inp["tokens"], s, ws)
    api.kve_check_device()
    return s


def _f64(t):
    return t.detach().cpu().double().numpy()


def _tensor_core_path(cfg):
    return cfg.dtype == "bf16" and cfg.d == 128 and cfg.batch * cfg.Hkv * cfg.n >= 128


def _sigma_p(K, V, Q, rows, c, hkv):
    """sd of the logit error from bf16 softmax numerators (module docstring); c [rows][Hq*d]."""
    hq, n, d = Q.shape
    g = hq // hkv
    out = np.zeros(len(rows))
    for r, i in enumerate(rows):
        if i >= n - 1:
            continue
        var = 0.0
        for h in range(hq):
            s = K[h // g, i + 1:] @ Q[h, i] / math.sqrt(d)
            a = np.exp(s - s.max())
            a /= a.sum()
            cv = V[h // g, i + 1:] @ c[r, h * d:(h + 1) * d]
            var += np.sum(a * a * cv * cv)
        out[r] = BF16_REL_SD * math.sqrt(var)
    return out


def _oracle_rows(inp, b, rows, hkv, bf16_p):
    """Oracle surprise, error scale and bf16-P sd at the listed positions of sequence b (W_U
    reduced to the rows the listed tokens use, which is all the logit reads)."""
    X = inp["tokens"][b].cpu().numpy().astype(np.int64)[rows]
    uniq, inv = np.unique(X, return_inverse=True)
    W_U = _f64(inp["W_U"][torch.as_tensor(uniq, device=inp["W_U"].device)])
    W_O, H = _f64(inp["W_O"]), _f64(inp["H_last"][b])[rows]
    K, V, Q = _f64(inp["K"][b]), _f64(inp["V"][b]), _f64(inp["Q_fresh"][b])
    o = cc.cc_attention_rows(K, V, Q, rows)
    z = cc.cc_logits(o, H, W_O, W_U, inv)
    r_abs = np.abs(H) + np.abs(o.reshape(len(rows), -1)) @ np.abs(W_O).T
    scale = np.einsum("nm,nm->n", np.abs(W_U[inv]), r_abs)
    sig = np.zeros(len(rows))
    if bf16_p:
        c = W_U[inv] @ W_O
        sig_o = BF16_REL_SD * np.sqrt(np.sum((c * o.reshape(len(rows), -1)) ** 2, axis=1))
        sig = np.sqrt(_sigma_p(K, V, Q, rows, c, hkv) ** 2 + sig_o ** 2)
    return -z, scale, sig


def _check_rows(cfg, inp, s_gpu, b, rows):
    n = cfg.n
    s_o, scale, sig = _oracle_rows(inp, b, rows, cfg.Hkv, _tensor_core_path(cfg))
    g = s_gpu[b].double().cpu().numpy()[rows]
    for k, i in enumerate(rows):
        if i < cfg.sink or i == n - 1:
            assert g[k] == np.inf, (b, i)
        else:
            assert np.isfinite(g[k]), (b, i)
            tol = SURPRISE_RTOL * scale[k] + 1e-6 + 6.0 * sig[k]
            assert abs(g[k] - s_o[k]) <= tol, (b, i, g[k], s_o[k], tol)


@pytest.mark.parametrize("name,kw", [
    ("tiny", {}),                                          # f32, GQA 2, n=203 (ragged tiles)
    ("tiny", dict(dtype="bf16", d=128, n=77, Hq=6, Hkv=2, sink=0, J=40)),
    ("tiny", dict(d=32, n=1, Hq=2, Hkv=1, sink=0, J=1)),   # one token: only the last
    ("tiny", dict(d=32, n=2, Hq=3, Hkv=3, sink=1, J=1)),
    ("tiny", dict(dtype="bf16", d=128, n=300, Hq=8, Hkv=2, d_model=256, batch=3, sink=4, J=250)),
    # tensor-core path: 3 heads per KV head, so CTA pairs straddle position blocks (the later tile
    # masks the earlier block entirely) and the last pair has a discarded second tile
    ("tiny", dict(dtype="bf16", d=128, n=389, Hq=6, Hkv=2, d_model=160, batch=2, sink=2, J=300)),
    ("tiny", dict(dtype="bf16", d=128, n=128, Hq=1, Hkv=1, d_model=64, batch=1, sink=1, J=64)),
    ("tiny", dict(dtype="bf16", d=64, n=150, Hq=4, Hkv=2, sink=2, J=100)),  # bf16 SIMT path
])
def test_surprise_matches_oracle_every_token(name, kw):
    cfg = synth.CC_CONFIGS[name].replace(**kw)
    inp = synth.cc_inputs(cfg, _dev())
    s = _run_surprise(cfg, inp)
    for b in range(cfg.batch):
        _check_rows(cfg, inp, s, b, list(range(cfg.n)))


def test_surprise_qwen7b_512_every_token():
    cfg = synth.CC_CONFIGS["qwen7b_512"]
    inp = synth.cc_inputs(cfg, _dev())
    s = _run_surprise(cfg, inp)
    _check_rows(cfg, inp, s, 0, list(range(cfg.n)))


def test_surprise_qwen7b_4096_sampled_tokens():
    """Full size: the oracle evaluates sampled positions one by one (sinks, the first and last
    tiles, the tail, random interior positions); every token is checked for the +inf rule."""
    cfg = synth.CC_CONFIGS["qwen7b_4096"]
    inp = synth.cc_inputs(cfg, _dev())
    s = _run_surprise(cfg, inp)
    rng = np.random.default_rng(7)
    rows = sorted(set([0, 3, 4, 5, 31, 32, 33, 63, 64, 4000, 4063, 4064, 4093, 4094, 4095]
                      + rng.integers(5, cfg.n - 1, size=24).tolist()))
    _check_rows(cfg, inp, s, 0, rows)
    g = s[0].cpu().numpy()
    assert np.all(np.isinf(g[:cfg.sink])) and np.isinf(g[-1])
    assert np.all(np.isfinite(g[cfg.sink:-1]))


def _select(cfg, s_gpu, K, V, X):
    pb = _pb(cfg)
    B, J = cfg.batch, cfg.J
    kept = torch.full((B, J), -1, dtype=torch.int32, device=_dev())
    Ko = torch.empty(B, cfg.Hkv, J, cfg.d, dtype=K.dtype, device=_dev())
    Vo = torch.empty_like(Ko)
    Xo = torch.empty(B, J, dtype=torch.int32, device=_dev())
    api.cc_select_compact(pb, s_gpu, K, V, X, kept, Ko, Vo, Xo)
    torch.cuda.synchronize()
    return kept, Ko, Vo, Xo


def _check_select(cfg, s_gpu, K, V, X, out):
    kept, Ko, Vo, Xo = out
    s = s_gpu.cpu().numpy()
    for b in range(cfg.batch):
        want = cc.cc_select(s[b], cfg.J)
        got = kept[b].cpu().numpy()
        assert got.tolist() == want.tolist(), b
        idx = torch.as_tensor(want.astype(np.int64), device=_dev())
        assert torch.equal(Ko[b], K[b][:, idx]) and torch.equal(Vo[b], V[b][:, idx])
        assert torch.equal(Xo[b], X[b][idx])


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("qwen7b_512", {}), ("qwen7b_4096", {})])
def test_select_compact_matches_oracle(name, kw):
    cfg = synth.CC_CONFIGS[name].replace(**kw)
    inp = synth.cc_inputs(cfg, _dev())
    s = _run_surprise(cfg, inp)
    _check_select(cfg, s, inp["K"], inp["V"], inp["tokens"],
                  _select(cfg, s, inp["K"], inp["V"], inp["tokens"]))


@pytest.mark.parametrize("n,J,levels,seed", [
    (10, 3, 3, 0), (1024, 700, 4, 1), (1025, 1, 2, 2), (3000, 2999, 5, 3), (3000, 3000, 5, 4),
    (5000, 1234, 1, 5),                       # every surprise equal: the lowest positions
    (4097, 2048, 1000000, 6),                 # nearly all distinct
])
def test_select_with_ties_and_edges(n, J, levels, seed):
    """Surprise vectors with many equal values, +inf and negative entries, sizes around the
    1024-thread scan blocks, J = 1 and J = n."""
    cfg = synth.CC_CONFIGS["tiny"].replace(n=n, J=J, batch=2, d=64, Hkv=2, Hq=2)
    g = torch.Generator(device="cpu").manual_seed(100 + seed)
    s = (torch.randint(0, levels, (2, n), generator=g).float() - levels / 2) * 0.5
    s[:, 0] = float("inf")
    s[:, n - 1] = float("inf")
    s = s.to(_dev())
    K = torch.randn(2, 2, n, 64, generator=g).to(_dev())
    V = torch.randn(2, 2, n, 64, generator=g).to(_dev())
    X = torch.randint(0, 300, (2, n), generator=g, dtype=torch.int32).to(_dev())
    _check_select(cfg, s, K, V, X, _select(cfg, s, K, V, X))


def test_token_id_out_of_range_is_reported():
    """An id outside [0, vocab) is read as 0 on the device and reported by kve_check_device."""
    cfg = synth.CC_CONFIGS["tiny"]
    inp = synth.cc_inputs(cfg, _dev())
    inp["tokens"][1, 17] = cfg.vocab
    pb = _pb(cfg)
    ws = torch.empty(api.cc_workspace_size(pb), dtype=torch.uint8, device=_dev())
    s = torch.empty(cfg.batch, cfg.n, dtype=torch.float32, device=_dev())
    api.cc_surprise(pb, inp["K"], inp["V"], inp["Q_fresh"], inp["H_last"], inp["W_O"],
                    inp["W_U"], inp["tokens"], s, ws)
    with pytest.raises(api.KveError) as e:
        api.kve_check_device()
    assert e.value.status == api.KVE_EINVAL
    api.kve_check_device()  # the word was cleared
