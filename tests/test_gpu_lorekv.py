"""GPU parity of the LORE-KV eviction pass against the fp64 oracle (called through the C-ABI).

Small configurations compare every unit element by element; they span several token tiles with a
ragged tail, GQA groups of 1, 4 and 5, both coefficient presets, causal and non-causal window
queries, and the all-kept edge case. The full-size workloads (Mistral-7B-, Llama-3.1-8B- and
Qwen2.5-14B-shaped) run in the benchmark's launch configuration and compare sampled units with
the oracle, plus properties checked on every unit.
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_02_gb300 import api, synth
from parity import (OMEGA_RTOL, SCORE_RTOL, assert_kept_matches,
                    assert_kept_valid_for_own_scores, assert_scores_close)

pytestmark = pytest.mark.gpu

CFG = synth.LorekvConfig
SMALL = {
    "tiny": synth.LOREKV_CONFIGS["tiny"],
    "bf16_gqa4_D": CFG("bf16_gqa4_D", "bf16", S=2, L=2, Hq=8, Hkv=2, d=128, d_model=256, n=1000,
                       vocab=5000, beta=1.0, gamma=1.0, lambda_D=0.3),
    "bf16_gqa5_E": CFG("bf16_gqa5_E", "bf16", S=1, L=1, Hq=10, Hkv=2, d=128, d_model=640,
                       n=2084, vocab=3000, B=512, outlier_frac=0.01),
    "f32_ragged_d32": CFG("f32_ragged_d32", "f32", S=1, L=2, Hq=4, Hkv=2, d=32, d_model=64,
                          n=300, vocab=300, B=64, keys="normal"),
    "bf16_noncausal": CFG("bf16_noncausal", "bf16", S=1, L=1, Hq=4, Hkv=1, d=128, d_model=512,
                          n=516, vocab=1000, window_causal=0, M=2, T=4, w=16),
    "f32_all_kept": CFG("f32_all_kept", "f32", S=1, L=1, Hq=2, Hkv=1, d=64, d_model=64,
                        n=36 + 96, vocab=64, keys="normal"),
}


# 80 units: enough (unit, query tile) pairs that the attention pass plans ranges of several
# 128-token tiles per CTA (the small configurations above plan one tile per range)
MULTITILE = CFG("bf16_multitile", "bf16", S=1, L=10, Hq=32, Hkv=8, d=128, d_model=512, n=2048,
                vocab=1000)
MULTITILE_UNITS = [(0, 0, 0), (0, 4, 3), (0, 9, 7)]
# GQA 5: 320 queries per KV head, so the attention CTAs hold one query tile each (rows 0-127,
# 128-255, 256-319) and double-buffer S over multi-tile ranges
MULTITILE_G5 = CFG("bf16_multitile_g5", "bf16", S=1, L=4, Hq=40, Hkv=8, d=128, d_model=512,
                   n=2048, vocab=1000)
MULTITILE_G5_UNITS = [(0, 0, 0), (0, 2, 5), (0, 3, 7)]
MULTITILE_CASES = {"gqa4": (MULTITILE, MULTITILE_UNITS), "gqa5": (MULTITILE_G5, MULTITILE_G5_UNITS)}


def _dev():
    return torch.device("cuda:0")


def _prepare(cfg, g):
    pb = api.LorekvProblem.from_config(cfg)
    Lf = torch.empty(cfg.L, cfg.Hq, cfg.d, cfg.d, device=_dev())
    G = torch.empty_like(Lf)
    api.lorekv_prepare_wo(pb, g["W_O"], Lf, G)
    return pb, Lf, G


def _all_units(cfg):
    return [(s, l, kh) for s in range(cfg.S) for l in range(cfg.L) for kh in range(cfg.Hkv)]


def _unit_index(cfg, s, l, kh):
    return (s * cfg.L + l) * cfg.Hkv + kh


@pytest.mark.parametrize("name", list(SMALL))
def test_prepare_wo_matches_oracle(name):
    cfg = SMALL[name]
    inp = synth.lorekv_inputs(cfg, "cpu")
    g = {k: v.to(_dev()) for k, v in inp.items()}
    _, Lf, G = _prepare(cfg, g)
    Lc, Gc = Lf.double().cpu().numpy(), G.double().cpu().numpy()
    for l in range(cfg.L):
        for h in range(cfg.Hq):
            Gr, Lr, st = oracle.gram_cholesky(inp["W_O"][l], cfg.d, h)
            assert st == oracle.OK
            assert np.allclose(Gc[l, h], Gr, rtol=1e-6, atol=1e-7 * np.abs(Gr).max())
            assert np.allclose(Lc[l, h], Lr, rtol=1e-6, atol=1e-7 * np.abs(Lr).max())


# (d_model, d_head): tensor-core Gram (bf16, d_head 128, d_model a multiple of 128) and each of
# its fall-backs to the double-precision kernel
_GRAM_SHAPES = [(384, 128), (1280, 128), (200, 128), (256, 64)]


@pytest.mark.parametrize("d_model,d", _GRAM_SHAPES, ids=[f"dm{a}-d{b}" for a, b in _GRAM_SHAPES])
def test_prepare_wo_gram_paths_match_oracle(d_model, d):
    """G and L of bf16 weights, on the tensor-core path and its fall-backs, against the oracle's
    double-precision Gram and Cholesky (LORE-KV page, Method, Eqs. 5-7)."""
    L, Hq = 2, 3
    gen = torch.Generator().manual_seed(d_model * 131 + d)
    W = (torch.randn(L, d_model, Hq * d, generator=gen) / d_model ** 0.5).to(torch.bfloat16)
    pb = api.LorekvProblem(1, L, Hq, 1, d, d_model, 256, 10, api.KVE_BF16)
    Lf = torch.empty(L, Hq, d, d, device=_dev())
    G = torch.empty_like(Lf)
    api.lorekv_prepare_wo(pb, W.to(_dev()), Lf, G)
    Lc, Gc = Lf.double().cpu().numpy(), G.double().cpu().numpy()
    for l in range(L):
        for h in range(Hq):
            Gr, Lr, st = oracle.gram_cholesky(W[l], d, h)
            assert st == oracle.OK
            assert np.allclose(Gc[l, h], Gr, rtol=1e-6, atol=1e-7 * np.abs(Gr).max()), (l, h)
            assert np.allclose(Lc[l, h], Lr, rtol=1e-6, atol=1e-7 * np.abs(Lr).max()), (l, h)


def test_prepare_wo_reports_not_positive_definite():
    # d_model < d_head: every Gram matrix is rank deficient
    pb = api.LorekvProblem(1, 1, 2, 1, 64, 16, 100, 10, api.KVE_F32)
    W = torch.randn(1, 16, 128, device=_dev())
    Lf = torch.empty(1, 2, 64, 64, device=_dev())
    with pytest.raises(api.KveError) as e:
        api.lorekv_prepare_wo(pb, W, Lf, torch.empty_like(Lf))
    assert e.value.status == api.KVE_ENOTPD


@pytest.mark.parametrize("name", list(SMALL))
def test_attention_statistics_match_oracle(name):
    cfg = SMALL[name]
    inp = synth.lorekv_inputs(cfg, "cpu")
    g = {k: v.to(_dev()) for k, v in inp.items()}
    pb = api.LorekvProblem.from_config(cfg)
    ws = torch.empty(api.lorekv_workspace_size(pb), dtype=torch.uint8, device=_dev())
    Qu = cfg.g * cfg.queries_per_head
    lse = torch.empty(cfg.units, Qu, device=_dev())
    o = torch.empty(cfg.units, Qu, cfg.d, device=_dev())
    api.lorekv_attention_stats(pb, g["K"], g["V"], g["Q_W"], g["Q_look"], lse, o, ws)
    api.kve_check_device()
    lse, o = lse.double().cpu().numpy(), o.double().cpu().numpy()
    tol = 1e-5 if cfg.dtype == "f32" else 2e-3
    for (s, l, kh) in _all_units(cfg):
        u = synth.unit_slice(cfg, inp, s, l, kh)
        eye = np.stack([np.eye(cfg.d)] * cfg.g)
        r = oracle.lorekv_unit(u["K"], u["V"], u["Q_W"], u["Q_look"], eye, np.ones(cfg.M) / cfg.M,
                               M=cfg.M, T=cfg.T, sink=cfg.sink, lambda_L=1.0, eps=cfg.eps,
                               window_causal=cfg.window_causal, want=("lse", "o"))
        ui = _unit_index(cfg, s, l, kh)
        lse_ref = r["lse"].reshape(-1)
        o_ref = r["o"].reshape(-1, cfg.d)
        assert np.allclose(lse[ui], lse_ref, rtol=0, atol=tol * np.maximum(1, np.abs(lse_ref)).max())
        err = np.linalg.norm(o[ui] - o_ref, axis=1)
        if cfg.dtype == "f32":
            assert np.all(err <= tol * np.linalg.norm(o_ref, axis=1) + 1e-6), (name, err.max())
        else:
            # bf16: every a_j reaches the tensor cores rounded to bf16 (relative error uniform in
            # [-2^-9, 2^-9]), so |o_gpu - o| has an RMS of 2^-9/sqrt(3) sqrt(sum_j a_j^2 |v_j|^2);
            # allow 4 sigma plus fp32 accumulation
            sigma = 2.0 ** -9 / np.sqrt(3.0) * _attention_weighted_vnorm(cfg, u, lse_ref)
            bound = 4.0 * sigma + 1e-5 * np.linalg.norm(o_ref, axis=1) + 1e-6
            assert np.all(err <= bound), (name, float((err / bound).max()))


def _run_pass(cfg, g):
    pb, Lf, G = _prepare(cfg, g)
    run = api.LorekvPass(pb, _dev())
    run.run(g, Lf, G)
    api.kve_check_device()
    return run


@pytest.mark.parametrize("name", list(SMALL))
def test_eviction_pass_matches_oracle(name):
    _check_full_pass(SMALL[name], name)


# Degenerate settings of the method: nothing to evict (n = sink + w), one trajectory of one
# lookahead query (M = T = 1), a single window query (w = 1), window-only aggregation
# (lambda_L = 0); tensor-core path (bf16, d_head 128) and CUDA-core path (fp32).
DEGENERATE = {
    "bf16_no_candidates": CFG("bf16_no_cand", "bf16", S=1, L=1, Hq=4, Hkv=1, d=128, d_model=256,
                              n=36, vocab=300),
    "bf16_M1_T1": CFG("bf16_m1t1", "bf16", S=1, L=2, Hq=4, Hkv=2, d=128, d_model=256, n=552,
                      vocab=300, M=1, T=1, B=64),
    "bf16_w1": CFG("bf16_w1", "bf16", S=1, L=1, Hq=8, Hkv=2, d=128, d_model=256, n=517,
                   vocab=300, w=1, B=64),
    "bf16_window_only": CFG("bf16_winonly", "bf16", S=1, L=1, Hq=4, Hkv=1, d=128, d_model=256,
                            n=548, vocab=300, lambda_L=0.0),
    "f32_window_only_M1": CFG("f32_winonly", "f32", S=1, L=1, Hq=4, Hkv=2, d=32, d_model=64,
                              n=300, vocab=300, lambda_L=0.0, M=1, T=2, w=8, B=64),
}


@pytest.mark.parametrize("name", list(DEGENERATE))
def test_degenerate_settings_match_oracle(name):
    _check_full_pass(DEGENERATE[name], name)


def _check_full_pass(cfg, name):
    """The whole pass (omega, scores, kept sets, compaction) against the oracle on every unit."""
    inp = synth.lorekv_inputs(cfg, "cpu")
    g = {k: v.to(_dev()) for k, v in inp.items()}
    run = _run_pass(cfg, g)
    ref = oracle.lorekv_config_units(cfg, inp, _all_units(cfg))
    S = run.scores.double().cpu().numpy()
    om = run.omega.double().cpu().numpy()
    kept = run.kept_idx.cpu().numpy()
    klen = run.kept_len.cpu().numpy()
    for (s, l, kh), r in ref.items():
        ui = _unit_index(cfg, s, l, kh)
        assert np.allclose(om[s], r["omega"], rtol=OMEGA_RTOL, atol=0), (name, s)
        assert_scores_close(S[ui], r["S"], cfg.dtype, f"{name} unit {ui}")
        assert klen[ui] == run.cap
        assert_kept_matches(kept[ui, :klen[ui]], r["S"], sink=cfg.sink, w=cfg.w, chunk=cfg.chunk,
                            B=cfg.B, rtol=SCORE_RTOL[cfg.dtype], what=f"{name} unit {ui}")
    # compaction is bit-exact given the GPU's own index set
    Kf = g["K"].reshape(cfg.units, cfg.n, cfg.d)
    Vf = g["V"].reshape(cfg.units, cfg.n, cfg.d)
    idx = run.kept_idx.long()
    assert torch.equal(run.K_out, torch.gather(Kf, 1, idx[..., None].expand(-1, -1, cfg.d)))
    assert torch.equal(run.V_out, torch.gather(Vf, 1, idx[..., None].expand(-1, -1, cfg.d)))


def _attention_weighted_vnorm(cfg, u, lse):
    """sqrt(sum_j a_{q,j}^2 |v_j|^2) for every query of the unit (fp64), with the kernels' masking:
    window query r of a causal window sees tokens <= n - w + r."""
    K = np.asarray(u["K"], dtype=np.float64)
    vn = np.linalg.norm(np.asarray(u["V"], dtype=np.float64), axis=1)
    qs = []
    for h in range(cfg.g):
        qs.append(np.asarray(u["Q_W"][h], dtype=np.float64).reshape(-1, cfg.d))
        qs.append(np.asarray(u["Q_look"][h], dtype=np.float64).reshape(-1, cfg.d))
    out = []
    row = 0
    for blk in qs:
        sc = blk @ K.T / np.sqrt(cfg.d)
        for i in range(blk.shape[0]):
            srow = sc[i].copy()
            is_window = blk.shape[0] == cfg.w and cfg.window_causal
            if is_window:
                srow[cfg.n - cfg.w + i + 1:] = -np.inf
            a = np.exp(srow - lse[row])
            out.append(float(np.sqrt((a * a) @ (vn * vn))))
            row += 1
    return np.array(out)


def _check_units(cfg, inp, run, units, what):
    ref = oracle.lorekv_config_units(cfg, inp, units)
    S = run.scores.double().cpu().numpy()
    kept = run.kept_idx.cpu().numpy()
    for (s, l, kh), r in ref.items():
        ui = _unit_index(cfg, s, l, kh)
        assert_scores_close(S[ui], r["S"], cfg.dtype, f"{what} unit {ui}")
        assert_kept_matches(kept[ui, :run.cap], r["S"], sink=cfg.sink, w=cfg.w, chunk=cfg.chunk,
                            B=cfg.B, rtol=SCORE_RTOL[cfg.dtype], what=f"{what} unit {ui}")


@pytest.mark.parametrize("case", list(MULTITILE_CASES))
def test_multitile_ranges_match_oracle(case):
    """Attention statistics and the whole pass when every attention CTA walks several K/V tiles
    (ring wrap-around, per-half partial merge; at GQA 5 also the single-tile CTAs' alternating S
    buffers)."""
    cfg, units = MULTITILE_CASES[case]
    inp = synth.lorekv_inputs(cfg, "cpu")
    g = {k: v.to(_dev()) for k, v in inp.items()}
    pb = api.LorekvProblem.from_config(cfg)
    ws = torch.empty(api.lorekv_workspace_size(pb), dtype=torch.uint8, device=_dev())
    Qu = cfg.g * cfg.queries_per_head
    lse = torch.empty(cfg.units, Qu, device=_dev())
    o = torch.empty(cfg.units, Qu, cfg.d, device=_dev())
    api.lorekv_attention_stats(pb, g["K"], g["V"], g["Q_W"], g["Q_look"], lse, o, ws)
    api.kve_check_device()
    lse, o = lse.double().cpu().numpy(), o.double().cpu().numpy()
    for (s, l, kh) in units:
        u = synth.unit_slice(cfg, inp, s, l, kh)
        eye = np.stack([np.eye(cfg.d)] * cfg.g)
        r = oracle.lorekv_unit(u["K"], u["V"], u["Q_W"], u["Q_look"], eye, np.ones(cfg.M) / cfg.M,
                               M=cfg.M, T=cfg.T, sink=cfg.sink, lambda_L=1.0, eps=cfg.eps,
                               window_causal=cfg.window_causal, want=("lse", "o"))
        ui = _unit_index(cfg, s, l, kh)
        lse_ref, o_ref = r["lse"].reshape(-1), r["o"].reshape(-1, cfg.d)
        assert np.allclose(lse[ui], lse_ref, rtol=0, atol=2e-3 * np.maximum(1, np.abs(lse_ref)).max())
        # o = sum_j a_j v_j with every a_j rounded to bf16 on its way to the tensor cores:
        # independent relative errors in [-2^-9, 2^-9] give |o_gpu - o| an RMS of
        # 2^-9/sqrt(3) sqrt(sum_j a_j^2 |v_j|^2); allow 4 sigma plus fp32 accumulation
        err = np.linalg.norm(o[ui] - o_ref, axis=1)
        sigma = 2.0 ** -9 / np.sqrt(3.0) * _attention_weighted_vnorm(cfg, u, lse_ref)
        bound = 4.0 * sigma + 1e-5 * np.linalg.norm(o_ref, axis=1) + 1e-6
        assert np.all(err <= bound), (ui, float((err / bound).max()))
    run = _run_pass(cfg, g)
    _check_units(cfg, inp, run, units, "multitile")


@pytest.mark.parametrize("case", list(MULTITILE_CASES))
def test_eviction_pass_rising_scores(case):
    """The second half of every unit's keys is shifted by 30 along the unit's mean query direction:
    nearly every query's running maximum rises by more than 2^8 (in exp2 units) half-way through
    the cache, which takes the attention pass's lazy-rescale path inside multi-tile ranges, while
    attention stays spread over the shifted half (largest probability about 0.2)."""
    cfg, units = MULTITILE_CASES[case]
    inp = synth.lorekv_inputs(cfg, "cpu")
    K = inp["K"].float()
    for s in range(cfg.S):
        for l in range(cfg.L):
            for kh in range(cfg.Hkv):
                heads = slice(kh * cfg.g, (kh + 1) * cfg.g)
                qs = torch.cat([inp["Q_W"][s, l, heads].reshape(-1, cfg.d),
                                inp["Q_look"][s, l, heads].reshape(-1, cfg.d)]).float()
                mu = qs.mean(0)
                K[s, l, kh, cfg.n // 2:] += 30.0 * mu / mu.norm()
    inp["K"] = K.to(inp["K"].dtype)
    g = {k: v.to(_dev()) for k, v in inp.items()}
    run = _run_pass(cfg, g)
    _check_units(cfg, inp, run, units, "rising")


def test_layer_chunks_match_whole_pass():
    """With lambda_D = 0 the units and omega do not depend on other layers, so the pass issued per
    chunk of layers (sub-shape views of the same buffers) gives the whole pass's results."""
    import dataclasses
    cfg = MULTITILE
    assert cfg.lambda_D == 0
    g = {k: v.to(_dev()) for k, v in synth.lorekv_inputs(cfg, "cpu").items()}
    pb, Lf, G = _prepare(cfg, g)
    whole = api.LorekvPass(pb, _dev())
    whole.run(g, Lf, G)
    cl, upc = 2, 2 * cfg.Hkv
    sub = api.LorekvPass(dataclasses.replace(pb, n_layers=cl), _dev())
    for c in range(cfg.L // cl):
        part = {k: (g[k][:, c * cl:(c + 1) * cl] if k in ("K", "V", "Q_W", "Q_look") else g[k])
                for k in g}
        sub.run(part, Lf[c * cl:(c + 1) * cl], G[c * cl:(c + 1) * cl])
        api.kve_check_device()
        u0, u1 = c * upc, (c + 1) * upc
        assert torch.allclose(sub.omega, whole.omega, rtol=1e-6, atol=0)
        S_w, S_c = whole.scores[u0:u1].double(), sub.scores.double()
        assert torch.allclose(S_c, S_w, rtol=1e-4, atol=1e-9 * float(S_w.max())), c
        # kept sets of the chunk are the top-B of the chunk's own scores
        kept = sub.kept_idx.cpu().numpy()
        Sc = S_c.cpu().numpy()
        for ui in range(upc):
            assert_kept_valid_for_own_scores(kept[ui], Sc[ui], sink=cfg.sink, w=cfg.w,
                                             chunk=cfg.chunk, B=cfg.B, what=f"chunk {c} unit {ui}")


def test_output_fidelity_matches_oracle():
    """Attention-output fidelity of the compressed cache: held-out queries (the generator's queries
    under another seed, seeing the whole cache) attend over the full K/V and over the compacted
    K'/V'; each query's cosine of the two outputs matches the oracle's fp64 attention over the same
    kept rows, and the reported mean is the mean of the cosines."""
    import dataclasses
    cfg = SMALL["bf16_gqa4_D"]
    inp = synth.lorekv_inputs(cfg, "cpu")
    held = synth.lorekv_inputs(cfg.replace(seed=cfg.seed + 1000), "cpu")
    g = {k: v.to(_dev()) for k, v in inp.items()}
    run = _run_pass(cfg, g)
    pe = dataclasses.replace(api.LorekvProblem.from_config(cfg), window_causal=0)
    pc = dataclasses.replace(pe, n_tokens=run.cap)  # the compacted cache as a cache of cap tokens
    Qw, Ql = held["Q_W"].to(_dev()), held["Q_look"].to(_dev())
    Qu = cfg.g * cfg.queries_per_head
    lse = torch.empty(cfg.units, Qu, device=_dev())
    o_full = torch.empty(cfg.units, Qu, cfg.d, device=_dev())
    o_comp = torch.empty_like(o_full)
    for pb, K, V, o in ((pe, g["K"], g["V"], o_full), (pc, run.K_out, run.V_out, o_comp)):
        ws = torch.empty(api.lorekv_workspace_size(pb), dtype=torch.uint8, device=_dev())
        api.lorekv_attention_stats(pb, K, V, Qw, Ql, lse, o, ws)
    cos = torch.empty(cfg.units * Qu, device=_dev())
    mean = torch.empty(1, device=_dev())
    api.lorekv_output_fidelity(o_full.view(-1, cfg.d), o_comp.view(-1, cfg.d), cos, mean)
    api.kve_check_device()
    cos_g = cos.double().cpu().numpy().reshape(cfg.units, Qu)
    kept = run.kept_idx.long().cpu().numpy()
    eye = np.stack([np.eye(cfg.d)] * cfg.g)
    for (s, l, kh) in _all_units(cfg):
        ui = _unit_index(cfg, s, l, kh)
        u, h = synth.unit_slice(cfg, inp, s, l, kh), synth.unit_slice(cfg, held, s, l, kh)
        idx = kept[ui, :run.cap]
        outs = []
        for K, V in ((u["K"], u["V"]), (u["K"][idx], u["V"][idx])):
            r = oracle.lorekv_unit(K, V, h["Q_W"], h["Q_look"], eye, np.ones(cfg.M) / cfg.M,
                                   M=cfg.M, T=cfg.T, sink=cfg.sink, lambda_L=1.0, eps=cfg.eps,
                                   window_causal=0, want=("o",))
            outs.append(r["o"].reshape(-1, cfg.d))
        of, oc = outs
        ref = (of * oc).sum(1) / (np.linalg.norm(of, axis=1) * np.linalg.norm(oc, axis=1))
        assert np.allclose(cos_g[ui], ref, rtol=0, atol=3e-3), (ui, float(np.abs(cos_g[ui] - ref).max()))
    assert float(mean.item()) == pytest.approx(float(cos_g.mean()), rel=1e-5)


def test_masked_logits_match_oracle():
    """Logits of -inf (masked vocabulary entries, common in real decoders) contribute nothing to
    lse, H and log q: omega and the scores match the oracle, which treats 0 log 0 as 0."""
    cfg = SMALL["bf16_gqa4_D"]
    inp = synth.lorekv_inputs(cfg, "cpu")
    gen = torch.Generator().manual_seed(5)
    mask = torch.rand(inp["logits"].shape, generator=gen) < 0.3
    rows = torch.arange(inp["sampled"].numel())
    mask.view(-1, cfg.vocab)[rows, inp["sampled"].view(-1).long()] = False  # y stays finite
    mask[..., :3] = True                                                     # a masked prefix
    inp["logits"] = inp["logits"].masked_fill(mask, float("-inf"))
    g = {k: v.to(_dev()) for k, v in inp.items()}
    run = _run_pass(cfg, g)
    om = run.omega.double().cpu().numpy()
    assert np.all(np.isfinite(om))
    S = run.scores.double().cpu().numpy()
    units = [(0, 0, 0), (1, 1, 1)]
    for (s, l, kh), r in oracle.lorekv_config_units(cfg, inp, units).items():
        assert np.allclose(om[s], r["omega"], rtol=OMEGA_RTOL, atol=0), s
        assert_scores_close(S[_unit_index(cfg, s, l, kh)], r["S"], cfg.dtype, "masked logits")


def test_scores_are_deterministic():
    cfg = SMALL["bf16_gqa4_D"]
    g = {k: v.to(_dev()) for k, v in synth.lorekv_inputs(cfg, "cpu").items()}
    a = _run_pass(cfg, g)
    S1, k1 = a.scores.clone(), a.kept_idx.clone()
    b = _run_pass(cfg, g)
    assert torch.equal(S1, b.scores) and torch.equal(k1, b.kept_idx)


FULL = ["mistral", "llama", "qwen"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload_sampled_units(name):
    cfg = synth.LOREKV_CONFIGS[name]
    torch.cuda.empty_cache()
    g = synth.lorekv_inputs(cfg, _dev())
    run = _run_pass(cfg, g)
    S = run.scores
    # every unit: protected tokens score 0, scores finite and non-negative, kept sets valid
    assert torch.isfinite(S).all() and (S >= 0).all()
    assert (S[:, :cfg.sink] == 0).all() and (S[:, cfg.n - cfg.w:] == 0).all()
    kept = run.kept_idx.cpu().numpy()
    Sc = S.cpu().numpy()
    for ui in range(cfg.units):
        assert_kept_valid_for_own_scores(kept[ui], Sc[ui], sink=cfg.sink, w=cfg.w,
                                         chunk=cfg.chunk, B=cfg.B, what=f"{name} unit {ui}")
    # sampled units against the oracle
    units = [(0, 0, 0), (cfg.S - 1, cfg.L // 2, cfg.Hkv - 1), (cfg.S - 1, cfg.L - 1, cfg.Hkv // 2)]
    ref = oracle.lorekv_config_units(cfg, g, units)
    om = run.omega.double().cpu().numpy()
    for (s, l, kh), r in ref.items():
        ui = _unit_index(cfg, s, l, kh)
        assert np.allclose(om[s], r["omega"], rtol=OMEGA_RTOL, atol=0)
        assert_scores_close(Sc[ui].astype(np.float64), r["S"], cfg.dtype, f"{name} unit {ui}")
        assert_kept_matches(kept[ui], r["S"], sink=cfg.sink, w=cfg.w, chunk=cfg.chunk, B=cfg.B,
                            rtol=SCORE_RTOL[cfg.dtype], what=f"{name} unit {ui}")
    idx = run.kept_idx.long()
    Kf = g["K"].reshape(cfg.units, cfg.n, cfg.d)
    assert torch.equal(run.K_out, torch.gather(Kf, 1, idx[..., None].expand(-1, -1, cfg.d)))
    del g, run
    torch.cuda.empty_cache()
