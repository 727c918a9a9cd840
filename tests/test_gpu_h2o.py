"""GPU parity of the H2O mode (prefill + per-step decode eviction) against the fp64 oracle.

Eviction decisions are compared teacher-forced: after every step the oracle scores the same
pre-eviction set; the GPU's evictee must have an oracle accumulated score within
min * (1 + 1e-3) + 1e-6 * max of the true minimum among the candidates, and the oracle then adopts
the GPU's retained set, so one near-tie cannot make the two runs diverge.
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_02_gb300 import api, synth

pytestmark = pytest.mark.gpu

OUT_RTOL = 2e-3
ACC_RTOL = 1e-4


def _dev():
    return torch.device("cuda:0")


def _unit_coords(cfg, u):
    b, rest = divmod(u, cfg.L * cfg.H)
    l, h = divmod(rest, cfg.H)
    return b, l, h


def _check_state(st_gpu, units, oracles, what):
    """Compare the exported state of the listed units with their oracle states."""
    pos = st_gpu["pos"].cpu().numpy()
    acc = st_gpu["acc"].double().cpu().numpy()
    cnt = st_gpu["count"].cpu().numpy()
    for u in units:
        o = oracles[u]
        valid = pos[u] >= 0
        assert cnt[u] == valid.sum() == len(o.pos), (what, u)
        gp = pos[u][valid]
        ga = acc[u][valid]
        order = np.argsort(gp)
        gp, ga = gp[order], ga[order]
        oo = np.argsort(o.pos)
        assert gp.tolist() == o.pos[oo].tolist(), (what, u)
        if len(o.pos):  # a budget of k_t = 0 leaves the unit's cache empty
            assert np.allclose(ga, o.acc[oo], rtol=ACC_RTOL, atol=1e-6 * o.acc.max()), (what, u)


def _check_prefill(ex, units, orc, cfg, hin):
    """The GPU's first compression keeps the r most recent prompt tokens plus the highest prefill
    scores; positions that differ from the oracle's choice must sit at the threshold within the
    accumulated-score tolerance. The oracle then adopts the GPU's set."""
    pos = ex["pos"].cpu().numpy()
    P = cfg.prompt
    k, r = oracle.h2o_budget(P, cfg.budget_frac)
    for u in units:
        o = orc[u]
        g_set = set(pos[u][pos[u] >= 0].tolist())
        o_set = set(o.pos.tolist())
        assert len(g_set) == len(o_set) == min(k, P), u
        assert set(range(P - r, P)) <= g_set, u
        diff = g_set ^ o_set
        if diff:
            cand = o.prefill_acc[: P - r]
            tau = np.sort(cand)[::-1][k - r - 1]
            for p in diff:
                assert abs(o.prefill_acc[p] - tau) <= ACC_RTOL * tau, (u, p)
            b, l, h = _unit_coords(cfg, u)
            o.adopt_prefill(g_set, hin["K"][b, l, h], hin["V"][b, l, h])


def _advance(o, q, k, v, kept_gpu, tn, frac, what):
    """One oracle step teacher-forced to the GPU's retained set; returns the oracle output and
    the magnitude sum_j p_j |v_j| of its terms."""
    o_ref, _, pre = o.step(q, k, v, evict=False)
    p, _ = oracle.h2o_attend(o.K, o.V, q)
    mag = p @ np.abs(o.V)
    k_t, r_t = oracle.h2o_budget(tn, frac)
    pre_pos = pre["pos"].tolist()
    gone = [p for p in pre_pos if p not in kept_gpu]
    want = max(len(pre_pos) - k_t, 0)
    assert len(gone) == want <= 1, (what, gone, want)
    assert kept_gpu <= set(pre_pos), what
    if gone:
        cand = [i for i, p in enumerate(pre_pos) if p < tn - r_t]
        accs = pre["acc"][cand]
        g_acc = pre["acc"][pre_pos.index(gone[0])]
        assert gone[0] < tn - r_t, f"{what}: evicted a protected recent token"
        assert g_acc <= accs.min() * (1 + 1e-3) + 1e-6 * pre["acc"].max(), what
    o.adopt(sorted(kept_gpu))
    return o_ref, mag


def _check_out(o_gpu, o_ref, mag, what, half_ulp=2.0 ** -11):
    """attn_out is written in the state's 16-bit type (fp16 here): each component carries that
    rounding (half an ulp, 2^-11 relative, plus the fp16 subnormal spacing); the fp32
    accumulation and exponentials add at most 1e-5 of the terms' magnitude
    mag_k = sum_j p_j |v_jk|. Both stay inside the rel 2e-3 budget wherever |o_k| is not a
    small difference of large terms."""
    err = np.abs(o_gpu - o_ref)
    lim = half_ulp * np.abs(o_ref) + 1e-5 * mag + 2.0 ** -24
    assert np.all(err <= lim), (what, float((err / lim).max()))
    assert np.all(err <= OUT_RTOL * np.abs(o_ref) + 1e-5 * mag + 2.0 ** -24), what


def _teacher_forced_run(cfg, hin, units, steps, check_kv=True):
    dev = _dev()
    st = api.h2o_state_create(cfg.batch, cfg.L, cfg.H, cfg.d, cfg.prompt + steps,
                              cfg.budget_frac, torch.float16)
    Kp, Vp, Qp = hin["K"], hin["V"], hin["Q"]
    st.prefill(Kp, Vp, Qp)
    orc = {}
    for u in units:
        b, l, h = _unit_coords(cfg, u)
        orc[u] = oracle.H2OUnit(Kp[b, l, h], Vp[b, l, h], Qp[b, l, h], cfg.budget_frac,
                                cfg.prompt + steps)
    ex = st.export()
    _check_prefill(ex, units, orc, cfg, hin)
    _check_state(ex, units, orc, "prefill")
    out = torch.empty(cfg.batch, cfg.L, cfg.H, cfg.d, dtype=torch.float16, device=dev)
    for t in range(steps):
        q, k, v = hin["q"][t], hin["k"][t], hin["v"][t]
        st.decode_step(q, k, v, out)
        ex = st.export()
        pos = ex["pos"].cpu().numpy()
        o_gpu = out.double().cpu().numpy().reshape(-1, cfg.d)
        tn = cfg.prompt + t + 1
        for u in units:
            b, l, h = _unit_coords(cfg, u)
            kept_gpu = set(pos[u][pos[u] >= 0].tolist())
            o_ref, mag = _advance(orc[u], q[b, l, h], k[b, l, h], v[b, l, h], kept_gpu, tn,
                                  cfg.budget_frac, (t, u))
            _check_out(o_gpu[u], o_ref, mag, (t, u))
        _check_state(ex, units, orc, f"step {t}")
        if check_kv:
            Kx, Vx = ex["K"].cpu(), ex["V"].cpu()
            for u in units:
                b, l, h = _unit_coords(cfg, u)
                for slot in np.flatnonzero(pos[u] >= 0):
                    p = int(pos[u][slot])
                    if p < cfg.prompt:
                        ks, vs = Kp[b, l, h, p], Vp[b, l, h, p]
                    else:
                        ks, vs = hin["k"][p - cfg.prompt][b, l, h], hin["v"][p - cfg.prompt][b, l, h]
                    assert torch.equal(Kx[u, slot], ks.cpu()), (t, u, p)
                    assert torch.equal(Vx[u, slot], vs.cpu()), (t, u, p)
    st.close()


def test_h2o_tiny_teacher_forced():
    cfg = synth.H2O_CONFIGS["tiny"]
    hin = {k: v.to(_dev()) for k, v in synth.h2o_inputs(cfg, "cpu").items()}
    _teacher_forced_run(cfg, hin, list(range(cfg.units)), cfg.steps)


_BUDGET_CASES = [("tiny", 1.0), ("tiny", 0.03), ("tiny", 0.01), ("d128", 0.01)]


@pytest.mark.parametrize("shape,frac", _BUDGET_CASES, ids=[f"{a}-{b}" for a, b in _BUDGET_CASES])
def test_h2o_budget_extremes_teacher_forced(shape, frac):
    """Budgets at the edges of H2O's rule (H2O page, Section 4.1, Algorithm 1): 1.0 never evicts;
    0.03 and 0.01 hold k_t = floor(frac t) = 0-3 tokens (the recent part r_t = floor(k_t / 2) is
    0 or 1, so the new token itself can be the one evicted, and the prefill compresses the prompt
    to one token or none). The budget crosses the C-ABI as a float, so both sides take the float's
    value (0.03f < 0.03: floor(0.03f * 100) = 2)."""
    frac32 = float(np.float32(frac))
    base = (synth.H2O_CONFIGS["tiny"] if shape == "tiny" else
            synth.H2OConfig("b128", "f16", batch=1, L=1, H=2, d=128, prompt=150, steps=40))
    cfg = base.replace(budget_frac=frac32)
    hin = {k: v.to(_dev()) for k, v in synth.h2o_inputs(cfg, "cpu").items()}
    _teacher_forced_run(cfg, hin, list(range(cfg.units)), cfg.steps)


def test_h2o_d128_batch_teacher_forced():
    cfg = synth.H2OConfig("mid", "f16", batch=2, L=2, H=3, d=128, prompt=512, steps=24)
    hin = {k: v.to(_dev()) for k, v in synth.h2o_inputs(cfg, "cpu").items()}
    _teacher_forced_run(cfg, hin, list(range(cfg.units)), cfg.steps)


def test_h2o_full_size_sampled_units():
    """OPT-30B-shaped decode (batch 64, 48 layers, 56 heads, prompt 512) for a few steps;
    sampled units checked teacher-forced, every unit checked for the budget invariants."""
    cfg = synth.H2O_CONFIGS["opt30b"]
    steps = 8
    torch.cuda.empty_cache()
    hin = synth.h2o_inputs(cfg, _dev(), steps=steps)
    units = [0, 1, cfg.units // 2, cfg.units - 1]
    dev = _dev()
    st = api.h2o_state_create(cfg.batch, cfg.L, cfg.H, cfg.d, cfg.prompt + cfg.steps,
                              cfg.budget_frac, torch.float16)
    st.prefill(hin["K"], hin["V"], hin["Q"])
    orc = {}
    for u in units:
        b, l, h = _unit_coords(cfg, u)
        orc[u] = oracle.H2OUnit(hin["K"][b, l, h], hin["V"][b, l, h], hin["Q"][b, l, h],
                                cfg.budget_frac, cfg.prompt + cfg.steps)
    pos0 = torch.empty(cfg.units, st.capacity, dtype=torch.int32, device=dev)
    acc0 = torch.empty(cfg.units, st.capacity, dtype=torch.float32, device=dev)
    cnt0 = torch.empty(cfg.units, dtype=torch.int32, device=dev)
    api._check(api.lib().h2o_export(st.h, None, None, pos0.data_ptr(), acc0.data_ptr(),
                                    cnt0.data_ptr(), torch.cuda.current_stream().cuda_stream))
    ex0 = {"pos": pos0, "acc": acc0, "count": cnt0}
    _check_prefill(ex0, units, orc, cfg, hin)
    _check_state(ex0, units, orc, "prefill")
    out = torch.empty(cfg.batch, cfg.L, cfg.H, cfg.d, dtype=torch.float16, device=dev)
    for t in range(steps):
        q, k, v = hin["q"][t], hin["k"][t], hin["v"][t]
        st.decode_step(q, k, v, out)
        pos = torch.empty(cfg.units, st.capacity, dtype=torch.int32, device=dev)
        acc = torch.empty(cfg.units, st.capacity, dtype=torch.float32, device=dev)
        cnt = torch.empty(cfg.units, dtype=torch.int32, device=dev)
        api._check(api.lib().h2o_export(st.h, None, None, pos.data_ptr(), acc.data_ptr(),
                                        cnt.data_ptr(), torch.cuda.current_stream().cuda_stream))
        tn = cfg.prompt + t + 1
        k_t, r_t = oracle.h2o_budget(tn, cfg.budget_frac)
        assert (cnt == k_t).all()
        assert torch.isfinite(out.float()).all()
        pos_c = pos.cpu().numpy()
        o_gpu = out.reshape(-1, cfg.d)[units].double().cpu().numpy()
        for i, u in enumerate(units):
            b, l, h = _unit_coords(cfg, u)
            kept_gpu = set(pos_c[u][pos_c[u] >= 0].tolist())
            o_ref, mag = _advance(orc[u], q[b, l, h], k[b, l, h], v[b, l, h], kept_gpu, tn,
                                  cfg.budget_frac, (t, u))
            _check_out(o_gpu[i], o_ref, mag, (t, u))
    st.close()
    del hin
    torch.cuda.empty_cache()


_PREFILL_CASES = [
    # (prompt length, dtype, (batch, layers, heads)): ragged last tiles, one to five 128-token
    # tiles, bf16 and f16, and more units than SMs (the prefill kernel walks units persistently)
    (100, "f16", (1, 1, 3)),
    (129, "bf16", (1, 2, 2)),
    (300, "f16", (1, 1, 4)),
    (512, "bf16", (1, 1, 2)),
    (640, "f16", (1, 1, 2)),
    (256, "f16", (2, 10, 16)),
]


@pytest.mark.parametrize("P,dtype,shape", _PREFILL_CASES,
                         ids=[f"P{c[0]}-{c[1]}-u{c[2][0] * c[2][1] * c[2][2]}" for c in _PREFILL_CASES])
def test_h2o_prefill_shapes(P, dtype, shape):
    """Prefill scores and the first compression at d_head 128 against the oracle: retained
    positions, their accumulated scores and their K/V rows."""
    b, L, H = shape
    cfg = synth.H2OConfig(f"prefill{P}", dtype, batch=b, L=L, H=H, d=128, prompt=P, steps=1)
    hin = {k: v.to(_dev()) for k, v in synth.h2o_inputs(cfg, "cpu", steps=1).items()}
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    st = api.h2o_state_create(b, L, H, 128, P + 1, cfg.budget_frac, tdt)
    st.prefill(hin["K"], hin["V"], hin["Q"])
    n = cfg.units
    units = list(range(n)) if n <= 16 else sorted({0, 1, 150, 151, 152, 153, n // 2, n - 2, n - 1})
    orc = {}
    for u in units:
        bb, l, h = _unit_coords(cfg, u)
        orc[u] = oracle.H2OUnit(hin["K"][bb, l, h], hin["V"][bb, l, h], hin["Q"][bb, l, h],
                                cfg.budget_frac, P + 1)
    ex = st.export()
    _check_prefill(ex, units, orc, cfg, hin)
    _check_state(ex, units, orc, "prefill")
    pos = ex["pos"].cpu().numpy()
    Kx, Vx = ex["K"].cpu(), ex["V"].cpu()
    for u in units:
        bb, l, h = _unit_coords(cfg, u)
        for slot in np.flatnonzero(pos[u] >= 0):
            p = int(pos[u][slot])
            assert torch.equal(Kx[u, slot], hin["K"][bb, l, h, p].cpu()), (u, p)
            assert torch.equal(Vx[u, slot], hin["V"][bb, l, h, p].cpu()), (u, p)
    st.close()


def test_h2o_prefill_allocates_nothing():
    """The state created by h2o_state_create holds the prefill's scratch: a prefill (and a decode
    step) leaves the device's free memory unchanged. A first state runs once beforehand so that
    loading the kernels is not counted."""
    cfg = synth.H2OConfig("prefill_noalloc", "f16", batch=2, L=2, H=8, d=128, prompt=384, steps=2)
    hin = {k: v.to(_dev()) for k, v in synth.h2o_inputs(cfg, "cpu", steps=2).items()}
    out = torch.empty(cfg.batch, cfg.L, cfg.H, cfg.d, dtype=torch.float16, device=_dev())
    states = []
    for _ in range(2):
        st = api.h2o_state_create(cfg.batch, cfg.L, cfg.H, cfg.d, cfg.prompt + 2, cfg.budget_frac,
                                  torch.float16)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        st.prefill(hin["K"], hin["V"], hin["Q"])
        st.decode_step(hin["q"][0], hin["k"][0], hin["v"][0], out)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        states.append(st)
    assert free1 == free0, f"prefill + decode step changed free device memory by {free0 - free1}"
    for st in states:
        st.close()
