"""Out-of-bounds write checks without a sanitizer: every output and workspace of the C-ABI calls
sits between two guard regions filled with a fixed byte pattern, and the guards must be intact
after the call (and the stream synchronised). The configurations cover the tensor-core and
CUDA-core paths, ragged tiles and GQA."""
import pytest
import torch

from kv_cache_eviction_02_gb300 import api, synth

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side
PATTERN = 0xA5


class Guarded:
    """A contiguous tensor of the given shape inside a byte buffer with guard regions."""

    def __init__(self, shape, dtype):
        n = 1
        for s in shape:
            n *= s
        es = torch.empty(0, dtype=dtype).element_size()
        self.nbytes = n * es
        self.buf = torch.full((GUARD + self.nbytes + GUARD,), PATTERN, dtype=torch.uint8,
                              device="cuda:0")
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(*shape)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        return bool((self.buf[:GUARD] == PATTERN).all() and
                    (self.buf[GUARD + self.nbytes:] == PATTERN).all())


def _ws(nbytes):
    return Guarded((max(nbytes, 1),), torch.uint8)


LOREKV = [
    synth.LOREKV_CONFIGS["tiny"],
    synth.LorekvConfig("bf16_gqa4", "bf16", S=2, L=2, Hq=8, Hkv=2, d=128, d_model=256, n=1000,
                       vocab=5000, beta=1.0, gamma=1.0, lambda_D=0.3),
    synth.LorekvConfig("f32_ragged_d32", "f32", S=1, L=2, Hq=4, Hkv=2, d=32, d_model=64, n=300,
                       vocab=300, B=64, keys="normal"),
]


@pytest.mark.parametrize("cfg", LOREKV, ids=lambda c: c.name)
def test_lorekv_calls_stay_inside_their_buffers(cfg):
    g = {k: v.to("cuda:0") for k, v in synth.lorekv_inputs(cfg, "cpu").items()}
    pb = api.LorekvProblem.from_config(cfg)
    f32 = torch.float32
    Lf, G = Guarded((cfg.L, cfg.Hq, cfg.d, cfg.d), f32), Guarded((cfg.L, cfg.Hq, cfg.d, cfg.d), f32)
    api.lorekv_prepare_wo(pb, g["W_O"], Lf.t, G.t)
    ws = _ws(api.lorekv_workspace_size(pb))
    units, Qu = cfg.units, cfg.g * cfg.queries_per_head
    scores, omega = Guarded((units, cfg.n), f32), Guarded((cfg.S, cfg.M), f32)
    api.lorekv_score(pb, g["K"], g["V"], g["Q_W"], g["Q_look"], Lf.t, G.t, g["logits"],
                     g["sampled"], scores.t, omega.t, ws.t)
    lse, o = Guarded((units, Qu), f32), Guarded((units, Qu, cfg.d), f32)
    api.lorekv_attention_stats(pb, g["K"], g["V"], g["Q_W"], g["Q_look"], lse.t, o.t, ws.t)
    cap = api.lorekv_kept_capacity(pb)
    dt = g["K"].dtype
    kept, klen = Guarded((units, cap), torch.int32), Guarded((units,), torch.int32)
    Ko, Vo = Guarded((units, cap, cfg.d), dt), Guarded((units, cap, cfg.d), dt)
    api.lorekv_select_compact(pb, scores.t, g["K"], g["V"], kept.t, klen.t, Ko.t, Vo.t)
    cos, mean = Guarded((units * Qu,), f32), Guarded((1,), f32)
    api.lorekv_output_fidelity(o.t.view(-1, cfg.d), o.t.view(-1, cfg.d), cos.t, mean.t)
    api.kve_check_device()
    for name, b in dict(L=Lf, G=G, ws=ws, scores=scores, omega=omega, lse=lse, o=o, kept=kept,
                        kept_len=klen, K_out=Ko, V_out=Vo, cos=cos, mean=mean).items():
        assert b.intact(), name


CC = [
    synth.CC_CONFIGS["tiny"],  # fp32, CUDA-core path
    synth.CC_CONFIGS["tiny"].replace(dtype="bf16", d=128, n=389, Hq=6, Hkv=2, d_model=160,
                                     batch=2, sink=2, J=300),  # tensor-core path
]


@pytest.mark.parametrize("cfg", CC, ids=lambda c: f"{c.dtype}_d{c.d}")
def test_counter_causal_calls_stay_inside_their_buffers(cfg):
    inp = synth.cc_inputs(cfg, "cuda:0")
    pb = api.CcProblem(cfg.batch, cfg.Hq, cfg.Hkv, cfg.d, cfg.d_model, cfg.n, cfg.vocab,
                       {"f32": api.KVE_F32, "bf16": api.KVE_BF16}[cfg.dtype], cfg.sink, cfg.J)
    ws = _ws(api.cc_workspace_size(pb))
    s = Guarded((cfg.batch, cfg.n), torch.float32)
    api.cc_surprise(pb, inp["K"], inp["V"], inp["Q_fresh"], inp["H_last"], inp["W_O"],
                    inp["W_U"], inp["tokens"], s.t, ws.t)
    dt = inp["K"].dtype
    kept, Xo = Guarded((cfg.batch, cfg.J), torch.int32), Guarded((cfg.batch, cfg.J), torch.int32)
    Ko, Vo = (Guarded((cfg.batch, cfg.Hkv, cfg.J, cfg.d), dt),
              Guarded((cfg.batch, cfg.Hkv, cfg.J, cfg.d), dt))
    api.cc_select_compact(pb, s.t, inp["K"], inp["V"], inp["tokens"], kept.t, Ko.t, Vo.t, Xo.t)
    api.kve_check_device()
    for name, b in dict(ws=ws, surprise=s, kept=kept, tokens_out=Xo, K_out=Ko, V_out=Vo).items():
        assert b.intact(), name


def test_refresh_cycle_export_stays_inside_its_buffers():
    cfg = synth.CC_CONFIGS["tiny"].replace(dtype="bf16", d=128, n=90, Hq=4, Hkv=2, d_model=256,
                                           batch=2, sink=2)
    inp = synth.cc_inputs(cfg, "cuda:0")
    J, h = 30, 8
    pb = api.CcProblem(cfg.batch, cfg.Hq, cfg.Hkv, cfg.d, cfg.d_model, J + h, cfg.vocab,
                       api.KVE_BF16, cfg.sink, J)
    cache = api.CcCache(pb)
    for t in range(0, 88, 4):
        sl = slice(t, t + 4)
        cache.step(inp["K"][:, :, sl].contiguous(), inp["V"][:, :, sl].contiguous(),
                   inp["Q_fresh"][:, :, sl].contiguous(), inp["H_last"][:, sl].contiguous(),
                   inp["tokens"][:, sl].contiguous(), inp["W_O"], inp["W_U"])
    n = cache.length
    bf = torch.bfloat16
    outs = dict(K=Guarded((2, 2, n, 128), bf), V=Guarded((2, 2, n, 128), bf),
                Q=Guarded((2, 4, n, 128), bf), H=Guarded((2, n, 256), bf),
                tokens=Guarded((2, n), torch.int32), pos=Guarded((2, n), torch.int32))
    from kv_cache_eviction_02_gb300.api import _ptr, _stream, lib, _check
    _check(lib().cc_cache_export(cache.h, *[_ptr(outs[k].t) for k in ("K", "V", "Q", "H",
                                                                       "tokens", "pos")],
                                 _stream(None)))
    api.kve_check_device()
    for name, b in outs.items():
        assert b.intact(), name
    cache.close()


def test_h2o_export_stays_inside_its_buffers():
    hc = synth.H2O_CONFIGS["tiny"]
    hin = synth.h2o_inputs(hc, "cpu", steps=3)
    st = api.H2OState(hc.batch, hc.L, hc.H, hc.d, hc.prompt + 3, hc.budget_frac, torch.float16)
    st.prefill(hin["K"].cuda(), hin["V"].cuda(), hin["Q"].cuda())
    out = Guarded((hc.batch, hc.L, hc.H, hc.d), torch.float16)
    for t in range(3):
        st.decode_step(hin["q"][t].cuda(), hin["k"][t].cuda(), hin["v"][t].cuda(), out.t)
    cap, u = st.capacity, st.units
    K, V = Guarded((u, cap, hc.d), torch.float16), Guarded((u, cap, hc.d), torch.float16)
    pos, acc = Guarded((u, cap), torch.int32), Guarded((u, cap), torch.float32)
    cnt = Guarded((u,), torch.int32)
    from kv_cache_eviction_02_gb300.api import _ptr, _stream, lib, _check
    _check(lib().h2o_export(st.h, _ptr(K.t), _ptr(V.t), _ptr(pos.t), _ptr(acc.t), _ptr(cnt.t),
                            _stream(None)))
    api.kve_check_device()
    for name, b in dict(attn_out=out, K=K, V=V, pos=pos, acc=acc, count=cnt).items():
        assert b.intact(), name
    st.close()
