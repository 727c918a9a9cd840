"""Seeded synthetic inputs for the LORE-KV eviction pass and the H2O decode mode.

This module only draws random tensors with the shapes and distributions of the workloads; it
holds none of the scoring, selection or attention arithmetic. Both the CUDA path (through the
binding) and the fp64 oracle read the tensors it returns, so the two sides always see the same
rounded input values.

Workloads (LORE-KV page, "Hyperparameters" table for w, M, T, lambda_L, eps, chunk and the /E and
/D presets; H2O page, Section 5 for the OPT-30B decode shape):

* ``tiny``     fp32, 1 layer, 1 KV head, 1 query head, d_head=64, n=512, vocab 1024, /E, B=128.
* ``mistral``  bf16, 32 layers, 32/8 heads, d_head=128, d_model=4096, n=16384, vocab 32000, /D.
* ``llama``    bf16, 32 layers, 32/8 heads, d_head=128, d_model=4096, n=131072, vocab 128256, /E,
               1 % of the keys carry an extra N(0, 3^2) outlier on channels {0, 32, 64, 96}.
* ``qwen``     bf16, 4 sequences, 48 layers, 40/8 heads, d_head=128, d_model=5120, n=32768,
               vocab 152064, /E, B=512.
* ``h2o``      fp16, batch 64, 48 layers, 56 heads, d_head=128, prompt 512 + 512 decode steps.

Distributions:
* ``normal`` keys (tiny): N(0,1); the key of token 0 has its component along the mean query
  direction replaced by 6x its magnitude, which makes token 0 an attention sink.
* ``zipf`` keys: k_i = g_i + s_i * mu with g ~ N(0,1), mu = 2 * u_hat (u_hat a random unit vector
  per layer and KV head) and s_i drawn from Zipf(1.1) clipped at 8 (P(s=j) proportional to
  j^-1.1 for j < 8, the remaining mass on 8). Queries are g + 2 * mu with the mu of their KV head.
* values N(0,1); logits N(0, 2^2); W_O ~ N(0, 1/d_model).
* the sampled lookahead token of each logits row is drawn from softmax(logits) with the
  Gumbel-max rule, argmax(z - log(-log U)).
"""
from __future__ import annotations

import dataclasses
import functools
import hashlib
import math

import torch

__all__ = ["LorekvConfig", "H2OConfig", "CcConfig", "LOREKV_CONFIGS", "H2O_CONFIGS",
           "CC_CONFIGS", "lorekv_inputs", "h2o_inputs", "cc_inputs", "unit_slice", "zipf_table"]


@dataclasses.dataclass(frozen=True)
class LorekvConfig:
    name: str
    dtype: str            # "f32" | "bf16"
    S: int                # independent sequences
    L: int                # layers
    Hq: int               # query heads
    Hkv: int              # KV heads
    d: int                # head dimension
    d_model: int
    n: int                # cached tokens per sequence
    vocab: int
    w: int = 32
    M: int = 4
    T: int = 8
    B: int = 128
    chunk: int = 4
    sink: int = 4
    beta: float = 1.0
    gamma: float = 1.3
    lambda_D: float = 0.0
    lambda_L: float = 1.0
    eps: float = 1e-6
    keys: str = "zipf"    # "normal" | "zipf"
    outlier_frac: float = 0.0
    window_causal: int = 1
    seed: int = 0

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    @property
    def units(self) -> int:
        return self.S * self.L * self.Hkv

    @property
    def queries_per_head(self) -> int:
        return self.w + self.M * self.T

    def replace(self, **kw) -> "LorekvConfig":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class H2OConfig:
    name: str
    dtype: str            # "f16"
    batch: int
    L: int
    H: int
    d: int
    prompt: int
    steps: int
    budget_frac: float = 0.2
    seed: int = 0

    @property
    def units(self) -> int:
        return self.batch * self.L * self.H

    @property
    def cap(self) -> int:
        return int(math.floor(self.budget_frac * (self.prompt + self.steps))) + 1

    def replace(self, **kw) -> "H2OConfig":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class CcConfig:
    """One counter-causal refresh: the last layer of ``batch`` sequences of ``n`` cached tokens,
    keeping ``J`` of them (J = floor(0.8 n): the refresh keeps J of J + h candidates with
    h = J/4)."""
    name: str
    dtype: str            # "f32" | "bf16"
    batch: int
    Hq: int
    Hkv: int
    d: int
    d_model: int
    n: int
    vocab: int
    sink: int
    J: int
    seed: int = 0

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    def replace(self, **kw) -> "CcConfig":
        return dataclasses.replace(self, **kw)


LOREKV_CONFIGS = {
    "tiny": LorekvConfig("tiny", "f32", S=1, L=1, Hq=1, Hkv=1, d=64, d_model=64, n=512,
                         vocab=1024, keys="normal"),
    "mistral": LorekvConfig("mistral", "bf16", S=1, L=32, Hq=32, Hkv=8, d=128, d_model=4096,
                            n=16384, vocab=32000, beta=1.0, gamma=1.0, lambda_D=0.3),
    "llama": LorekvConfig("llama", "bf16", S=1, L=32, Hq=32, Hkv=8, d=128, d_model=4096,
                          n=131072, vocab=128256, outlier_frac=0.01),
    "qwen": LorekvConfig("qwen", "bf16", S=4, L=48, Hq=40, Hkv=8, d=128, d_model=5120, n=32768,
                         vocab=152064, B=512),
}

H2O_CONFIGS = {
    "opt30b": H2OConfig("opt30b", "f16", batch=64, L=48, H=56, d=128, prompt=512, steps=512),
    "tiny": H2OConfig("tiny", "f16", batch=1, L=1, H=2, d=64, prompt=64, steps=64),
}

CC_CONFIGS = {
    # Qwen2.5-7B-shaped last layer: 28 query heads, 4 KV heads, d_head 128, d_model 3584
    "qwen7b_512": CcConfig("qwen7b_512", "bf16", batch=1, Hq=28, Hkv=4, d=128, d_model=3584,
                           n=512, vocab=152064, sink=4, J=409),
    "qwen7b_4096": CcConfig("qwen7b_4096", "bf16", batch=1, Hq=28, Hkv=4, d=128, d_model=3584,
                            n=4096, vocab=152064, sink=4, J=3276),
    "tiny": CcConfig("tiny", "f32", batch=2, Hq=4, Hkv=2, d=64, d_model=96, n=203, vocab=300,
                     sink=3, J=150),
}

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def _seed(*parts) -> int:
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


@functools.lru_cache(maxsize=None)
def zipf_table(a: float = 1.1, clip: int = 8, terms: int = 2_000_000) -> torch.Tensor:
    """Cumulative probabilities of Zipf(a) clipped at ``clip`` (mass of j >= clip put on clip)."""
    j = torch.arange(1, terms + 1, dtype=torch.float64)
    w = j.pow(-a)
    # zeta(a) = sum_{j<=terms} j^-a + tail, tail by the integral estimate (terms^(1-a))/(a-1)
    zeta = w.sum().item() + terms ** (1.0 - a) / (a - 1.0) - 0.5 * terms ** (-a)
    p = (torch.arange(1, clip, dtype=torch.float64).pow(-a) / zeta).tolist()
    p.append(1.0 - sum(p))
    return torch.tensor(p, dtype=torch.float64).cumsum(0)


def _zipf(shape, gen, device) -> torch.Tensor:
    cdf = zipf_table().to(device=device, dtype=torch.float32)
    u = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
    idx = torch.searchsorted(cdf, u.contiguous(), right=True).clamp_(max=cdf.numel() - 1)
    return (idx + 1).to(torch.float32)


def _unit_vectors(count: int, d: int, gen, device) -> torch.Tensor:
    u = torch.randn(count, d, generator=gen, device=device, dtype=torch.float64)
    return (u / u.norm(dim=1, keepdim=True)).to(torch.float32)


def lorekv_inputs(cfg: LorekvConfig, device="cpu") -> dict:
    """All inputs of one LORE-KV pass, laid out as the C-ABI expects.

    K, V    [S][L][Hkv][n][d]       cfg.dtype
    Q_W     [S][L][Hq][w][d]        cfg.dtype (window queries, the last w prompt positions)
    Q_look  [S][L][Hq][M*T][d]      cfg.dtype (row m*T+t: trajectory m, lookahead token t)
    W_O     [L][d_model][Hq*d]      cfg.dtype (o_proj weight: out_features x in_features)
    logits  [S][M*T][vocab]         fp32
    sampled [S][M*T]                int32
    """
    dt = _TORCH_DTYPE[cfg.dtype]
    dev = torch.device(device)
    S, L, Hq, Hkv, d, n, g = cfg.S, cfg.L, cfg.Hq, cfg.Hkv, cfg.d, cfg.n, cfg.g
    MT = cfg.M * cfg.T
    K = torch.empty(S, L, Hkv, n, d, dtype=dt, device=dev)
    V = torch.empty_like(K)
    QW = torch.empty(S, L, Hq, cfg.w, d, dtype=dt, device=dev)
    QL = torch.empty(S, L, Hq, MT, d, dtype=dt, device=dev)
    for s in range(S):
        for l in range(L):
            gen = _gen(dev, cfg.seed, cfg.name, "layer", s, l)
            gk = torch.randn(Hkv, n, d, generator=gen, device=dev, dtype=torch.float32)
            gv = torch.randn(Hkv, n, d, generator=gen, device=dev, dtype=torch.float32)
            gqw = torch.randn(Hq, cfg.w, d, generator=gen, device=dev, dtype=torch.float32)
            gql = torch.randn(Hq, MT, d, generator=gen, device=dev, dtype=torch.float32)
            if cfg.keys == "zipf":
                # the direction is shared by every sequence: it is a property of the layer/head
                u = _unit_vectors(Hkv, d, _gen(dev, cfg.seed, cfg.name, "mu", l), dev)
                mu = 2.0 * u                                    # [Hkv][d]
                sz = _zipf((Hkv, n), gen, dev)                  # [Hkv][n]
                gk += sz[..., None] * mu[:, None, :]
                if cfg.outlier_frac > 0:
                    hit = torch.rand(Hkv, n, generator=gen, device=dev) < cfg.outlier_frac
                    extra = 3.0 * torch.randn(Hkv, n, 4, generator=gen, device=dev)
                    ch = torch.tensor([0, 32, 64, 96], device=dev)
                    gk[:, :, ch] += extra * hit[..., None]
                muq = mu.repeat_interleave(g, dim=0)            # query head h -> KV head h // g
                gqw += 2.0 * muq[:, None, :]
                gql += 2.0 * muq[:, None, :]
            else:
                # sink: token 0's component along the mean query direction becomes 6x its size
                qall = torch.cat([gqw, gql], dim=1).reshape(-1, d).double()
                uq = qall.mean(0)
                uq = uq / uq.norm()
                for kh in range(Hkv):
                    k0 = gk[kh, 0].double()
                    c = torch.dot(k0, uq)
                    gk[kh, 0] = (k0 - c * uq + 6.0 * c.abs() * uq).float()
            K[s, l] = gk.to(dt)
            V[s, l] = gv.to(dt)
            QW[s, l] = gqw.to(dt)
            QL[s, l] = gql.to(dt)
            del gk, gv, gqw, gql
    gw = _gen(dev, cfg.seed, cfg.name, "W_O")
    W_O = torch.empty(L, cfg.d_model, Hq * d, dtype=dt, device=dev)
    for l in range(L):
        W_O[l] = (torch.randn(cfg.d_model, Hq * d, generator=gw, device=dev)
                  / math.sqrt(cfg.d_model)).to(dt)
    logits = torch.empty(S, MT, cfg.vocab, dtype=torch.float32, device=dev)
    sampled = torch.empty(S, MT, dtype=torch.int32, device=dev)
    for s in range(S):
        gl = _gen(dev, cfg.seed, cfg.name, "logits", s)
        z = 2.0 * torch.randn(MT, cfg.vocab, generator=gl, device=dev, dtype=torch.float32)
        u = torch.rand(MT, cfg.vocab, generator=gl, device=dev, dtype=torch.float64)
        u = u.clamp_(min=1e-300)
        gumbel = -torch.log(-torch.log(u))
        sampled[s] = torch.argmax(z.double() + gumbel, dim=1).to(torch.int32)
        logits[s] = z
    return {"K": K, "V": V, "Q_W": QW, "Q_look": QL, "W_O": W_O, "logits": logits,
            "sampled": sampled}


def unit_slice(cfg: LorekvConfig, inputs: dict, s: int, l: int, kh: int) -> dict:
    """The tensors one unit (sequence s, layer l, KV head kh) reads, as float64 CPU tensors."""
    g = cfg.g
    hs = slice(kh * g, kh * g + g)
    f = lambda t: t.detach().to("cpu").to(torch.float64)
    return {
        "K": f(inputs["K"][s, l, kh]), "V": f(inputs["V"][s, l, kh]),
        "Q_W": f(inputs["Q_W"][s, l, hs]), "Q_look": f(inputs["Q_look"][s, l, hs]),
        "W_O": f(inputs["W_O"][l]),
    }


def h2o_inputs(cfg: H2OConfig, device="cpu", steps=None) -> dict:
    """Prompt K/V/Q [B][L][H][P][d] and per-step decode q/k/v [steps][B][L][H][d], fp16.

    Keys (prompt and decode) are Zipf-biased as in the LORE-KV generator; prompt queries are
    g + 2*mu; decode queries are N(0,1).
    """
    dt = _TORCH_DTYPE[cfg.dtype]
    dev = torch.device(device)
    Bt, L, H, d, P = cfg.batch, cfg.L, cfg.H, cfg.d, cfg.prompt
    steps = cfg.steps if steps is None else steps
    Kp = torch.empty(Bt, L, H, P, d, dtype=dt, device=dev)
    Vp = torch.empty_like(Kp)
    Qp = torch.empty_like(Kp)
    mus = []
    for l in range(L):
        mu = 2.0 * _unit_vectors(H, d, _gen(dev, cfg.seed, cfg.name, "mu", l), dev)
        mus.append(mu)
        for b in range(Bt):
            gen = _gen(dev, cfg.seed, cfg.name, "prompt", b, l)
            gk = torch.randn(H, P, d, generator=gen, device=dev)
            gk += _zipf((H, P), gen, dev)[..., None] * mu[:, None, :]
            Kp[b, l] = gk.to(dt)
            Vp[b, l] = torch.randn(H, P, d, generator=gen, device=dev).to(dt)
            Qp[b, l] = (torch.randn(H, P, d, generator=gen, device=dev)
                        + 2.0 * mu[:, None, :]).to(dt)
    mu_all = torch.stack(mus)                                # [L][H][d]
    q = torch.empty(steps, Bt, L, H, d, dtype=dt, device=dev)
    k = torch.empty_like(q)
    v = torch.empty_like(q)
    for t in range(steps):
        gen = _gen(dev, cfg.seed, cfg.name, "step", t)
        q[t] = torch.randn(Bt, L, H, d, generator=gen, device=dev).to(dt)
        gk = torch.randn(Bt, L, H, d, generator=gen, device=dev)
        gk += _zipf((Bt, L, H), gen, dev)[..., None] * mu_all[None]
        k[t] = gk.to(dt)
        v[t] = torch.randn(Bt, L, H, d, generator=gen, device=dev).to(dt)
    return {"K": Kp, "V": Vp, "Q": Qp, "q": q, "k": k, "v": v}


def cc_inputs(cfg: CcConfig, device="cpu") -> dict:
    """All inputs of one counter-causal refresh, laid out as the C-ABI expects.

    K, V     [batch][Hkv][n][d]     cfg.dtype (Zipf-biased keys along a per-KV-head direction mu)
    Q_fresh  [batch][Hq][n][d]      cfg.dtype (g + 2 mu of the query head's KV head)
    H_last   [batch][n][d_model]    cfg.dtype, N(0, 1)
    W_O      [d_model][Hq*d]        cfg.dtype, N(0, 1/d_model)
    W_U      [vocab][d_model]       cfg.dtype, N(0, 1/d_model)
    tokens   [batch][n]             int32, uniform over the vocabulary
    """
    dt = _TORCH_DTYPE[cfg.dtype]
    dev = torch.device(device)
    B, Hq, Hkv, d, n, dm = cfg.batch, cfg.Hq, cfg.Hkv, cfg.d, cfg.n, cfg.d_model
    mu = 2.0 * _unit_vectors(Hkv, d, _gen(dev, cfg.seed, cfg.name, "mu"), dev)
    K = torch.empty(B, Hkv, n, d, dtype=dt, device=dev)
    V = torch.empty_like(K)
    Q = torch.empty(B, Hq, n, d, dtype=dt, device=dev)
    H = torch.empty(B, n, dm, dtype=dt, device=dev)
    X = torch.empty(B, n, dtype=torch.int32, device=dev)
    for b in range(B):
        gen = _gen(dev, cfg.seed, cfg.name, "seq", b)
        gk = torch.randn(Hkv, n, d, generator=gen, device=dev)
        gk += _zipf((Hkv, n), gen, dev)[..., None] * mu[:, None, :]
        K[b] = gk.to(dt)
        V[b] = torch.randn(Hkv, n, d, generator=gen, device=dev).to(dt)
        Q[b] = (torch.randn(Hq, n, d, generator=gen, device=dev)
                + 2.0 * mu.repeat_interleave(cfg.g, dim=0)[:, None, :]).to(dt)
        H[b] = torch.randn(n, dm, generator=gen, device=dev).to(dt)
        X[b] = torch.randint(0, cfg.vocab, (n,), generator=gen, device=dev, dtype=torch.int32)
    gw = _gen(dev, cfg.seed, cfg.name, "weights")
    W_O = (torch.randn(dm, Hq * d, generator=gw, device=dev) / math.sqrt(dm)).to(dt)
    W_U = torch.empty(cfg.vocab, dm, dtype=dt, device=dev)
    for r0 in range(0, cfg.vocab, 16384):   # bounded float32 temporaries
        r1 = min(cfg.vocab, r0 + 16384)
        W_U[r0:r1] = (torch.randn(r1 - r0, dm, generator=gw, device=dev) / math.sqrt(dm)).to(dt)
    return {"K": K, "V": V, "Q_fresh": Q, "H_last": H, "W_O": W_O, "W_U": W_U, "tokens": X}
