"""lorekv_score_noalloc: the scoring pass for callers that cannot allocate device memory.

Such callers (code inside a memory budget owned by a framework or a serving runtime, or with no
device allocator at hand) get the same pass with its scratch in a fixed array inside the library.
This file is collected last so that a run stopping at the first failure has already run every
other test; it passes alone in a fresh process and after the others.
"""
import numpy as np
import pytest
import torch

from kv_cache_eviction_02_gb300 import api, synth
from parity import SCORE_RTOL, assert_scores_close

CFG = synth.LorekvConfig("noalloc_bf16", "bf16", S=1, L=2, Hq=8, Hkv=2, d=128, d_model=256,
                         n=1060, vocab=3000, beta=1.0, gamma=1.0, lambda_D=0.3)


def test_noalloc_rejects_shapes_beyond_its_fixed_scratch():
    """A shape whose workspace exceeds the fixed 64 MiB is refused before anything is launched."""
    big = api.LorekvProblem.from_config(synth.LOREKV_CONFIGS["llama"])
    assert api.lorekv_workspace_size(big) > 64 << 20
    with pytest.raises(api.KveError) as e:
        api.lorekv_score_noalloc(big, *([1] * 10), stream=0)
    assert e.value.status == api.KVE_EWORKSPACE
    assert "64 MiB" in str(e.value) or str(64 << 20) in str(e.value)


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    dev = torch.device("cuda:0")
    pb = api.LorekvProblem.from_config(CFG)
    assert api.lorekv_workspace_size(pb) <= 64 << 20
    runs = []
    for seed in (0, 1):   # different inputs on the two calls: stale scratch must not matter
        cfg = CFG.replace(seed=seed)
        g = {k: v.to(dev) for k, v in synth.lorekv_inputs(cfg, "cpu").items()}
        Lf = torch.empty(cfg.L, cfg.Hq, cfg.d, cfg.d, device=dev)
        G = torch.empty_like(Lf)
        api.lorekv_prepare_wo(pb, g["W_O"], Lf, G)
        runs.append((g, Lf, G))
    refs = []
    for g, Lf, G in runs:
        S = torch.empty(pb.units, pb.n_tokens, device=dev)
        om = torch.empty(pb.n_seq, pb.M, device=dev)
        ws = torch.empty(api.lorekv_workspace_size(pb), dtype=torch.uint8, device=dev)
        api.lorekv_score(pb, g["K"], g["V"], g["Q_W"], g["Q_look"], Lf, G, g["logits"],
                         g["sampled"], S, om, ws)
        refs.append((S.double().cpu().numpy(), om.double().cpu().numpy()))
    for (g, Lf, G), (S_ref, om_ref) in zip(runs, refs):
        S = torch.full((pb.units, pb.n_tokens), float("nan"), device=dev)
        om = torch.full((pb.n_seq, pb.M), float("nan"), device=dev)
        api.lorekv_score_noalloc(pb, g["K"], g["V"], g["Q_W"], g["Q_look"], Lf, G, g["logits"],
                                 g["sampled"], S, om)
        api.kve_check_device()
        S, om = S.double().cpu().numpy(), om.double().cpu().numpy()
        assert np.allclose(om, om_ref, rtol=1e-5, atol=0)
        for u in range(pb.units):
            assert_scores_close(S[u], S_ref[u], "bf16", f"unit {u}")
    assert SCORE_RTOL["bf16"] == 2e-3
