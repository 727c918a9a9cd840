"""C-ABI checks that need no GPU: the library builds, loads and exports every function that
include/kvevict.h declares; argument validation and the host-side fault hook work before any
CUDA call is made."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def api():
    from kv_cache_eviction_02_gb300 import _build, api as a
    _build.build()
    a.lib()
    return a


def _declared_functions():
    with open(os.path.join(ROOT, "include", "kvevict.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(", src,
                       flags=re.M)
    return sorted(set(names))


def test_header_declares_the_exported_api(api):
    names = _declared_functions()
    assert "lorekv_score" in names and "h2o_decode_step" in names
    assert set(names) == set(api.EXPORTED)


def test_library_exports_every_declared_symbol(api):
    out = subprocess.run(["nm", "-D", "--defined-only", api.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for name in _declared_functions():
        assert name in exported, name
        assert getattr(api.lib(), name) is not None


def _pb(api, **kw):
    base = dict(n_seq=1, n_layers=2, n_q_heads=8, n_kv_heads=2, d_head=128, d_model=256,
                n_tokens=1000, vocab=500, dtype=api.KVE_BF16, budget_B=128)
    base.update(kw)
    return api.LorekvProblem(**base)


def test_workspace_size_and_capacity(api):
    pb = _pb(api)
    ws = api.lorekv_workspace_size(pb)
    assert ws > 0 and ws % 256 == 0
    assert api.lorekv_kept_capacity(pb) == 4 + 128 + 32
    assert api.lorekv_kept_capacity(_pb(api, n_tokens=36 + 128)) == 36 + 128   # all kept
    # more tokens -> more workspace
    assert api.lorekv_workspace_size(_pb(api, n_tokens=2000)) > ws


@pytest.mark.parametrize("bad", [
    dict(n_tokens=1001),            # (n - sink - w) not a multiple of chunk
    dict(budget_B=130),             # B not a multiple of chunk
    dict(n_q_heads=7),              # not a multiple of n_kv_heads
    dict(d_head=96),                # unsupported head size
    dict(n_tokens=20),              # fewer tokens than sink + w
    dict(M=40),                     # too many trajectories
    dict(n_seq=16385),              # 65540 units: beyond the launch grids' y extent
    dict(n_tokens=1 << 29),         # 4 units x 2^29 K/V rows: beyond 32-bit row indices
])
def test_invalid_shapes_are_rejected_without_a_gpu(api, bad):
    pb = _pb(api, **bad)
    assert api.lorekv_workspace_size(pb) == 0
    with pytest.raises(api.KveError) as e:
        api.lorekv_kept_capacity(pb)
    assert e.value.status == api.KVE_EINVAL


def test_score_rejects_bad_arguments_before_touching_the_gpu(api):
    L = api.lib()
    pb = _pb(api)
    sh, pr = pb.shape(), pb.params()
    fake = ctypes.c_void_p(256)
    # missing workspace
    st = L.lorekv_score(ctypes.byref(sh), ctypes.byref(pr), fake, fake, fake, fake, fake, fake,
                        fake, fake, fake, fake, None, 0, None)
    assert st == api.KVE_EWORKSPACE
    assert "workspace" in L.kve_last_error().decode()
    # wrong dtype
    sh.dtype = api.KVE_F16
    st = L.lorekv_score(ctypes.byref(sh), ctypes.byref(pr), fake, fake, fake, fake, fake, fake,
                        fake, fake, fake, fake, fake, 1 << 40, None)
    assert st == api.KVE_EDTYPE
    # null tensors
    sh.dtype = api.KVE_BF16
    st = L.lorekv_score(ctypes.byref(sh), ctypes.byref(pr), None, fake, fake, fake, fake, fake,
                        fake, fake, fake, fake, fake, 1 << 40, None)
    assert st == api.KVE_EINVAL


def test_fidelity_rejects_bad_arguments_before_touching_the_gpu(api):
    L = api.lib()
    assert L.lorekv_output_fidelity(None, None, 4, 128, None, None, None) == api.KVE_EINVAL
    fake = ctypes.c_void_p(256)  # never dereferenced: the checks run first
    assert L.lorekv_output_fidelity(fake, fake, 0, 128, fake, None, None) == api.KVE_EINVAL
    assert L.lorekv_output_fidelity(fake, fake, 4, 0, fake, None, None) == api.KVE_EINVAL


def _cc(api, **kw):
    base = dict(n_seq=2, n_q_heads=28, n_kv_heads=4, d_head=128, d_model=3584, n_tokens=512,
                vocab=1000, dtype=api.KVE_BF16, sink=4, keep_J=410)
    base.update(kw)
    return api.CcProblem(**base)


def test_cc_workspace_size_covers_the_attention_outputs(api):
    ws = api.cc_workspace_size(_cc(api))
    assert ws >= 2 * 512 * 28 * 128 * 4 and ws % 256 == 0
    assert api.cc_workspace_size(_cc(api, n_tokens=1024)) > ws


@pytest.mark.parametrize("bad", [
    dict(n_q_heads=27),            # not a multiple of n_kv_heads
    dict(d_head=96),               # unsupported head size
    dict(keep_J=0), dict(keep_J=513),
    dict(sink=-1), dict(sink=513),
    dict(dtype=2),                 # f16 not supported here
    dict(vocab=0),
    dict(n_seq=4096, n_tokens=1 << 16, keep_J=512),  # query rows beyond 32-bit indices
])
def test_cc_invalid_shapes_are_rejected_without_a_gpu(api, bad):
    pb = _cc(api, **bad)
    assert api.cc_workspace_size(pb) == 0
    L, sh, fake = api.lib(), pb.shape(), ctypes.c_void_p(256)
    st = L.cc_surprise(ctypes.byref(sh), fake, fake, fake, fake, fake, fake, fake, fake, fake,
                       1 << 40, None)
    assert st in (api.KVE_EINVAL, api.KVE_EDTYPE)
    st = L.cc_select_compact(ctypes.byref(sh), fake, fake, fake, fake, fake, fake, fake, fake, None)
    assert st in (api.KVE_EINVAL, api.KVE_EDTYPE)


def test_cc_rejects_bad_arguments_before_touching_the_gpu(api):
    L, sh, fake = api.lib(), _cc(api).shape(), ctypes.c_void_p(256)
    st = L.cc_surprise(ctypes.byref(sh), fake, fake, fake, fake, fake, fake, fake, fake, None, 0,
                       None)
    assert st == api.KVE_EWORKSPACE and "workspace" in L.kve_last_error().decode()
    st = L.cc_surprise(ctypes.byref(sh), fake, None, fake, fake, fake, fake, fake, fake, fake,
                       1 << 40, None)
    assert st == api.KVE_EINVAL
    st = L.cc_select_compact(ctypes.byref(sh), fake, fake, fake, None, fake, fake, fake, fake, None)
    assert st == api.KVE_EINVAL


def test_h2o_create_validates_arguments(api):
    L = api.lib()
    h = ctypes.c_void_p()
    assert L.h2o_state_create(ctypes.byref(h), 1, 1, 2, 96, 100, 0.2, api.KVE_F16) == api.KVE_EINVAL
    assert L.h2o_state_create(ctypes.byref(h), 1, 1, 2, 64, 100, 1.5, api.KVE_F16) == api.KVE_EINVAL
    assert L.h2o_state_create(ctypes.byref(h), 1, 1, 2, 64, 100, 0.2, api.KVE_F32) == api.KVE_EDTYPE
    assert L.h2o_state_create(ctypes.byref(h), 1, 1, 2, 64, 100000, 0.2, api.KVE_F16) == api.KVE_EINVAL
    # 2^21 units x 1024 positions: prompt rows beyond 32-bit indices (checked before allocating)
    assert L.h2o_state_create(ctypes.byref(h), 1 << 11, 32, 32, 64, 1024, 0.2,
                              api.KVE_F16) == api.KVE_EINVAL
    assert not h.value
    assert L.h2o_decode_step(None, None, None, None, None, None) == api.KVE_EINVAL


def test_injected_failure_is_reported_then_cleared(api):
    pb = _pb(api)
    api.kve_inject_failure(api.KVE_ECUDA, 2)
    for _ in range(2):
        with pytest.raises(api.KveError) as e:
            api.lorekv_prepare_wo(pb, 1, 1, 1, 0)
        assert e.value.status == api.KVE_ECUDA
        assert "injected" in str(e.value)
    # the hook is used up: the next call validates normally (null pointers -> EINVAL)
    with pytest.raises(api.KveError) as e:
        api.lorekv_prepare_wo(pb, None, None, None, 0)
    assert e.value.status == api.KVE_EINVAL
    api.kve_inject_failure(0, 0)


def test_cc_cache_create_validates_arguments(api):
    L = api.lib()
    h = ctypes.c_void_p()
    for bad in (dict(keep_J=512, n_tokens=512),       # no room for a chunk
                dict(keep_J=3, sink=4),                 # sinks plus the last token do not fit
                dict(d_head=96), dict(dtype=2)):
        sh = _cc(api, **bad).shape()
        assert L.cc_cache_create(ctypes.byref(h), ctypes.byref(sh)) in (api.KVE_EINVAL,
                                                                         api.KVE_EDTYPE)
        assert not h.value
    sh = _cc(api).shape()
    assert L.cc_cache_create(None, ctypes.byref(sh)) == api.KVE_EINVAL
    fake = ctypes.c_void_p(256)
    assert L.cc_cache_append(None, fake, fake, fake, fake, fake, 1, None) == api.KVE_EINVAL
    assert L.cc_cache_refresh(None, fake, fake, None) == api.KVE_EINVAL
    assert L.cc_cache_length(None) == -api.KVE_EINVAL


def test_binding_checks_tensors_against_the_shape(api):
    """A tensor of another element type, or shorter than the declared shape needs, is refused
    in the binding before its address reaches the library."""
    import torch
    pb = _pb(api)  # bf16, 4 units x 1000 tokens x d 128
    kv = pb.units * pb.n_tokens * pb.d_head
    K = torch.zeros(kv, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="dtype"):
        api.lorekv_score(pb, K.float(), None, None, None, None, None, None, None, None, None, None)
    with pytest.raises(ValueError, match="elements"):
        api.lorekv_score(pb, K[:-1], None, None, None, None, None, None, None, None, None, None)
    with pytest.raises(ValueError, match="elements"):
        api.lorekv_attention_stats(pb, None, None, None, None, torch.zeros(10), None,
                                   torch.zeros(1, dtype=torch.uint8))
    cap = api.lorekv_kept_capacity(pb)
    with pytest.raises(ValueError, match="kept_idx"):
        api.lorekv_select_compact(pb, None, None, None,
                                  torch.zeros(pb.units * cap - 1, dtype=torch.int32), None, None,
                                  None)
    # every size right: the binding goes on to the device check (CPU tensors are refused there)
    with pytest.raises(ValueError, match="CUDA"):
        api.lorekv_score(pb, K, K, None, None, None, None, None, None, None, None, None)
