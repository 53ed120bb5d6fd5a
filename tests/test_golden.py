"""Hand-worked examples under tests/golden/, each derived in closed form from the definition
on the page it cites (the pages print no numeric example of their own).  The oracle must
reproduce every one of them (CPU), and so must the CUDA path through the C ABI (GPU):
a check of both sides against values that come from neither."""
import json
import os

import numpy as np
import pytest

from oracle import cluster as cl
from oracle import kl as okl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _pad(rows, width):
    out = np.zeros((len(rows), width), np.float32)
    for i, row in enumerate(rows):
        out[i, :len(row)] = row
    return out


def _drift_case():
    g = load("drift_cosine.json")
    d, r = g["d"], g["r"]
    H = _pad(g["h2"], d)[None]                         # [1, N, d]
    P = np.zeros((d, r), np.float32)
    P[0, 0] = P[1, 1] = 1.0
    cached = _pad(g["cached2"], r)[None]               # [1, N, r]
    return g, H, P, cached


def _entropy_case():
    g = load("entropy_commit.json")
    logits = np.asarray(g["logits"], np.float32)
    valid = np.asarray(g["valid"], np.uint8)
    return g, logits, valid


def _check_entropy(g, valid, tok, conf, ent, E, full):
    live = valid.astype(bool)
    np.testing.assert_allclose(np.asarray(conf)[live], np.asarray(g["conf"], dtype=object)[live].astype(float),
                               rtol=1e-6)
    np.testing.assert_allclose(np.asarray(ent)[live], np.asarray(g["entropy"], dtype=object)[live].astype(float),
                               rtol=1e-6)
    np.testing.assert_array_equal(tok, g["token"])
    np.testing.assert_allclose(E, g["max_entropy"], rtol=1e-6)
    np.testing.assert_array_equal(full, g["full_next"])


def _kl_case(which="main"):
    g = load("kl_drift_three_rows.json")
    r = g["r"]
    if which == "main":
        return g, _pad(g["cur4"], r)[None], _pad(g["cached4"], r)[None], np.asarray(g["drift"])
    s = g["same"]
    cur = _pad(s["cur4"], r)[None]
    return g, cur, cur.copy(), np.asarray(s["drift"])


# --------------------------------------------------------------------------- oracle (CPU)
def test_golden_drift_cosine_oracle(orc):
    g, H, P, cached = _drift_case()
    _, drift = orc.proxy_score(H, P, cached)
    np.testing.assert_allclose(drift[0], g["drift"], atol=1e-6)


def test_golden_select_oracle(orc):
    g = load("select_forced_topk.json")
    for c in g["cases"]:
        idx, cnt = orc.select_topk(np.asarray([c["drift"]], np.float32), np.asarray([c["forced"]], np.int32),
                                   c["k"], g["min_drift"])
        assert int(cnt[0]) == c["count"], c["why"]
        np.testing.assert_array_equal(idx[0, :c["count"]], c["idx"])
        assert np.all(idx[0, c["count"]:] == -1)


def test_golden_budget_oracle(orc):
    g = load("budget_schedule.json")
    for l, want, _ in g["rho"]:
        assert orc.rho(l) == pytest.approx(want, rel=1e-14)
    for rho, N, want, _ in g["budget"]:
        assert orc.budget(rho, N) == want


def test_golden_budget_library_host_logic():
    """The library's budget schedule is host code (no launch): checked here without a GPU."""
    import shutil
    import sparse_kv_cache_rank_gb300 as pkg
    from sparse_kv_cache_rank_gb300 import binding as B
    if not os.path.exists(B.LIB_PATH):
        if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("nvcc not available to build libdllm.so")
        pkg.build()
    g = load("budget_schedule.json")
    for l, want, _ in g["rho"]:
        assert B.dllm_layer_rho(l) == pytest.approx(want, rel=1e-14)
    for rho, N, want, _ in g["budget"]:
        assert B.dllm_layer_budget(rho, N) == want


def test_golden_entropy_commit_oracle(orc):
    g, logits, valid = _entropy_case()
    tok, conf, ent, E, full = orc.commit_entropy(logits, valid, g["conf_thresh"], g["tau"])
    _check_entropy(g, valid, tok, conf, ent, E, full)


@pytest.mark.parametrize("which", ["main", "same"])
def test_golden_kl_oracle(which):
    _, cur, cached, want = _kl_case(which)
    np.testing.assert_allclose(okl.kl_drift(cur, cached)[0], want, atol=1e-12)


def test_golden_nvfp4_oracle():
    g = load("nvfp4_block.json")
    block = np.asarray([g["block"]], np.float32)
    codes, sc = cl.nvfp4_quantize(block, g["g"])
    assert int(sc[0, 0]) == g["scale_code"]
    np.testing.assert_array_equal(codes[0], g["codes"])
    np.testing.assert_array_equal(cl.nvfp4_dequantize(codes, sc, g["g"])[0], block[0])


# --------------------------------------------------------------------------- CUDA path (GPU)
@pytest.fixture(scope="module")
def Bg():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_cache_rank_gb300 import binding
    binding.lib()
    binding.check_status(reset=True)
    return binding


def _dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.to(dtype) if dtype is not None else t).cuda()


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_golden_drift_cosine_gpu(Bg, dtype):
    import torch
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g, H, P, cached = _drift_case()
    _, drift = Bg.dllm_proxy_score(_dev(H, dt), _dev(P.T.copy(), dt), _dev(cached))
    np.testing.assert_allclose(drift.cpu().numpy()[0], g["drift"], atol=1e-6)


@pytest.mark.gpu
def test_golden_select_gpu(Bg):
    g = load("select_forced_topk.json")
    for c in g["cases"]:
        idx, cnt = Bg.dllm_select_topk(_dev(np.asarray([c["drift"]], np.float32)),
                                       _dev(np.asarray([c["forced"]], np.int32)), c["k"], g["min_drift"])
        assert int(cnt.cpu()[0]) == c["count"], c["why"]
        got = idx.cpu().numpy()[0]
        np.testing.assert_array_equal(got[:c["count"]], c["idx"])
        assert np.all(got[c["count"]:] == -1)


@pytest.mark.gpu
def test_golden_entropy_commit_gpu(Bg):
    g, logits, valid = _entropy_case()
    out = Bg.dllm_commit_entropy(_dev(logits), _dev(valid), g["conf_thresh"], g["tau"])
    _check_entropy(g, valid, *(t.cpu().numpy() for t in out))


@pytest.mark.gpu
@pytest.mark.parametrize("which", ["main", "same"])
def test_golden_kl_gpu(Bg, which):
    _, cur, cached, want = _kl_case(which)
    D = Bg.dllm_kl_drift(_dev(cur), _dev(cached))
    np.testing.assert_allclose(D.cpu().numpy()[0], want, atol=1e-6)


@pytest.mark.gpu
def test_golden_nvfp4_gpu(Bg):
    g = load("nvfp4_block.json")
    block = np.asarray([g["block"]], np.float32)
    codes, sc = Bg.dllm_nvfp4_quantize(_dev(block), g["g"])
    packed = codes.cpu().numpy()[0]
    got = np.empty(16, np.uint8)
    got[0::2], got[1::2] = packed & 15, packed >> 4    # low nibble = even element
    assert int(sc.cpu()[0, 0]) == g["scale_code"]
    np.testing.assert_array_equal(got, g["codes"])
    back = Bg.dllm_nvfp4_dequantize(codes, sc, g["g"]).cpu().numpy()[0]
    np.testing.assert_array_equal(back, block[0])
