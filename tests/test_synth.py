"""The seeded input module that the oracle and the CUDA path share (it holds none of the
method's arithmetic): its bf16 rounding against PyTorch's conversion, and the input
recipe (drift model, block layout, weights) against its stated shapes and statistics."""
import dataclasses

import numpy as np
import pytest

from sparse_kv_cache_rank_gb300 import synth


def test_round_bf16_matches_torch_round_to_nearest_even():
    torch = pytest.importorskip("torch")
    g = synth.rng(5)
    x = (g.standard_normal(200000) * np.exp2(g.integers(-140, 120, 200000))).astype(np.float32)
    # exact halfway cases (the 16 dropped bits are 0x8000), both parities of the kept bit
    u = g.integers(0, 2 ** 31, 4096, dtype=np.uint64).astype(np.uint32) & np.uint32(0x7EFF0000)
    halves = (u | np.uint32(0x8000)).view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 3.4e38, -3.4e38, 1.0, -1.0],
                       np.float32)
    x = np.concatenate([x, halves, -halves, special])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = synth.round_bf16(x)
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))
    nan = np.array([np.nan, -np.nan], np.float32)
    assert np.isnan(synth.round_bf16(nan)).all()


def test_drift_model_recipe():
    sh = dataclasses.replace(synth.LLADA_LAYER, B=2, N=1000, d=256, dtype="f32")
    Hp, Hc, hot = synth.hidden_pair(sh, 3)
    assert Hp.shape == Hc.shape == (2, 1000, 256) and hot.shape == (2, 100)
    for b in range(2):
        assert np.all(np.diff(hot[b]) > 0) and hot[b].min() >= 0 and hot[b].max() < 1000
        moved = np.zeros(1000, bool)
        moved[hot[b]] = True
        delta = Hc[b] - Hp[b]
        assert delta[~moved].std() == pytest.approx(0.05, rel=0.02)
        assert delta[moved].std() == pytest.approx(np.hypot(0.05, 0.5), rel=0.02)
    assert Hp.std() == pytest.approx(1.0, rel=0.02)
    Hp2, Hc2, hot2 = synth.hidden_pair(sh, 3)
    assert np.array_equal(Hc, Hc2) and np.array_equal(hot, hot2)        # seeded
    assert not np.array_equal(synth.hidden_pair(sh, 4)[1], Hc)


def test_block_layout_recipe():
    sh = synth.TINY
    masked, recent = synth.block_layout(sh, 9, block_index=1)
    start = sh.prompt + sh.block
    assert masked.shape == (1, sh.block - sh.k_recent) and recent.shape == (1, sh.k_recent)
    both = np.concatenate([masked[0], recent[0]])
    assert sorted(both.tolist()) == list(range(start, start + sh.block))
    assert np.all(np.diff(masked[0]) > 0) and np.all(np.diff(recent[0]) > 0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_layer_weights_recipe(dtype):
    sh = dataclasses.replace(synth.TINY, dtype=dtype)
    w = synth.layer_weights(sh, 11)
    shapes = {"w_q": (sh.d_q, sh.d), "w_k": (sh.d_kv, sh.d), "w_v": (sh.d_kv, sh.d), "w_o": (sh.d, sh.d_q),
              "w_g": (sh.F, sh.d), "w_u": (sh.F, sh.d), "w_d": (sh.d, sh.F), "gamma1": (sh.d,),
              "gamma2": (sh.d,)}
    for k, s in shapes.items():
        assert w[k].shape == s and w[k].dtype == np.float32
    assert np.all(w["gamma1"] == 1) and np.all(w["gamma2"] == 1)
    assert w["w_g"].std() == pytest.approx(0.02, rel=0.02)
    if dtype == "bf16":
        for k in shapes:
            assert np.array_equal(synth.round_bf16(w[k]), w[k])           # bf16-representable
