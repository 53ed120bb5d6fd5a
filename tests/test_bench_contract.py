"""The benchmark's command-line contract, checked on the CPU: the reference arm (the CPU
oracle) prints one JSON line with the keys and units of the native arm, only rank 0
prints under a multi-rank launch, and the native arm fails loudly (non-zero exit, no
line) when there is no GPU instead of falling back to the CPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra=None, timeout=300):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    sys.path.insert(0, ROOT)
    import bench
    # the small workload keeps this CPU check short; the default is the LLaDA-8B-shaped layer
    r = _run(["--impl", "reference", "--steps", "1", "--warmup", "3", "--reference-workload", "tiny-fp32"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] == pytest.approx(1e3 / d["value"], rel=1e-9)
    assert "workload" in d["config"] and "tiny-fp32" in d["config"]["workload"]
    assert d["config"]["parallelism"] == "replicas x1"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] >= 1 and cb["sample"] and cb["cpu_model"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    r = _run(["--impl", "reference", "--steps", "1", "--warmup", "3", "--reference-workload", "tiny-fp32"],
             {"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_native_arm_fails_loudly_without_a_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = _run(["--steps", "1", "--warmup", "3", "--no-stack", "--no-configs", "--no-cpu-baseline"])
    assert r.returncode != 0
    assert not any(l.strip().startswith("{") for l in r.stdout.splitlines())


def test_kernel_work_model_follows_the_launches():
    """The bench's per-kernel work model (the roofline's algorithmic bytes) names the
    kernels each configuration launches: at the LLaDA-8B-shaped layer the selection
    kernel computes the drift from the proxy projection's K-slice partials (no cosine
    kernel); at 16 x 8192 tokens the projection's epilogue does (no split, no cosine
    kernel, a separate gather beyond N = 4096); the fp32 layer's selection kernel takes the
    drift from the fp32 proxies."""
    sys.path.insert(0, ROOT)
    import dataclasses
    import bench
    from sparse_kv_cache_rank_gb300 import binding, synth
    if not os.path.exists(binding.LIB_PATH):
        pytest.skip("libdllm.so not built")
    llada = bench.layer_kernel_work(synth.LLADA_LAYER, 164)
    assert "cosine" not in llada and "gather" not in llada
    B, N, r = 1, 1024, 128
    assert llada["select"][0] == 8 * B * N + 4 * B + 2 * 164 * 4096 * 2 + 8 * 164 * r + 8 * B * N * r + 4 * B * N
    wide = bench.layer_kernel_work(dataclasses.replace(synth.LLADA_LAYER, B=16, N=8192), 164)
    assert "cosine" not in wide and "gather" in wide
    tiny = bench.layer_kernel_work(synth.TINY, 96)
    assert "cosine" not in tiny and "rmsnorm2" in tiny
    for w in (llada, wide, tiny):
        assert all(v[0] > 0 for v in w.values())


@pytest.mark.parametrize("n", [1, 5, 16, 17, 20, 37, 100, 1000])
def test_e2e_batches_cover_every_step(n):
    """The end-to-end leg's batches cover the steps exactly once, never exceed the cap,
    and start and end with single steps once there are enough of them (the first step
    waits for one upload, the last read-back is one step's)."""
    sys.path.insert(0, ROOT)
    import bench
    b = bench.e2e_batches(n, 4)
    assert sum(b) == n and all(1 <= x <= 4 for x in b)
    assert b[0] == 1 and b[-1] == 1
    if n > 16:
        assert max(b) == 4 and len(b) < n
