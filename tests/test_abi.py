"""C-ABI checks that need no GPU: the library builds and loads, exports every entry
point declared in include/dllm.h, its host-side budget logic agrees with the oracle,
and invalid arguments are rejected with error codes before any launch."""
import ctypes as C
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dllm.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dllm_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def dl():
    import sparse_kv_cache_rank_gb300 as pkg
    from sparse_kv_cache_rank_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("nvcc not available to build libdllm.so")
        pkg.build()
    return binding


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("dllm_proxy_score", "dllm_select_topk", "dllm_sparse_layer_refresh",
              "dllm_commit_entropy", "dllm_pack_layer", "dllm_check_status"):
        assert n in names


def test_library_exports_every_declared_symbol(dl):
    L = C.CDLL(dl.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(L, n)]
    assert not missing, missing
    assert set(_declared()) <= set(dl.exported_symbols()) | {"dllm_last_error", "dllm_version"}
    assert dl.lib().dllm_version() == 113


def test_budget_logic_matches_oracle(dl, orc):
    for l in range(32):
        assert dl.dllm_layer_rho(l) == pytest.approx(orc.rho(l), rel=1e-15)
        assert dl.dllm_layer_rho(l, sigma_left=3.0, sigma_right=9.0) == pytest.approx(
            orc.rho(l, sigma_left=3.0, sigma_right=9.0), rel=1e-15)
    for rho in (0.0, 1e-9, 0.05, 0.16, 0.25, 0.3, 0.5, 1.0, 1.5):
        for N in (1, 7, 256, 768, 1024, 2048, 8192):
            assert dl.dllm_layer_budget(rho, N) == orc.budget(rho, N)


def _err(dl):
    return dl.lib().dllm_last_error().decode()


def test_invalid_arguments_fail_before_launch(dl):
    L = dl.lib()
    p = C.c_void_p(256)   # never dereferenced: every case below fails validation first
    # null pointers / bad sizes
    assert L.dllm_proxy_score(None, p, p, p, p, 1, 8, 64, 32, 1, None, 0, None) == -1
    assert "null" in _err(dl)
    assert L.dllm_proxy_score(p, p, p, p, p, 1, 8, 64, 31, 1, None, 0, None) == -2       # r % 32
    assert L.dllm_proxy_score(p, p, p, p, p, 1, 8, 100, 32, 1, None, 0, None) == -2      # d % 64 (bf16)
    assert L.dllm_proxy_score(p, p, p, p, p, 0, 8, 64, 32, 1, None, 0, None) == -1
    assert L.dllm_proxy_score(C.c_void_p(258), p, p, p, p, 1, 8, 64, 32, 1, None, 0, None) == -1   # alignment
    assert L.dllm_proxy_score(p, p, p, p, p, 1 << 16, 1 << 16, 64, 32, 1, None, 0, None) == -1   # B*N > int
    assert L.dllm_select_topk(p, None, 0, -1, 0.0, p, p, 1, 8, None) == -1      # k < 0
    assert L.dllm_select_topk(p, None, 0, 4, 0.0, p, p, 1, 20000, None) == -1   # N too large
    assert L.dllm_select_topk(None, None, 0, 4, 0.0, p, p, 1, 8, None) == -1
    # commit: workspace too small, M too large
    assert L.dllm_commit_entropy(p, p, 1, 4, 16, 0.9, 2.0, p, p, p, p, p, p, 0, None) == -3
    assert L.dllm_commit_entropy(p, p, 1, 2000, 16, 0.9, 2.0, p, p, p, p, p, p, 1 << 20, None) == -1
    # B*M past the int range: rejected before any row count is formed
    big = 1 << 22
    assert L.dllm_commit_entropy(p, p, big, 1024, 16, 0.9, 2.0, p, p, p, p, p, p, 1 << 20, None) == -1
    assert L.dllm_commit_workspace_bytes(big, 1024, 16) == 0
    # allocation-free commit: more rows than its fixed array holds (also where B*M wraps an int)
    assert L.dllm_commit_entropy_noalloc(p, p, big, 1024, 16, 0.9, 2.0, p, p, p, p, p, None) == -2
    assert "allocation-free" in _err(dl)
    assert L.dllm_commit_entropy_noalloc(p, p, 17, 1024, 16, 0.9, 2.0, p, p, p, p, p, None) == -2
    # pack: unsupported head dim, misaligned destination
    desc = dl.dllm_layer()
    args = [p] * 9
    assert L.dllm_pack_layer(*args, 64, 1, 1, 32, 64, 1e-5, 1e4, 1, 1, p, 1 << 30, C.byref(desc), None) == -2
    assert L.dllm_pack_layer(*args, 64, 1, 1, 64, 64, 1e-5, 1e4, 1, 1, C.c_void_p(272), 1 << 30,
                             C.byref(desc), None) == -1
    assert L.dllm_pack_layer(*args, 64, 1, 1, 64, 64, 1e-5, 1e4, 1, 1, p, 16, C.byref(desc), None) == -3
    # refresh: layer checks, k_max > N, aliasing, workspace
    desc = dl.dllm_layer(p.value, p.value, p.value, p.value, p.value, p.value, p.value,
                         128, 1, 1, 128, 128, 1e-5, 1e4, 1, 1)
    ws_need = L.dllm_refresh_workspace_bytes(C.byref(desc), 1, 16, 4)
    assert ws_need > 0
    rf = L.dllm_sparse_layer_refresh
    assert rf(C.byref(desc), p, p, p, 17, p, p, C.c_void_p(512), None, None, 0, 1, 16, p, ws_need, None) == -1
    assert rf(C.byref(desc), p, p, p, 4, p, p, p, None, None, 0, 1, 16, p, ws_need, None) == -1
    assert "alias" in _err(dl)
    assert rf(C.byref(desc), p, p, p, 4, p, p, C.c_void_p(512), None, None, 0, 1, 16, p, 8, None) == -3
    assert rf(C.byref(desc), p, p, p, 4, p, p, C.c_void_p(512), p, None, 0, 1, 16, p, ws_need, None) == -1
    bad = dl.dllm_layer(p.value, p.value, p.value, p.value, p.value, p.value, p.value,
                        128, 1, 1, 96, 128, 1e-5, 1e4, 1, 1)
    assert rf(C.byref(bad), p, p, p, 4, p, p, C.c_void_p(512), None, None, 0, 1, 16, p, ws_need, None) == -2
    # read-back of several caches: n outside [1, 4], a null cache, a misaligned one, row sizes
    srcs = (C.c_void_p * 3)(256, 512, 768)
    dsts = (C.c_void_p * 3)(1024, 1280, 1536)
    rb = (C.c_int * 3)(8192, 8192, 8192)
    gn = L.dllm_gather_rows_n
    assert gn(0, srcs, dsts, rb, p, p, 4, 1, 16, None) == -1
    assert gn(5, srcs, dsts, rb, p, p, 4, 1, 16, None) == -1
    assert gn(3, srcs, dsts, rb, p, p, 17, 1, 16, None) == -1            # k_max > N
    assert gn(3, (C.c_void_p * 3)(256, None, 768), dsts, rb, p, p, 4, 1, 16, None) == -1
    assert "cache 1" in _err(dl)
    assert gn(3, (C.c_void_p * 3)(256, 520, 768), dsts, rb, p, p, 4, 1, 16, None) == -1   # alignment
    assert gn(3, srcs, dsts, (C.c_int * 3)(8192, 8200, 8192), p, p, 4, 1, 16, None) == -1


def test_binding_fails_loudly_without_cuda_tensors(dl):
    import torch
    H = torch.zeros((1, 8, 64), dtype=torch.bfloat16)
    Pt = torch.zeros((32, 64), dtype=torch.bfloat16)
    pc = torch.zeros((1, 8, 32), dtype=torch.float32)
    with pytest.raises(dl.DllmError):
        dl.dllm_proxy_score(H, Pt, pc)
