"""The allocation-free vocabulary entry point (dllm_commit_entropy_noalloc), called
through the C ABI: for callers that cannot allocate device memory it keeps its scratch
in a fixed device array of the library.  Its outputs must equal those of
dllm_commit_entropy (with a caller workspace) on two consecutive calls, which also
shows that the shared array's leftover contents from the first call do not leak into
the second.  This file is collected last on purpose."""
import ctypes as C

import numpy as np
import pytest

from sparse_kv_cache_rank_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

RTOL = 1e-4   # the fp32-reduction tolerance of the parity tests


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_cache_rank_gb300 import binding
    binding.lib()
    return binding


def _case(B_, M, V, seed, scale):
    logits = synth.commit_logits(B_, M, V, seed, std=3.0 * scale)
    valid = np.ones((B_, M), np.uint8)
    valid[-1, ::4] = 0
    return torch.from_numpy(logits).cuda(), torch.from_numpy(valid).cuda()


def _compare(ref, got):
    tok_r, conf_r, ent_r, E_r, full_r = (t.cpu().numpy() for t in ref)
    tok_g, conf_g, ent_g, E_g, full_g = (t.cpu().numpy() for t in got)
    np.testing.assert_allclose(conf_g, conf_r, rtol=RTOL, atol=1e-9)
    np.testing.assert_allclose(ent_g, ent_r, rtol=RTOL, atol=1e-6)
    np.testing.assert_allclose(E_g, E_r, rtol=RTOL, atol=1e-6)
    np.testing.assert_array_equal(tok_g, tok_r)
    np.testing.assert_array_equal(full_g, full_r)


def test_noalloc_matches_workspace_entry_point_twice(B):
    # two different problems back to back through the same device array
    for (Bq, M, V, seed, scale) in [(2, 32, 126464, 7, 0.43), (1, 24, 4096, 8, 10.0)]:
        logits, valid = _case(Bq, M, V, seed, scale)
        ref = B.dllm_commit_entropy(logits, valid)
        got = B.dllm_commit_entropy_noalloc(logits, valid)
        torch.cuda.synchronize()
        _compare(ref, got)


def test_noalloc_rejects_oversized_problems(B):
    # 17 x 1024 rows need one state each: more than the 16384 the array holds
    Bq, M, V = 17, 1024, 16
    logits = torch.zeros((Bq, M, V), device="cuda")
    valid = torch.ones((Bq, M), dtype=torch.uint8, device="cuda")
    out = [torch.empty((Bq, M), dtype=torch.int32, device="cuda")] + \
          [torch.empty((Bq, M), device="cuda") for _ in range(2)] + \
          [torch.empty((Bq,), device="cuda"), torch.empty((Bq,), dtype=torch.int32, device="cuda")]
    rc = B.lib().dllm_commit_entropy_noalloc(
        C.c_void_p(logits.data_ptr()), C.c_void_p(valid.data_ptr()), Bq, M, V, 0.9, 2.0,
        *[C.c_void_p(t.data_ptr()) for t in out], None)
    assert rc == -2
    assert b"allocation-free" in B.lib().dllm_last_error()
