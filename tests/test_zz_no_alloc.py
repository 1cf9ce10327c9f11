"""mxq_grouped_dbias_noalloc: per-expert dbias for callers that cannot
allocate device memory (its scratch is a fixed file-scope device array).

Called through the C ABI on two calls in a row with different inputs and
groupings, so that a stale partial from the first call would show up in the
second. It runs the same kernels in the same order as mxq_grouped_dbias
(which takes a caller workspace), so the two results must be identical bit
for bit; both must also be within the dbias tolerance of the other tests,
1e-5 * sum|dY| per column, of the oracle's fp64 per-expert sums. Collected
last so that a run stopping at the first failure has run every other test;
it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _call_noalloc(L, dy, ms, out, status):
    M, N = dy.shape
    return L.mxq_grouped_dbias_noalloc(dy.data_ptr(), M, N, ms.numel(), ms.data_ptr(), out.data_ptr(),
                                       status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _call_with_workspace(L, dy, ms, out):
    M, N = dy.shape
    ws = torch.empty(max(16, (M // 128) * N * 4), dtype=torch.uint8, device="cuda")
    return L.mxq_grouped_dbias(dy.data_ptr(), M, N, ms.numel(), ms.data_ptr(), out.data_ptr(), None,
                               ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_dbias_matches_workspace_dbias_twice():
    import oracle as orc
    from tests._gpu import bf16_to_f64, lib, require_gpu

    require_gpu()
    L = lib().mxq.lib()
    cases = [
        (8192, 2048, [2048, 0, 4096, 2048], 1),     # (M/128)*N = 131072 partials
        (1024, 640, [384, 640, 0], 2),              # smaller: a stale tail of call 1 must not leak in
    ]
    for M, N, splits, seed in cases:
        g = torch.Generator(device="cuda").manual_seed(seed)
        dy = torch.randn((M, N), generator=g, device="cuda").to(torch.bfloat16)
        ms = torch.tensor(splits, dtype=torch.int64, device="cuda")
        E = len(splits)
        got = torch.full((E, N), float("nan"), dtype=torch.float32, device="cuda")
        ref = torch.full((E, N), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _call_noalloc(L, dy, ms, got, status) == 0
        assert _call_with_workspace(L, dy, ms, ref) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), (M, N, "not bit-identical")
        bits = dy.view(torch.int16).cpu().numpy().view(np.uint16)
        want = orc.grouped_dbias(bits, np.array(splits, np.int64))
        a = np.abs(bf16_to_f64(bits))
        off = np.concatenate([[0], np.cumsum(splits)])
        for e in range(E):
            tol = 1e-5 * a[off[e]:off[e + 1]].sum(axis=0) + 1e-30
            for name, t in (("noalloc", got), ("workspace", ref)):
                diff = np.abs(t[e].double().cpu().numpy() - want[e])
                assert np.all(diff <= tol), (name, M, N, e)
            if splits[e] == 0:
                assert bool((got[e] == 0).all())


def test_noalloc_dbias_rejects_oversized_problem():
    from tests._gpu import lib, require_gpu

    require_gpu()
    L = lib().mxq.lib()
    M, N = 128 * 1025, 2048                         # 1025 * 2048 partials > 2,097,152
    dy = torch.empty((128, 128), dtype=torch.bfloat16, device="cuda")   # never read: rejected on the host
    ms = torch.tensor([M], dtype=torch.int64, device="cuda")
    out = torch.empty((1, N), dtype=torch.float32, device="cuda")
    rc = L.mxq_grouped_dbias_noalloc(dy.data_ptr(), M, N, 1, ms.data_ptr(), out.data_ptr(), None,
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == -9
    assert L.mxq_error_string(rc).decode().startswith("(M/128)*N exceeds")
