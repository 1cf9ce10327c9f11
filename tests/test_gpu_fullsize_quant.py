"""GPU parity at full size: group_quantize of every workload's weights (the
uniform-member mode, rowwise + colwise, swizzled scales) and of its bf16
output gradients (rowwise + colwise, swizzled), bit for bit against the oracle.

Weights are E uniform members of N rows each ([DI]: one grouped weight
(E, out, in) quantized with per-member swizzled scale bases; [FM]: the forward
GEMM reads the rowwise copy, dgrad the colwise copy). Where the oracle's fp64
copy of a whole weight would not fit comfortably on the host (the 128-expert
workload: 1.88 G elements), whole 128-row x full-K slabs are compared byte for
byte with their scale atoms -- the first and last slab of every expert and
seeded random ones. Slab j of expert e is quantized by the oracle as a member
of its own; its rowwise atoms sit at (e N + 128 j) / 128 * (K / 128) atoms into
the GPU's rowwise scales, its colwise atom for column block kb at
e K N / 32 + (kb (N / 128) + j) * 512 bytes into the colwise scales.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from synth import WORKLOADS, make_inputs
from tests._gpu import dev_bf16, first_diff, host, lib, require_gpu

pytestmark = pytest.mark.gpu

FULL_LIMIT = 1 << 29  # elements up to which the oracle quantizes the whole tensor


@pytest.fixture(scope="module")
def mxq():
    require_gpu()
    return lib()


def _equal(got, want, what):
    got = np.asarray(got).reshape(want.shape)
    assert np.array_equal(got, want), (what, first_diff(got, want))


def _check_whole(q, o, what):
    for dk, ok in (("row_data", "row_q"), ("row_scale", "row_s"), ("col_data", "col_q"), ("col_scale", "col_s")):
        _equal(host(q[dk]), o[ok], f"{what} {ok}")


def _slabs(E, N, seed, extra=24):
    per = N // 128
    s = {(e, 0) for e in range(E)} | {(e, per - 1) for e in range(E)}
    rng = np.random.default_rng(seed)
    for _ in range(extra):
        s.add((int(rng.integers(E)), int(rng.integers(per))))
    return sorted(s)


def _check_slabs(q, w, E, N, K, what, seed):
    row_q = q["row_data"].view(E * N, K)
    col_q = q["col_data"].view(E * N, K)
    nkb = K // 128
    for e, j in _slabs(E, N, seed):
        r0 = e * N + 128 * j
        o = orc.quantize_weights(w[e, 128 * j:128 * j + 128][None], swizzled=True)
        tag = f"{what} expert {e} slab {j}"
        _equal(host(row_q[r0:r0 + 128]), o["row_q"], tag + " row_q")
        _equal(host(col_q[r0:r0 + 128]), o["col_q"], tag + " col_q")
        a = (r0 // 128) * nkb * 512
        _equal(host(q["row_scale"][a:a + nkb * 512]), o["row_s"], tag + " row_s")
        base = e * K * N // 32
        idx = base + (np.arange(nkb)[:, None] * (N // 128) + j) * 512 + np.arange(512)[None, :]
        got = host(q["col_scale"][torch.from_numpy(idx.ravel()).cuda()])
        _equal(got, o["col_s"], tag + " col_s")


WEIGHTS = [(n, "w") for n in WORKLOADS] + [(n, "w2") for n, w in WORKLOADS.items() if w.F]


@pytest.mark.parametrize("name,key", WEIGHTS, ids=[f"{n}-{k}" for n, k in WEIGHTS])
def test_full_size_weight_quantize(mxq, name, key):
    wl = WORKLOADS[name]
    w = make_inputs(wl, which=(key,))[key]
    E, N, K = w.shape
    q = mxq.group_quantize(dev_bf16(w).view(E * N, K), None, E=E)
    torch.cuda.synchronize()
    if E * N * K <= FULL_LIMIT:
        _check_whole(q, orc.quantize_weights(w, swizzled=True), f"{name} {key}")
    else:
        _check_slabs(q, w, E, N, K, f"{name} {key}", wl.wid)


GRADS = [(n, "dy") for n in WORKLOADS] + [(n, "dy2") for n, w in WORKLOADS.items() if w.F and not w.prequant_dy]


@pytest.mark.parametrize("name,key", GRADS, ids=[f"{n}-{k}" for n, k in GRADS])
def test_full_size_gradient_quantize(mxq, name, key):
    """The bf16 output gradient of each workload's grouped linears, quantized row + col."""
    wl = WORKLOADS[name]
    d = make_inputs(wl, which=(key,))
    dy, ms = d[key], d["m_splits"]
    q = mxq.group_quantize(dev_bf16(dy), torch.from_numpy(ms).cuda())
    _check_whole(q, orc.group_quantize(dy, ms, swizzled=True), f"{name} {key}")
