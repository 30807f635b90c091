"""GEMM launches that overlap the previous kernel (programmatic dependent launch).

Each GEMM kernel may start while the kernel before it in the stream is still
running; it streams weights at once but reads A, and writes C, the split-K
partials and counters, only after the earlier kernel has completed.  A chain
X -> Y = X W1 -> X' = Y W2 written back over X exercises both hazards: the
second GEMM reads what the first writes (Y), and overwrites what the first
reads (X).  Every pair of kernel families runs back to back with no host
synchronization, eagerly and replayed from a CUDA graph, and both results are
checked against the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
from tests._util import bits_of, c_values, packed_from
from w4a16_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu

TOL = 1e-2
M, K1, N1 = 4, 4096, 512

FAMILIES = {
    "gemv": dict(kernel="gemv", split_k=2),
    "tc_decode": dict(kernel="tc_decode", block_m=16, dq_warps=8),
    "tc": dict(kernel="tc", block_m=16, split_k=4, dq_warps=8),
    "dm_cluster": dict(kernel="decode_mma", block_m=8, split_k=2, dq_warps=1),
    "dm_streamk": dict(kernel="decode_mma", block_m=8, split_k=0, dq_warps=4),
}
PAIRS = [("gemv", "gemv"), ("tc_decode", "tc_decode"), ("tc", "tc"), ("gemv", "tc_decode"),
         ("tc_decode", "gemv"), ("tc", "tc_decode"), ("tc_decode", "tc"), ("dm_cluster", "dm_cluster"),
         ("dm_streamk", "dm_streamk"), ("dm_cluster", "dm_streamk"), ("dm_streamk", "tc"),
         ("tc", "dm_cluster"), ("gemv", "dm_streamk")]


@pytest.fixture(scope="module")
def chain():
    qw1, a = synth.random_problem(41, M, K1, N1, 128, "f16")
    qw2, _ = synth.random_problem(42, 1, N1, K1, 128, "f16")
    w1 = oracle.dequant_bits(qw1.q, qw1.scales, qw1.zeros, 128, "f16")
    w2 = oracle.dequant_bits(qw2.q, qw2.scales, qw2.zeros, 128, "f16")
    return packed_from(qw1), packed_from(qw2), a, w1, w2


def _check(y, x_new, a_bits, w1, w2, what):
    y_ref = oracle.gemm_ref(a_bits, w1, "f16")
    assert oracle.max_err_ratio(c_values(y), y_ref, rel=TOL) <= 1.0, ("first GEMM", what)
    # the second GEMM's reference uses the first one's output as produced
    x_ref = oracle.gemm_ref(bits_of(y), w2, "f16")
    assert oracle.max_err_ratio(c_values(x_new), x_ref, rel=TOL) <= 1.0, ("second GEMM", what)


@pytest.mark.parametrize("first,second", PAIRS)
def test_back_to_back_chain(chain, first, second):
    W1, W2, a_bits, w1, w2 = chain
    x0 = binding.acts_to_device(a_bits, torch.float16)
    X = torch.empty_like(x0)
    Y = torch.empty((M, N1), dtype=torch.float16, device="cuda")
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for _ in range(5):
            X.copy_(x0)
            Y.fill_(float("nan"))
            binding.gemm(X, W1, out=Y, config=FAMILIES[first], stream=st)
            binding.gemm(Y, W2, out=X, config=FAMILIES[second], stream=st)
        torch.cuda.synchronize()
    binding.poll_error(st)
    _check(Y, X, a_bits, w1, w2, (first, second, "eager"))

    # the same pair captured in a graph (programmatic edges), replayed twice
    with torch.cuda.stream(st):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            X.copy_(x0)
            Y.fill_(float("nan"))
            binding.gemm(X, W1, out=Y, config=FAMILIES[first], stream=st)
            binding.gemm(Y, W2, out=X, config=FAMILIES[second], stream=st)
        X.fill_(float("nan"))
        g.replay()
        g.replay()
        torch.cuda.synchronize()
    binding.poll_error(st)
    _check(Y, X, a_bits, w1, w2, (first, second, "graph"))
    assert np.isfinite(c_values(X)).all()


@pytest.mark.parametrize("family", sorted(FAMILIES))
def test_pack_then_gemm_on_the_same_stream(family):
    """The kernels request the packed weights before waiting for the previous
    kernel: a GEMM launched right after the repack that writes its weights,
    on the same stream and with no synchronization between, must still see
    them complete."""
    qw, a = synth.random_problem(43, M, K1, N1, 128, "f16")
    w = oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 128, "f16")
    p = binding.to_device(qw)
    A = binding.acts_to_device(a, torch.float16)
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    for _ in range(3):
        W = binding.pack(p.q, p.scales, p.zeros, qw.group, stream=st)
        C = torch.empty((M, N1), dtype=torch.float16, device="cuda")
        with torch.cuda.stream(st):
            binding.gemm(A, W, out=C, config=FAMILIES[family], stream=st)
        st.synchronize()
        binding.poll_error(st)
        assert oracle.max_err_ratio(c_values(C), oracle.gemm_ref(a, w, "f16"), rel=TOL) <= 1.0
        W.free(stream=st)
        st.synchronize()
