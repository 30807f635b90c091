"""GPU parity of the W4A16 GEMM against the CPU oracle.

Tolerance (per element, fp32 accumulation): |C - C_ref| <= 1e-2 (|C_ref| +
rms(C_ref)), C_ref the float64 oracle GEMM of A with W = RNE_T(s*(q-z)).
Exact cases: q == z gives C == 0, one-hot rows reproduce W's rows, and
power-of-two scales with small-integer activations give C == C_ref exactly.
"""

import numpy as np
import pytest
import torch

import oracle
from tests._util import TORCH_DT, gemm_poisoned, bits_of, c_values, oracle_sampled, packed_from, sample_indices
from w4a16_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _run(qw, a_bits, config=None):
    W = packed_from(qw)
    A = binding.acts_to_device(a_bits, TORCH_DT[qw.dtype])
    C = gemm_poisoned(A, W, config=config)
    torch.cuda.synchronize()
    binding.poll_error()
    return C, W


# (block_m, dq_warps) pairs whose pipeline cannot keep every parity wait within
# one phase (four dequant warpgroups need STAGES % 4 == 0 and 13 / 7 TMEM A slots)
ILLEGAL = {(16, 16), (64, 16), (256, 16)}
DECODE_ILLEGAL = {(64, 12), (64, 16)}   # 3-4 warpgroups leave too few TMEM columns at block_m 64


def _decode_variants(M):
    """Every legal tcgen05-decode variant and, for M <= 16, the register-MMA
    decode kernel on persistent grids of one and of all resident CTAs per SM,
    with one, two and four K-groups, and in clusters of 4 and of 16 CTAs per
    tile, and the tensor-core GEMV."""
    out = [dict(kernel="tc_decode", block_m=bm, dq_warps=dq)
           for bm in (16, 32, 64) for dq in (4, 8, 12, 16) if (bm, dq) not in DECODE_ILLEGAL]
    if M <= 16:
        out += [dict(kernel="decode_mma", split_k=1), dict(kernel="decode_mma", split_k=0),
                dict(kernel="decode_mma", split_k=0, dq_warps=8),
                dict(kernel="decode_mma", split_k=1, dq_warps=16),
                dict(kernel="decode_mma", split_k=4, dq_warps=1),
                dict(kernel="decode_mma", split_k=16, dq_warps=1),
                dict(kernel="decode_mma", split_k=8, dq_warps=2),
                dict(kernel="gemv", split_k=2, dq_warps=1)]
    return out


def _variants(M):
    out = []
    if M <= 8:
        out += [dict(kernel="gemv", split_k=1), dict(kernel="gemv", split_k=3)]
    if M <= 16:
        out += [dict(kernel="gemv", split_k=1, dq_warps=1), dict(kernel="gemv", split_k=3, dq_warps=1)]
    if M <= 16:
        out += [dict(kernel="decode_mma", split_k=1), dict(kernel="decode_mma", split_k=3),
                dict(kernel="decode_mma", split_k=2, dq_warps=8),
                dict(kernel="decode_mma", split_k=1, dq_warps=16),
                dict(kernel="decode_mma", split_k=3, dq_warps=1)]
    for bm in (16, 32, 64, 128, 256):
        for sk in (1, 3):
            for dq in (4, 8, 16):
                if (bm, dq) in ILLEGAL:
                    continue                      # rejected: see test_illegal_variants
                if bm >= 128 and dq != 8 and sk == 3:
                    continue
                out.append(dict(kernel="tc", block_m=bm, split_k=sk, dq_warps=dq))
    for bm in (16, 32, 64):
        for dq in (4, 8, 12, 16):
            if (bm, dq) in DECODE_ILLEGAL:
                continue
            out.append(dict(kernel="tc_decode", block_m=bm, dq_warps=dq))
    return out


SMALL = [
    # M, K, N, G, dtype, sym
    (1, 512, 384, 128, "f16", False),
    (3, 512, 256, 128, "bf16", False),
    (16, 1024, 384, 64, "f16", True),
    (17, 512, 256, 128, "f16", False),
    (100, 768, 256, 128, "bf16", False),
    (257, 512, 384, 64, "f16", True),
    (5, 320, 256, 64, "bf16", True),      # 5 K blocks: a partial 4-block stage
    (40, 1216, 128, 64, "f16", False),    # 19 K blocks, 3 row tiles of 16, one column tile
]


@pytest.mark.parametrize("M,K,N,G,dt,sym", SMALL)
def test_small_all_variants(M, K, N, G, dt, sym):
    qw, a = synth.random_problem(M + K + N, M, K, N, G, dt, sym,
                                 act_dist="student_t3" if sym else "normal")
    w = oracle.dequant_bits(qw.q, qw.scales, qw.zeros, G, dt)
    c_ref = oracle.gemm_ref(a, w, dt)
    W = packed_from(qw)
    A = binding.acts_to_device(a, TORCH_DT[dt])
    for cfg in _variants(M):
        C = gemm_poisoned(A, W, config=cfg)
        torch.cuda.synchronize()
        binding.poll_error()
        r = oracle.max_err_ratio(c_values(C), c_ref, rel=TOL)
        assert r <= 1.0, (cfg, r)


def test_repeated_runs_are_identical():
    """Many launches of the deepest-pipelined variants give bit-identical C
    (catches pipeline races that only show under some schedules)."""
    M, K, N = 512, 4096, 2048
    qw, a = synth.random_problem(23, M, K, N, 128, "bf16")
    c_ref = oracle.gemm_ref(a[:64], oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 128, "bf16"), "bf16")
    W = packed_from(qw)
    A = binding.acts_to_device(a, torch.bfloat16)
    for cfg in (dict(kernel="tc", block_m=256, split_k=1, dq_warps=4),
                dict(kernel="tc", block_m=128, split_k=1, dq_warps=8),
                dict(kernel="tc", block_m=32, split_k=2, dq_warps=16),
                dict(kernel="tc", block_m=16, split_k=4, dq_warps=8)):
        first = gemm_poisoned(A, W, config=cfg)
        torch.cuda.synchronize()
        assert oracle.max_err_ratio(c_values(first)[:64], c_ref, rel=TOL) <= 1.0, cfg
        for _ in range(25):
            C = gemm_poisoned(A, W, config=cfg)
            torch.cuda.synchronize()
            assert torch.equal(C.view(torch.int16), first.view(torch.int16)), cfg


@pytest.mark.parametrize("M", [1, 4, 16, 64, 200])
def test_auto_selection_is_deterministic(M):
    qw, a = synth.random_problem(11, M, 2048, 512)
    C1, W = _run(qw, a)
    A = binding.acts_to_device(a, torch.float16)
    C2 = gemm_poisoned(A, W)
    torch.cuda.synchronize()
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
    c_ref = oracle.gemm_ref(a, oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 128, "f16"), "f16")
    assert oracle.max_err_ratio(c_values(C1), c_ref, rel=TOL) <= 1.0


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_q_equal_zero_gives_exact_zero(dt):
    M, K, N, G = 40, 512, 256, 128
    qw, a = synth.random_problem(3, M, K, N, G, dt)
    q = np.repeat(qw.zeros, G, axis=0)
    qz = synth.QuantWeight(q, qw.scales, qw.zeros, G, dt)
    W = packed_from(qz)
    A = binding.acts_to_device(a, TORCH_DT[dt])
    A8 = A[:8].contiguous()
    for cfg in [None, dict(kernel="tc", block_m=64, split_k=2)] + _decode_variants(M):
        C = gemm_poisoned(A, W, config=cfg)
        torch.cuda.synchronize()
        assert torch.count_nonzero(C.float()) == 0, cfg
    for cfg in [dict(kernel="gemv", split_k=2), dict(kernel="decode_mma", split_k=4)]:
        C = gemm_poisoned(A8, W, config=cfg)
        torch.cuda.synchronize()
        assert torch.count_nonzero(C.float()) == 0, cfg
    binding.poll_error()


def test_one_hot_rows_reproduce_dequantized_weight():
    K, N, G = 512, 256, 128
    qw, _ = synth.random_problem(4, 1, K, N, G)
    w = oracle.dequant_bits(qw.q, qw.scales, qw.zeros, G, "f16")
    ks = [0, 1, 63, 64, 127, 128, 255, 256, 511]
    a = np.zeros((len(ks), K), np.uint16)
    for i, k in enumerate(ks):
        a[i, k] = 0x3C00
    W = packed_from(qw)
    A = binding.acts_to_device(a, torch.float16)
    for cfg in [dict(kernel="tc", block_m=16, split_k=1), dict(kernel="tc", block_m=16, split_k=3),
                dict(kernel="tc", block_m=128, split_k=1, dq_warps=8),
                dict(kernel="tc", block_m=32, split_k=5, dq_warps=8),
                dict(kernel="decode_mma", split_k=4)] + _decode_variants(len(ks)):
        C = gemm_poisoned(A, W, config=cfg)
        torch.cuda.synchronize()
        assert np.array_equal(bits_of(C), w[ks]), cfg
    # the CUDA-core GEMV takes at most 8 rows: the last 8 one-hot rows
    A8 = A[1:].contiguous()
    for cfg in [dict(kernel="gemv", split_k=1), dict(kernel="gemv", split_k=4),
                dict(kernel="decode_mma", split_k=1)]:
        C = gemm_poisoned(A8, W, config=cfg)
        torch.cuda.synchronize()
        assert np.array_equal(bits_of(C), w[ks[1:]]), cfg
    binding.poll_error()


def test_identity_activation_reproduces_weight():
    """A = I (M = K = 256): C == W exactly (tensor-core path)."""
    K = N = 256
    qw, _ = synth.random_problem(6, 1, K, N, 128)
    w = oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 128, "f16")
    a = np.where(np.eye(K, dtype=bool), np.uint16(0x3C00), np.uint16(0))
    W = packed_from(qw)
    A = binding.acts_to_device(a, torch.float16)
    for cfg in [dict(kernel="tc", block_m=bm) for bm in (64, 128, 256)] + \
            [c for c in _decode_variants(K) if c["kernel"] == "tc_decode"]:
        C = gemm_poisoned(A, W, config=cfg)
        torch.cuda.synchronize()
        assert np.array_equal(bits_of(C), w), cfg
    # the register-MMA decode kernel takes at most 16 rows: slabs of I
    for k0 in (0, 96, 240):
        for cfg in (dict(split_k=1), dict(split_k=2), dict(split_k=1, dq_warps=16),
                    dict(split_k=4, dq_warps=1)):
            C = gemm_poisoned(A[k0:k0 + 16].contiguous(), W, config=dict(kernel="decode_mma", **cfg))
            torch.cuda.synchronize()
            assert np.array_equal(bits_of(C), w[k0:k0 + 16]), (k0, cfg)
        # the tensor-core GEMV takes up to 16 rows too
        for sk in (1, 3):
            C = gemm_poisoned(A[k0:k0 + 16].contiguous(), W, config=dict(kernel="gemv", split_k=sk, dq_warps=1))
            torch.cuda.synchronize()
            assert np.array_equal(bits_of(C), w[k0:k0 + 16]), (k0, sk)
    binding.poll_error()


@pytest.mark.parametrize("M", [1, 5, 48, 300])
def test_power_of_two_scales_are_exact(M):
    """Scales 2^-e and integer activations keep every partial sum exact."""
    K, N, G = 512, 256, 64
    rng = np.random.default_rng(M)
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    z = rng.integers(6, 10, size=(K // G, N), dtype=np.uint8)
    s = oracle.rne_f16_bits(np.exp2(-rng.integers(6, 10, size=(K // G, N)).astype(np.float64)))
    a_int = rng.integers(-2, 3, size=(M, K))
    a_int[rng.random((M, K)) < 0.75] = 0
    a = oracle.rne_f16_bits(a_int.astype(np.float64))
    qw = synth.QuantWeight(q, s, z, G, "f16")
    c_ref = oracle.gemm_ref(a, oracle.dequant_bits(q, s, z, G, "f16"), "f16")
    assert np.all(np.abs(c_ref) < 2048)
    W = packed_from(qw)
    A = binding.acts_to_device(a, torch.float16)
    cfgs = [None, dict(kernel="tc", block_m=16, split_k=4), dict(kernel="tc", block_m=64, split_k=2),
            dict(kernel="tc", block_m=256)] + _decode_variants(M)
    if M <= 8:
        cfgs += [dict(kernel="gemv", split_k=1), dict(kernel="gemv", split_k=3)]
    if M <= 16:
        cfgs += [dict(kernel="decode_mma", split_k=8)]
    for cfg in cfgs:
        C = gemm_poisoned(A, W, config=cfg)
        torch.cuda.synchronize()
        assert np.array_equal(c_values(C), c_ref), cfg
    binding.poll_error()


def test_symmetric_equals_asymmetric_with_zero_eight():
    M, K, N, G = 24, 512, 256, 64
    qw, a = synth.random_problem(8, M, K, N, G, "f16", True)
    Ws = packed_from(qw)
    Wa = packed_from(synth.QuantWeight(qw.q, qw.scales, np.full((K // G, N), 8, np.uint8), G, "f16"))
    A = binding.acts_to_device(a, torch.float16)
    assert torch.equal(binding.dequant(Ws).view(torch.int16), binding.dequant(Wa).view(torch.int16))
    for cfg in [None, dict(kernel="tc", block_m=32, split_k=2)] + _decode_variants(M):
        Cs = gemm_poisoned(A, Ws, config=cfg)
        Ca = gemm_poisoned(A, Wa, config=cfg)
        torch.cuda.synchronize()
        assert torch.equal(Cs.view(torch.int16), Ca.view(torch.int16)), cfg
    binding.poll_error()


def test_long_k_every_legal_variant():
    """K = 8192 (128 blocks): many wrap-arounds of every stage and TMEM ring."""
    M, K, N = 40, 8192, 256
    qw, a = synth.random_problem(21, M, K, N)
    c_ref = oracle.gemm_ref(a, oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 128, "f16"), "f16")
    W = packed_from(qw)
    A = binding.acts_to_device(a, torch.float16)
    for bm in (16, 32, 64, 128, 256):
        for dq in (4, 8, 16):
            if (bm, dq) in ILLEGAL:
                continue
            for sk in (1, 2):
                C = gemm_poisoned(A, W, config=dict(kernel="tc", block_m=bm, split_k=sk, dq_warps=dq))
                torch.cuda.synchronize()
                binding.poll_error()
                assert oracle.max_err_ratio(c_values(C), c_ref, rel=TOL) <= 1.0, (bm, dq, sk)
    for bm in (16, 32, 64):
        for dq in (4, 8, 12, 16):
            if (bm, dq) in DECODE_ILLEGAL:
                continue
            cfg = dict(kernel="tc_decode", block_m=bm, dq_warps=dq)
            C = gemm_poisoned(A, W, config=cfg)
            torch.cuda.synchronize()
            binding.poll_error()
            assert oracle.max_err_ratio(c_values(C), c_ref, rel=TOL) <= 1.0, cfg


@pytest.mark.parametrize("M,G,dt", [(1, 128, "f16"), (16, 64, "bf16"), (9, 128, "bf16")])
def test_long_k_decode_mma(M, G, dt):
    """K = 8192: many wrap-arounds of the copy ring, tiles cut between CTAs of
    persistent grids of several sizes, both group sizes and types."""
    K, N = 8192, 384
    qw, a = synth.random_problem(31 + M, M, K, N, G, dt)
    c_ref = oracle.gemm_ref(a, oracle.dequant_bits(qw.q, qw.scales, qw.zeros, G, dt), dt)
    W = packed_from(qw)
    A = binding.acts_to_device(a, TORCH_DT[dt])
    cfgs = [dict(split_k=sk) for sk in (1, 2, 3, 5, 0)] + \
        [dict(split_k=sk, dq_warps=dq) for sk in (1, 2) for dq in (8, 16)] + \
        [dict(split_k=sk, dq_warps=1) for sk in (1, 2, 7, 16)]
    for cfg in cfgs:
        C = gemm_poisoned(A, W, config=dict(kernel="decode_mma", **cfg))
        torch.cuda.synchronize()
        binding.poll_error()
        assert oracle.max_err_ratio(c_values(C), c_ref, rel=TOL) <= 1.0, cfg


@pytest.mark.parametrize("K,N,G", [(256, 16384, 128), (1024, 8192, 64), (4096, 1152, 128)])
@pytest.mark.parametrize("M", [1, 16])
def test_stream_k_segments_decode_mma(K, N, G, M):
    """Persistent grids whose CTAs cover whole tiles, the end of one tile and
    the start of the next, or a piece strictly inside one tile; compared
    with the oracle on every output."""
    qw, a = synth.random_problem(40 + K // 64 + M, M, K, N, G, "f16")
    c_ref = oracle.gemm_ref(a, oracle.dequant_bits(qw.q, qw.scales, qw.zeros, G, "f16"), "f16")
    W = packed_from(qw)
    A = binding.acts_to_device(a, torch.float16)
    for cfg in [dict(split_k=sk) for sk in (1, 2, 0)] + \
            [dict(split_k=sk, dq_warps=dq) for dq in (8, 16) for sk in (1, 0)]:
        cfg = dict(kernel="decode_mma", **cfg)
        C = gemm_poisoned(A, W, config=cfg)
        torch.cuda.synchronize()
        binding.poll_error()
        assert oracle.max_err_ratio(c_values(C), c_ref, rel=TOL) <= 1.0, cfg
        # determinism: a second launch is bit-identical
        C2 = gemm_poisoned(A, W, config=cfg)
        torch.cuda.synchronize()
        assert torch.equal(C.view(torch.int16), C2.view(torch.int16)), cfg


@pytest.mark.parametrize("K,G", [(256, 128), (1024, 64), (14336, 128)])
@pytest.mark.parametrize("M", [1, 11])
def test_cluster_split_decode_mma(K, G, M):
    """Cluster split-K: one cluster of S CTAs per tile, each taking an equal
    group-aligned K range (the last one shorter, or empty when the groups do
    not divide evenly), partial sums added through distributed shared
    memory; one and two K-groups per CTA.  Cluster sizes up to 16 (capped
    for larger M), against the oracle on every output, and bit-identical on
    a second launch."""
    N = 640
    qw, a = synth.random_problem(70 + K // 64 + M, M, K, N, G, "bf16")
    c_ref = oracle.gemm_ref(a, oracle.dequant_bits(qw.q, qw.scales, qw.zeros, G, "bf16"), "bf16")
    W = packed_from(qw)
    A = binding.acts_to_device(a, torch.bfloat16)
    for sk, dq in [(s, 1) for s in (1, 2, 3, 5, 8, 11, 16)] + [(s, 2) for s in (2, 5, 16)]:
        cfg = dict(kernel="decode_mma", split_k=sk, dq_warps=dq)
        C = gemm_poisoned(A, W, config=cfg)
        torch.cuda.synchronize()
        binding.poll_error()
        assert oracle.max_err_ratio(c_values(C), c_ref, rel=TOL) <= 1.0, sk
        C2 = gemm_poisoned(A, W, config=cfg)
        torch.cuda.synchronize()
        assert torch.equal(C.view(torch.int16), C2.view(torch.int16)), sk


def test_illegal_variants_are_rejected():
    """Variants whose parity waits could run two phases ahead are refused."""
    qw, a = synth.random_problem(22, 16, 512, 256)
    W = packed_from(qw)
    A = binding.acts_to_device(a, torch.float16)
    for bm, _ in sorted(ILLEGAL):
        with pytest.raises(binding.TmError) as e:
            binding.gemm(A, W, config=dict(kernel="tc", block_m=bm, dq_warps=16))
        assert e.value.status == binding.TM_ERR_UNSUPPORTED
    for bm, dq in ((128, 8), (16, 2), (48, 8), (16, 20), (64, 12), (64, 16)):
        with pytest.raises(binding.TmError) as e:
            binding.gemm(A, W, config=dict(kernel="tc_decode", block_m=bm, dq_warps=dq))
        assert e.value.status == binding.TM_ERR_UNSUPPORTED
    # the register-MMA decode kernel takes at most 16 rows, and 4, 8 or 16
    # consumer warps (1: clusters)
    A17 = binding.acts_to_device(np.zeros((17, 512), np.uint16), torch.float16)
    with pytest.raises(binding.TmError) as e:
        binding.gemm(A17, W, config=dict(kernel="decode_mma"))
    assert e.value.status == binding.TM_ERR_UNSUPPORTED
    for dq in (3, 12, 32):
        with pytest.raises(binding.TmError) as e:
            binding.gemm(A[:4].contiguous(), W, config=dict(kernel="decode_mma", dq_warps=dq))
        assert e.value.status == binding.TM_ERR_UNSUPPORTED


def test_m_zero_is_noop_and_argument_errors():
    qw, a = synth.random_problem(9, 4, 256, 256)
    W = packed_from(qw)
    A = torch.zeros((0, 256), dtype=torch.float16, device="cuda")
    C = gemm_poisoned(A, W)
    assert C.shape == (0, 256)
    A = binding.acts_to_device(a, torch.float16)
    A9 = binding.acts_to_device(np.zeros((9, 256), np.uint16), torch.float16)
    with pytest.raises(binding.TmError) as e:
        binding.gemm(A9, W, config=dict(kernel="gemv"))     # GEMV takes M <= 8
    assert e.value.status == binding.TM_ERR_UNSUPPORTED
    A17 = binding.acts_to_device(np.zeros((17, 256), np.uint16), torch.float16)
    for dq in (1, 2):                                       # tensor-core GEMV: M <= 16; dq_warps 0 or 1
        with pytest.raises(binding.TmError) as e:
            binding.gemm(A17 if dq == 1 else A, W, config=dict(kernel="gemv", dq_warps=dq))
        assert e.value.status == binding.TM_ERR_UNSUPPORTED
    with pytest.raises(binding.TmError) as e:
        binding.gemm(A, W, config=dict(kernel="tc", block_m=48))
    assert e.value.status == binding.TM_ERR_UNSUPPORTED
    with pytest.raises(binding.TmError) as e:
        binding.gemm(A, W, config=dict(kernel="tc", block_m=16, split_k=5))
    assert e.value.status == binding.TM_ERR_UNSUPPORTED
    Abig = torch.zeros(4 * 256 + 8, dtype=torch.float16, device="cuda")[1:1 + 4 * 256].view(4, 256)
    with pytest.raises(binding.TmError) as e:
        gemm_poisoned(Abig, W)
    assert e.value.status == binding.TM_ERR_INVALID_ARG


# ---------------------------------------------------------------- full size
FULL = [(wl, si, M) for wl in ("decode_8b", "prefill_8b", "class_70b", "sym_g64")
        for si in range(len(synth.WORKLOADS[wl].shapes)) for M in synth.WORKLOADS[wl].ms]


@pytest.fixture(scope="module")
def weight_cache():
    cache = {}
    yield cache
    cache.clear()


@pytest.mark.parametrize("wl,si,M", FULL, ids=lambda x: str(x))
def test_full_size_sampled(wl, si, M, weight_cache):
    """Every (workload, shape, M) at full size, in the launch configuration the
    benchmark times (the variant tm_tune measures fastest, then tm_gemm_w4a16);
    sampled rows and columns are checked against the oracle."""
    key = (wl, si)
    if key not in weight_cache:
        weight_cache.clear()
        qw = synth.weight(wl, si)
        weight_cache[key] = (qw, packed_from(qw))
    qw, W = weight_cache[key]
    a = synth.activations(wl, si, M)
    A = binding.acts_to_device(a, TORCH_DT[qw.dtype])
    binding.tune(W, [M])                      # the benchmark's selection procedure
    C = gemm_poisoned(A, W)
    torch.cuda.synchronize()
    binding.poll_error()
    rows = sample_indices(M, 96, seed=M)
    cols = sample_indices(qw.N, 192, seed=qw.N + si)
    c_ref = oracle_sampled(qw, a, rows, cols)
    r = oracle.max_err_ratio(c_values(C, rows, cols), c_ref, rel=TOL)
    assert r <= 1.0, r


def test_alternating_problems_decode_kernel():
    """Stale-data races hide when one problem is repeated: a slot read too early
    returns the previous launch's identical data.  Two weights of one shape
    (the second is the first with its tiles rotated by one) alternate, every
    launch is compared bit for bit with the first launch of its problem, and
    those first launches are checked against the oracle.  The shape and M
    give every CTA a cut tile followed by whole tiles, where a failure showed."""
    M, G = 32, 64
    qw = synth.weight("sym_g64", 0)
    a = synth.activations("sym_g64", 0, M)
    roll = lambda x: np.ascontiguousarray(np.roll(x, 128, axis=1))
    qw2 = synth.QuantWeight(roll(qw.q), roll(qw.scales), None, qw.group, qw.dtype)
    A = binding.acts_to_device(a, torch.float16)
    Ws = [packed_from(qw), packed_from(qw2)]
    cols = sample_indices(qw.N, 160, seed=5)
    rows = np.arange(M)
    refs = [oracle_sampled(q, a, rows, cols) for q in (qw, qw2)]
    for cfg in (dict(kernel="tc_decode", block_m=64, dq_warps=4),
                dict(kernel="tc_decode", block_m=32, dq_warps=8),
                dict(kernel="tc_decode", block_m=16, dq_warps=8)):
        first = []
        for i in range(2):
            C = gemm_poisoned(A, Ws[i], config=cfg)
            torch.cuda.synchronize()
            assert oracle.max_err_ratio(c_values(C, rows, cols), refs[i], rel=TOL) <= 1.0, (cfg, i)
            first.append(C.view(torch.int16).clone())
        for r in range(40):
            C = gemm_poisoned(A, Ws[r % 2], config=cfg)
            torch.cuda.synchronize()
            assert torch.equal(C.view(torch.int16), first[r % 2]), (cfg, r)
        binding.poll_error()


def test_alternating_problems_decode_mma():
    """The same stale-data check for the register-MMA decode kernel: two
    weights of one shape alternate, each launch is compared bit for bit with
    the first launch of its problem, and those with the oracle."""
    M = 16
    qw = synth.weight("sym_g64", 0)
    a = synth.activations("sym_g64", 0, 32)[:M].copy()
    roll = lambda x: np.ascontiguousarray(np.roll(x, 128, axis=1))
    qw2 = synth.QuantWeight(roll(qw.q), roll(qw.scales), None, qw.group, qw.dtype)
    A = binding.acts_to_device(a, torch.float16)
    Ws = [packed_from(qw), packed_from(qw2)]
    cols = sample_indices(qw.N, 160, seed=6)
    rows = np.arange(M)
    refs = [oracle_sampled(q, a, rows, cols) for q in (qw, qw2)]
    for cfg in (dict(kernel="decode_mma", split_k=0), dict(kernel="decode_mma", split_k=1),
                dict(kernel="decode_mma", split_k=1, dq_warps=16),
                dict(kernel="decode_mma", split_k=8, dq_warps=1)):
        first = []
        for i in range(2):
            C = gemm_poisoned(A, Ws[i], config=cfg)
            torch.cuda.synchronize()
            assert oracle.max_err_ratio(c_values(C, rows, cols), refs[i], rel=TOL) <= 1.0, (cfg, i)
            first.append(C.view(torch.int16).clone())
        for r in range(30):
            C = gemm_poisoned(A, Ws[r % 2], config=cfg)
            torch.cuda.synchronize()
            assert torch.equal(C.view(torch.int16), first[r % 2]), (cfg, r)
        binding.poll_error()
