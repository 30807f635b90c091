"""Decode attention over a low-bit KV cache (tm_attn_decode) against the
oracle: ragged lengths, every KV width and dtype, grouped-query layouts up
to 16 heads per KV head, units split over CTAs, exact special cases, cache
contents past the length, determinism, full-size sampled cases and the
argument checks."""

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as at
from w4a16_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def _dev(p: synth.KVProblem):
    dt = TORCH_DT[p.dtype]

    def h16(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(dt)

    return dict(q=h16(p.q), k_cache=torch.from_numpy(p.k_codes).cuda(), k_scale=h16(p.k_scale),
                k_zero=torch.from_numpy(p.k_zero).cuda(), v_cache=torch.from_numpy(p.v_codes).cuda(),
                v_scale=h16(p.v_scale), v_zero=torch.from_numpy(p.v_zero).cuda(),
                lens=torch.from_numpy(p.lens.astype(np.int32)).cuda())


def _run(p, chunk_tiles=0, d=None):
    d = d or _dev(p)
    o = binding.attn_decode(**d, kv_bits=p.bits, sm_scale=p.sm_scale, chunk_tiles=chunk_tiles)
    binding.poll_error()
    return o


def _bits(o):
    return o.view(torch.int16).cpu().numpy().view(np.uint16)


def _vals(o, dtype):
    return oracle.act_bits_to_f64(_bits(o), dtype)


def _ref(p):
    return at.attn_decode_ref(p.q, p.k_codes, p.k_scale, p.k_zero, p.v_codes, p.v_scale, p.v_zero,
                              p.lens, p.bits, p.dtype, p.sm_scale)


def _check(got, ref):
    assert np.isfinite(got).all()
    ratio = oracle.max_err_ratio(got, ref)
    assert ratio <= 1.0, ratio


LENS = [1, 63, 64, 65, 200, 0, 256, 130]


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (8, 2), (16, 2), (32, 2)])
@pytest.mark.parametrize("chunk_tiles", [0, 1, 3])
def test_ragged_parity(bits, dtype, Hq, Hkv, chunk_tiles):
    p = synth.kv_problem(10 + Hq, B=len(LENS), Hq=Hq, Hkv=Hkv, D=128, lens=LENS, L_max=256, bits=bits, dtype=dtype)
    got = _vals(_run(p, chunk_tiles), dtype)
    _check(got, _ref(p))
    assert np.all(got[5] == 0.0)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_single_token_is_exact(bits, dtype):
    """P = 1 exactly: O is the dequantized value row, bit for bit."""
    p = synth.kv_problem(20, B=3, Hq=8, Hkv=2, D=128, lens=[1, 1, 1], L_max=128, bits=bits, dtype=dtype)
    got = _bits(_run(p))
    for b in range(3):
        for hq in range(8):
            h = hq // 4
            vc = p.v_codes[b, h, :1] if bits == 8 else at.unpack_kv4(p.v_codes[b, h, :1])
            want = at.kv_dequant_bits(vc, p.v_scale[b, h, :1], p.v_zero[b, h, :1], dtype)[0]
            assert np.array_equal(got[b, hq], want), (b, hq)


@pytest.mark.parametrize("bits", [8, 4])
def test_equal_keys_average_values(bits):
    p = synth.kv_problem(21, B=2, Hq=4, Hkv=1, D=128, lens=[100, 700], L_max=768, bits=bits)
    p.k_codes[:] = p.k_codes[:, :, :1]
    p.k_scale[:] = p.k_scale[:, :, :1]
    p.k_zero[:] = p.k_zero[:, :, :1]
    got = _vals(_run(p, chunk_tiles=2), "f16")
    ref = _ref(p)
    assert np.allclose(got, ref, rtol=2e-3, atol=2e-3 * np.abs(ref).max())


@pytest.mark.parametrize("bits", [8, 4])
def test_cache_past_length_is_never_read_into_the_result(bits):
    p = synth.kv_problem(22, B=4, Hq=8, Hkv=2, D=128, lens=[5, 64, 100, 191], L_max=192, bits=bits)
    clean = _bits(_run(p, chunk_tiles=1))
    nan16 = np.uint16(0x7E00)
    for b, n in enumerate(p.lens):
        p.k_codes[b, :, n:] = 0xFF
        p.v_codes[b, :, n:] = 0xFF
        p.k_scale[b, :, n:] = nan16
        p.v_scale[b, :, n:] = nan16
        p.k_zero[b, :, n:] = 0
        p.v_zero[b, :, n:] = 0
    dirty = _bits(_run(p, chunk_tiles=1))
    assert np.array_equal(clean, dirty)


def test_repeat_is_bit_identical_and_lengths_clamp():
    p = synth.kv_problem(23, B=6, Hq=32, Hkv=8, D=128, lens=[900, 1, 4000, 64, 0, 2500], L_max=4096)
    d = _dev(p)
    a = _bits(_run(p, d=d))
    b = _bits(_run(p, d=d))
    assert np.array_equal(a, b)
    # a length beyond L_max reads as L_max, a negative one as 0
    d["lens"] = torch.tensor([5000, -3, 4000, 64, 0, 2500], dtype=torch.int32, device="cuda")
    c = _vals(_run(p, d=d), "f16")
    p.lens = np.array([4096, 0, 4000, 64, 0, 2500], dtype=np.int32)
    ref = _ref(p)
    _check(c, ref)


@pytest.mark.parametrize("name", ["attn_8b_kv8", "attn_8b_kv4"])
def test_full_size_sampled(name):
    """The bench's largest-context case, checked on a sample of sequences."""
    wl = synth.ATTN_WORKLOADS[name]
    ci = 1
    lens = synth.attn_lens(name, ci)
    p = synth.kv_problem(100 + ci, B=len(lens), Hq=wl.Hq, Hkv=wl.Hkv, D=wl.D, lens=lens, bits=wl.bits,
                         dtype=wl.dtype)
    got = _vals(_run(p), wl.dtype)
    rng = np.random.default_rng(5)
    pick = sorted(set([0, len(lens) - 1] + list(rng.choice(len(lens), 3, replace=False))))
    sub = synth.KVProblem(p.q[pick], p.k_codes[pick], p.k_scale[pick], p.k_zero[pick], p.v_codes[pick],
                          p.v_scale[pick], p.v_zero[pick], p.lens[pick], p.bits, p.dtype, p.sm_scale)
    _check(got[pick], _ref(sub))


def test_argument_checks():
    p = synth.kv_problem(24, B=1, Hq=4, Hkv=2, D=128, lens=[10], L_max=64)
    d = _dev(p)
    with pytest.raises(binding.TmError):
        binding.attn_decode(**{**d, "q": d["q"][:, :3]}, kv_bits=8, sm_scale=0.1)   # Hq % Hkv
    with pytest.raises(binding.TmError):
        binding.attn_decode(**d, kv_bits=6, sm_scale=0.1)
    with pytest.raises(binding.TmError):
        binding.attn_decode(**{**d, "q": d["q"][:, :, :64].contiguous()}, kv_bits=8, sm_scale=0.1)
    with pytest.raises(binding.TmError):
        binding.attn_decode(**d, kv_bits=8, sm_scale=float("inf"))
    plan = binding.attn_decode_plan(16, 32, 8, 8192, 8)
    assert plan["chunk_tiles"] >= 1 and plan["grid"] >= 1


def test_chain_with_gemms_back_to_back():
    """A GEMM writes the queries, the attention reads them and writes O, a
    second GEMM reads O: programmatic dependent launches in one stream with
    no synchronization between, eager and replayed from a CUDA graph."""
    from tests._util import bits_of, c_values, packed_from

    B, Hq, Hkv = 4, 8, 2
    p = synth.kv_problem(30, B=B, Hq=Hq, Hkv=Hkv, D=128, lens=[300, 64, 1, 129], L_max=320)
    qw1, x = synth.random_problem(44, B, 256, Hq * 128, 128, "f16")
    qw2, _ = synth.random_problem(45, 1, Hq * 128, 256, 128, "f16")
    w1 = oracle.dequant_bits(qw1.q, qw1.scales, qw1.zeros, 128, "f16")
    w2 = oracle.dequant_bits(qw2.q, qw2.scales, qw2.zeros, 128, "f16")
    W1, W2 = packed_from(qw1), packed_from(qw2)
    d = _dev(p)
    del d["q"]
    X = binding.acts_to_device(x, torch.float16)
    Qb = torch.empty((B, Hq * 128), dtype=torch.float16, device="cuda")
    O = torch.empty((B, Hq, 128), dtype=torch.float16, device="cuda")
    Y = torch.empty((B, 256), dtype=torch.float16, device="cuda")
    torch.cuda.synchronize()
    st = torch.cuda.Stream()

    def run():
        binding.gemm(X, W1, out=Qb, stream=st)
        binding.attn_decode(Qb.view(B, Hq, 128), **d, kv_bits=8, sm_scale=p.sm_scale, out=O, stream=st)
        binding.gemm(O.view(B, Hq * 128), W2, out=Y, stream=st)

    def check(what):
        assert oracle.max_err_ratio(c_values(Qb), oracle.gemm_ref(x, w1, "f16")) <= 1.0, what
        o_ref = at.attn_decode_ref(bits_of(Qb).reshape(B, Hq, 128), p.k_codes, p.k_scale, p.k_zero, p.v_codes,
                                   p.v_scale, p.v_zero, p.lens, 8, "f16", p.sm_scale)
        _check(_vals(O, "f16"), o_ref)
        y_ref = oracle.gemm_ref(bits_of(O.view(B, Hq * 128)), w2, "f16")
        assert oracle.max_err_ratio(c_values(Y), y_ref) <= 1.0, what

    with torch.cuda.stream(st):
        for _ in range(3):
            Qb.fill_(float("nan"))
            O.fill_(float("nan"))
            run()
    st.synchronize()
    binding.poll_error(st)
    check("eager")
    with torch.cuda.stream(st):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            Qb.fill_(float("nan"))
            O.fill_(float("nan"))
            run()
        Y.fill_(float("nan"))
        g.replay()
        g.replay()
    st.synchronize()
    binding.poll_error(st)
    check("graph")
