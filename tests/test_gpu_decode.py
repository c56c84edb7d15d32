"""Single-token INT4 decode kernel (FP16 operands, per-group power-of-two activation scaling)
against the float64 oracle, through qgemm_dense with M = 1.

The kernel stages each scale group of the activations as FP16 after multiplying it by the
power of two that puts the group's largest magnitude in [2^14, 2^15); the cases below cover
the group splits the launcher picks for several K, ragged N, bias and second-level scales,
and activations whose groups span many binades (tiny, huge, all-zero, subnormal entries).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import qgemm as OQ
from qwtest import dense_w4a16, dev, qw, repack, u16_view

pytestmark = pytest.mark.gpu


def assert_parity(C, R, absum, what=""):
    ok, ratio, frob = OQ.check_bf16_result(C, R, absum)
    assert ok, f"{what}: worst |err|/bound = {ratio:.3g}, rel frob = {frob:.3g}"


@pytest.mark.parametrize("bits", [4, 3, 2])
@pytest.mark.parametrize("N,K", [(1000, 512), (1032, 2048), (1000, 4096), (4104, 14336),
                                 (1032, 16384), (2056, 5120), (1000, 128), (1032, 640)])
def test_decode_shapes(bits, N, K):
    """K = 512 .. 16384 (4 to 128 groups: one to sixteen warps per CTA), N not a multiple of
    16; K = 128 and 640 have no split with whole ring batches and take the staged kernel.
    INT4 runs on FP16 operands, INT3 and INT2 on BF16 operands.  Every case has about a
    thousand outputs or more: with a few dozen, BF16 rounding of the exact result alone can
    exceed the Frobenius bound."""
    p = synth.w4a16_problem(1, N, K, bits=bits, cfg_id=700 + K // 128)
    C = dense_w4a16(p)
    R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K, bits)
    assert_parity(C, R, S, f"decode INT{bits} {N}x{K}")


def test_decode_int4_bias_and_scale2():
    Q = qw()
    N, K = 1000, 4096
    p = synth.w4a16_problem(1, N, K, bits=4, cfg_id=731, bias=True)
    wfmt = Q.QW_W_INT4_G128_BF16 | Q.QW_W_SCALE2
    d, wp, sp = repack(wfmt, 1, N, K, p["w_canon"], p["s_canon"])
    rng = np.random.default_rng(5)
    t = (2.0 ** rng.integers(-3, 4, N)).astype(np.float32)  # powers of two: exact either way
    err = Q.new_error_flag()
    Q.qw_repack_scale2(d, dev(t), sp, err)
    assert Q.qw_read_error(err) == 0
    C = torch.full((1, N), -1, dtype=torch.int16, device="cuda")
    Q.qgemm_dense(d, wp, sp, Q.QW_A_BF16, dev(p["A"].view(np.int16)), None,
                  dev(p["bias"][0].view(np.int16)), C, 1, None, 0, err)
    assert Q.qw_read_error(err) == 0
    R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K, 4)
    R2, S2 = OQ.apply_scale2(R, S, t, p["bias"][0])
    assert_parity(u16_view(C), R2, S2, "decode bias + scale2")


def _scaled_activations(K, exps, cfg):
    """N(0,1) activations with group g multiplied by 2^exps[g] (None: an all-zero group)."""
    rng = np.random.default_rng(cfg)
    a = rng.standard_normal((1, K))
    for g, e in enumerate(exps):
        a[0, g * 128:(g + 1) * 128] = 0.0 if e is None else a[0, g * 128:(g + 1) * 128] * 2.0 ** e
    return synth.to_bf16_bits(a)


@pytest.mark.parametrize("bits", [4, 3])
@pytest.mark.parametrize("exps", [
    [0, -60, 60, None, -20, 20, 100, -100],       # groups many binades apart, one all zero
    [-100] * 8,                                   # every group tiny
    [100] * 8,                                    # every group huge
])
def test_decode_group_magnitudes(bits, exps):
    """INT4's per-group power-of-two scaling keeps every group exact, whatever its
    magnitude (INT3 takes BF16 operands as they are): each output is checked against its
    own sum of |a w| (no absolute floor)."""
    N, K = 520, 128 * len(exps)
    p = synth.w4a16_problem(1, N, K, bits=bits, cfg_id=740)
    p["A"] = _scaled_activations(K, exps, 741)
    C = dense_w4a16(p)
    R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K, bits)
    c = torch.from_numpy(C.astype(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.all(np.isfinite(c))
    bad = np.abs(c - R) > 2.0 ** -7 * S
    assert not bad.any(), f"{bad.sum()} outputs outside 2^-7 sum|a w|"


def test_decode_int4_tiny_entries_below_the_group_maximum():
    """Entries 2^-30 .. 2^-40 times the group maximum (and BF16 subnormals) land on FP16
    subnormals or zero after the group scaling; their contribution stays far inside the
    tolerance."""
    N, K = 264, 1024
    p = synth.w4a16_problem(1, N, K, bits=4, cfg_id=750)
    rng = np.random.default_rng(751)
    a = rng.standard_normal((1, K))
    a[0, 1::3] *= 2.0 ** -rng.integers(30, 41, a[0, 1::3].size)
    a[0, 2::17] = 1e-39  # BF16 subnormal
    p["A"] = synth.to_bf16_bits(a)
    C = dense_w4a16(p)
    R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K, 4)
    assert_parity(C, R, S, "tiny entries")


@pytest.mark.parametrize("chained", [False, True])
def test_stream_read_reads_every_word(chained):
    """The diagnostic streaming read folds every 32-bit word it reads: the XOR of the
    per-CTA words equals the XOR of the whole buffer (any grid, any order)."""
    Q = qw()
    rng = np.random.default_rng(3)
    words = rng.integers(0, 2 ** 32, (1 << 20) + 12, dtype=np.uint64).astype(np.uint32)
    src = torch.from_numpy(words.view(np.int32)).cuda()
    sink = torch.zeros(Q.QW_STREAM_READ_SINK_WORDS, dtype=torch.int32, device="cuda")
    Q.qw_stream_read(src, words.nbytes, sink, chained)
    torch.cuda.synchronize()
    got = np.bitwise_xor.reduce(sink.cpu().numpy().view(np.uint32))
    assert got == np.bitwise_xor.reduce(words)


def _split_call(Q, wfmt, N, K, w_canon, s_canon, A, bias=None, t=None):
    d, wp, sp = repack(wfmt | (Q.QW_W_SCALE2 if t is not None else 0), 1, N, K, w_canon, s_canon)
    err = Q.new_error_flag()
    if t is not None:
        Q.qw_repack_scale2(d, dev(t), sp, err)
    C = torch.full((1, N), -1, dtype=torch.int16, device="cuda")
    b = None if bias is None else dev(bias.view(np.int16))
    Q.qgemm_dense(d, wp, sp, Q.QW_A_BF16, dev(A.view(np.int16)), None, b, C, 1, None, 0, err)
    assert Q.qw_read_error(err) == 0
    return u16_view(C)


@pytest.mark.parametrize("N,K", [(512, 16384), (1000, 32768), (200, 16384), (760, 24576)])
def test_decode_split_k_bias_scale2(N, K):
    """At most half as many 16-row blocks as SMs and K of 128 groups or more (the shapes the
    launcher splits; S = 8, 4, 8 and 6 slices here): K is split across the CTAs of a
    cluster, whose rank 0
    adds the slice sums in rank order through distributed shared memory, then applies the
    second-level scales and the bias.  Two calls give identical bits."""
    Q = qw()
    p = synth.w4a16_problem(1, N, K, bits=4, cfg_id=760 + K // 1024, bias=True)
    rng = np.random.default_rng(K + N)
    t = (2.0 ** rng.integers(-3, 4, N)).astype(np.float32)
    C1 = _split_call(Q, Q.QW_W_INT4_G128_BF16, N, K, p["w_canon"], p["s_canon"], p["A"],
                     p["bias"][0], t)
    C2 = _split_call(Q, Q.QW_W_INT4_G128_BF16, N, K, p["w_canon"], p["s_canon"], p["A"],
                     p["bias"][0], t)
    assert np.array_equal(C1, C2), "split-K results must be deterministic"
    R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K, 4)
    R2, S2 = OQ.apply_scale2(R, S, t, p["bias"][0])
    assert_parity(C1, R2, S2, f"split decode {N}x{K}")


@pytest.mark.parametrize("kind", ["int3", "int2", "int1", "fp4"])
def test_decode_split_k_formats(kind):
    """The split schedule for every format the decode kernel takes (1000 x 16384)."""
    Q = qw()
    N, K = 1000, 16384
    if kind == "fp4":
        p = synth.fp4w_problem(1, N, K, cfg_id=771)
        wfmt = Q.QW_W_FP4E2M1_G128_BF16
        R, S = OQ.fp4w_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K)
    else:
        bits = {"int3": 3, "int2": 2, "int1": 1}[kind]
        p = synth.w4a16_problem(1, N, K, bits=bits, cfg_id=772 + bits)
        wfmt = {3: Q.QW_W_INT3_G128_BF16, 2: Q.QW_W_INT2_G128_BF16,
                1: Q.QW_W_INT1_G128_BF16}[bits]
        R, S = OQ.w4a16_from_canonical(p["A"], p["w_canon"][0], p["s_canon"][0], K, bits)
    C = _split_call(Q, wfmt, N, K, p["w_canon"], p["s_canon"], p["A"])
    assert_parity(C, R, S, f"split decode {kind}")
