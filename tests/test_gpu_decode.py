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
