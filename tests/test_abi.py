"""The C-ABI library loads, exports every symbol include/qw.h declares, and rejects bad
arguments on the host (no GPU needed: validation happens before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "qw.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(q\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def Q():
    import moe_qw_repack_gb300.qw as q
    return q


def test_header_declares_the_boundary():
    fns = header_functions()
    for name in ("qw_repack", "qw_unpack", "qw_repack_query", "qgemm_dense", "qgemm_moe_grouped",
                 "qgemm_moe_route", "qgemm_moe_permute", "qgemm_workspace_size",
                 "qw_repack_scale2", "qw_unpack_scale2"):
        assert name in fns


def test_library_exports_every_declared_symbol(Q):
    lib = ctypes.CDLL(Q.lib_path())
    for name in header_functions():
        assert hasattr(lib, name), name
    assert set(header_functions()) <= set(Q.EXPORTS)


def test_binding_constants_and_descriptor_match_the_header(Q):
    """The binding's enum values, the QW_W_SCALE2 flag and the descriptor struct (field
    order and C types) are those include/qw.h declares."""
    src = open(os.path.join(ROOT, "include", "qw.h")).read()
    code = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    enums = dict((k, int(v)) for k, v in re.findall(r"\b(QW_[A-Z0-9_]+)\s*=\s*(\d+)", code))
    assert len(enums) >= 8 + 8 + 3
    for name, value in enums.items():
        assert getattr(Q, name) == value, name
    flag = re.search(r"#define\s+QW_W_SCALE2\s+(0x[0-9A-Fa-f]+)", code)
    assert flag and Q.QW_W_SCALE2 == int(flag.group(1), 16)
    body = re.search(r"typedef struct qw_packed_desc \{(.*?)\} qw_packed_desc;", code, re.S).group(1)
    fields = []
    for ctype, names in re.findall(r"(int32_t|uint64_t)\s+([^;]+);", body):
        for n in names.split(","):
            fields.append((n.strip(), ctypes.c_int32 if ctype == "int32_t" else ctypes.c_uint64))
    assert [(n, t) for n, t in Q.PackedDesc._fields_] == fields
    assert ctypes.sizeof(Q.PackedDesc) == 8 * 4 + 4 * 8


def test_status_strings(Q):
    for s in range(8):
        assert Q.status_str(s)
    assert Q.status_str(99) == "unknown status"


@pytest.mark.parametrize("wfmt,N,K,npad,kpad,wb,sb", [
    (0, 2048, 2048, 2048, 2048, 2048 * 2048 // 2, 2048 * 16 * 2),
    (0, 40, 256, 48, 256, 48 * 256 // 2, 256),  # scales padded to 256 B
    (1, 4096, 4096, 4096, 4096, 4096 * 4096 * 3 // 8, 4096 * 32 * 2),
    (2, 3072, 4096, 3072, 4096, 3072 * 2048, 3072 * 128),
    (2, 640, 96, 640, 128, 640 * 64, 640 * 4),
    (7, 14336, 4096, 14336, 4096, 14336 * 4096, 14336 * 32 * 2),  # E4M3: one byte per weight
    (7, 40, 384, 48, 384, 48 * 384, 512),
    (8, 40, 384, 48, 384, 48 * 384 // 8, 512),  # INT1: one bit per weight
    (9, 14336, 4096, 14336, 4096, 14336 * 4096 // 2, 14336 * 32 * 2),  # E2M1: half a byte
])
def test_repack_query_sizes(Q, wfmt, N, K, npad, kpad, wb, sb):
    d = Q.qw_repack_query(wfmt, 1, N, K)
    assert (d.N_pad, d.K_pad, d.w_bytes, d.s_bytes) == (npad, kpad, wb, sb)


def test_repack_query_rejects(Q):
    for args in [(0, 1, 16, 100), (1, 1, 16, 64), (2, 1, 16, 48), (10, 1, 16, 128), (0, 0, 16, 128),
                 (0, 1, 0, 128), (7, 1, 16, 64), (8, 1, 16, 96), (9, 1, 16, 64)]:
        with pytest.raises(Q.QwError):
            Q.qw_repack_query(*args)


def test_repack_query_int32_limits(Q):
    """Sizes whose padding would overflow int32 are refused; the largest accepted ones give
    padded sizes and byte counts that are exact."""
    big = 2**31 - 1
    for args in [(0, 1, big, 128), (Q.QW_W_MXFP4_G32, 1, big, 128),
                 (Q.QW_W_MXFP4_G32, 1, 128, 2**31 - 32), (Q.QW_W_NVFP4_G16, 1, 128, 2**31 - 32),
                 (0, 2, 2**30, 128)]:  # N_pad * E = 2^31
        with pytest.raises(Q.QwError):
            Q.qw_repack_query(*args)
    kmax = 2**31 - 256
    d = Q.qw_repack_query(Q.QW_W_NVFP4_G16, 1, 128, kmax)
    assert (d.N_pad, d.K_pad, d.w_bytes) == (128, kmax, 128 * kmax // 2)
    d = Q.qw_repack_query(0, 1, kmax, 128)
    assert (d.N_pad, d.w_bytes, d.s_bytes) == (kmax, kmax // 16 * 1024, kmax * 2)


def test_gemm_host_validation(Q):
    d = Q.qw_repack_query(Q.QW_W_MXFP4_G32, 1, 256, 256)
    good = 1 << 20  # fake, never dereferenced: every call below fails validation first
    with pytest.raises(Q.QwError) as e:  # wrong activation format for MXFP4 weights
        Q.qgemm_dense(d, good, good, Q.QW_A_BF16, good, None, None, good, 4, stream=0)
    assert e.value.status == Q.QW_ERR_UNSUPPORTED
    with pytest.raises(Q.QwError) as e:  # missing activation scales
        Q.qgemm_dense(d, good, good, Q.QW_A_MXFP8_G32, good, None, None, good, 4, stream=0)
    assert e.value.status == Q.QW_ERR_INVALID_ARG
    with pytest.raises(Q.QwError) as e:  # misaligned packed weights
        Q.qgemm_dense(d, good + 16, good, Q.QW_A_MXFP8_G32, good, good, None, good, 4, stream=0)
    assert e.value.status == Q.QW_ERR_ALIGNMENT
    with pytest.raises(Q.QwError) as e:  # negative M
        Q.qgemm_dense(d, good, good, Q.QW_A_MXFP8_G32, good, good, None, good, -1, stream=0)
    assert e.value.status == Q.QW_ERR_INVALID_ARG
    bad = Q.qw_repack_query(Q.QW_W_MXFP4_G32, 1, 256, 256)
    bad.N_pad = 128  # tampered descriptor
    with pytest.raises(Q.QwError) as e:
        Q.qgemm_dense(bad, good, good, Q.QW_A_MXFP8_G32, good, good, None, good, 4, stream=0)
    assert e.value.status == Q.QW_ERR_INVALID_ARG
    d2 = Q.qw_repack_query(Q.QW_W_MXFP4_G32, 8, 256, 256)
    with pytest.raises(Q.QwError) as e:  # dense call with several experts
        Q.qgemm_dense(d2, good, good, Q.QW_A_MXFP8_G32, good, good, None, good, 4, stream=0)
    assert e.value.status == Q.QW_ERR_INVALID_ARG
    with pytest.raises(Q.QwError) as e:  # grouped call without workspace
        Q.qgemm_moe_grouped(d2, good, good, Q.QW_A_MXFP8_G32, good, good, good, 100, None, good,
                            None, 0, stream=0)
    assert e.value.status == Q.QW_ERR_WORKSPACE
    # M == 0 is a valid no-op that launches nothing
    Q.qgemm_dense(d, good, good, Q.QW_A_MXFP8_G32, good, good, None, good, 0, stream=0)


def test_grouped_indexed_host_validation(Q):
    good = 1 << 20
    d = Q.qw_repack_query(Q.QW_W_MXFP4_G32, 8, 256, 256)
    cases = [  # (T, topk, total_rows, workspace bytes, expected status)
        (10, 2, 21, 1 << 20, Q.QW_ERR_INVALID_ARG),   # more rows than T * topk pairs
        (10, 0, 4, 1 << 20, Q.QW_ERR_INVALID_ARG),    # topk < 1
        (-1, 2, 0, 1 << 20, Q.QW_ERR_INVALID_ARG),    # negative T
        (10, 2, 20, 0, Q.QW_ERR_WORKSPACE),           # no workspace
    ]
    for T, k, rows, ws, want in cases:
        with pytest.raises(Q.QwError) as e:
            Q.qgemm_moe_grouped_indexed(d, good, good, Q.QW_A_MXFP8_G32, good, good, T, good, k,
                                        good, rows, None, good, good if ws else None, ws,
                                        stream=0)
        assert e.value.status == want, (T, k, rows, ws)
    di = Q.qw_repack_query(Q.QW_W_INT4_G128_BF16, 8, 256, 256)
    with pytest.raises(Q.QwError) as e:  # the indexed path takes the MX formats only
        Q.qgemm_moe_grouped_indexed(di, good, good, Q.QW_A_BF16, good, None, 10, good, 2, good,
                                    20, None, good, good, 1 << 20, stream=0)
    assert e.value.status == Q.QW_ERR_UNSUPPORTED
    # zero rows: a valid no-op
    Q.qgemm_moe_grouped_indexed(d, good, good, Q.QW_A_MXFP8_G32, good, good, 10, good, 2, good,
                                0, None, good, None, 0, stream=0)


def test_route_host_validation(Q):
    good = 1 << 20
    for T, E, k in [(-1, 8, 2), (4, 8, 0), (4, 8, 33), (4, 4, 8), (4, 2048, 8)]:
        with pytest.raises(Q.QwError) as e:
            Q.qgemm_moe_route(good, T, E, k, good, good, good, good, 1 << 30, stream=0)
        assert e.value.status == Q.QW_ERR_INVALID_ARG
    with pytest.raises(Q.QwError) as e:
        Q.qgemm_moe_route(good, 4, 8, 2, good, good, good, good, 0, stream=0)
    assert e.value.status == Q.QW_ERR_WORKSPACE
    assert Q.qgemm_moe_route_workspace_size(4096, 256, 8) == 128 * 256 * 4


def test_permute_host_validation(Q):
    good = 1 << 20
    with pytest.raises(Q.QwError) as e:  # BF16 row of 12 bytes is not 16-byte aligned
        Q.qgemm_moe_permute(Q.QW_A_BF16, good, None, 6, good, 4, 2, good, None, stream=0)
    assert e.value.status == Q.QW_ERR_ALIGNMENT
    Q.qgemm_moe_permute(Q.QW_A_BF16, good, None, 64, good, 0, 2, good, None, stream=0)  # P == 0


def test_timeout_probe_validation(Q):
    with pytest.raises(Q.QwError):
        Q.qw_test_wait_timeout(None, 1000, stream=0)
    with pytest.raises(Q.QwError):
        Q.qw_test_wait_timeout(1 << 20, 3_000_000_000, stream=0)


def test_activation_steps_host_validation(Q):
    good = 1 << 20
    for K, status in [(48, Q.QW_ERR_UNSUPPORTED), (16, Q.QW_ERR_INVALID_ARG)]:
        with pytest.raises(Q.QwError) as e:
            Q.qw_quantize_mxfp8(good, 4, K, good, good, stream=0)
        assert e.value.status == status
    with pytest.raises(Q.QwError) as e:  # A not 16-byte aligned
        Q.qw_quantize_mxfp8(good + 8, 4, 64, good, good, stream=0)
    assert e.value.status == Q.QW_ERR_ALIGNMENT
    Q.qw_quantize_mxfp8(good, 0, 64, good, good, stream=0)  # no rows: a no-op
    with pytest.raises(Q.QwError) as e:
        Q.qw_silu_mul(good, 4, 12, good, stream=0)
    assert e.value.status == Q.QW_ERR_UNSUPPORTED
    with pytest.raises(Q.QwError) as e:
        Q.qw_silu_mul(good, 4, 64, good + 4, stream=0)
    assert e.value.status == Q.QW_ERR_ALIGNMENT
    assert Q.qgemm_moe_combine_workspace_size(4096, 8) == 4096 * 8 * 4 + 256
    for T, E, k, N, status in [(4, 8, 0, 64, Q.QW_ERR_INVALID_ARG), (4, 8, 9, 64, Q.QW_ERR_INVALID_ARG),
                               (4, 8, 2, 12, Q.QW_ERR_UNSUPPORTED)]:
        with pytest.raises(Q.QwError) as e:
            Q.qgemm_moe_combine(good, good, good, good, T, E, k, N, good, good, 1 << 20, stream=0)
        assert e.value.status == status
    with pytest.raises(Q.QwError) as e:
        Q.qgemm_moe_combine(good, good, good, good, 4, 8, 2, 64, good, good, 8, stream=0)
    assert e.value.status == Q.QW_ERR_WORKSPACE


def test_scale2_flag_sizes_and_host_validation(Q):
    """The second-level scale plane adds FP32 [E][N_pad] (rounded to 256 bytes) to s_bytes;
    unknown flag bits are rejected; the scale2 entry points want the flag (host checks only)."""
    for wfmt in (Q.QW_W_INT4_G128_BF16, Q.QW_W_MXFP4_G32, Q.QW_W_NVFP4_G16, Q.QW_W_FP8E4M3_G128_BF16):
        base = Q.qw_repack_query(wfmt, 3, 200, 512)
        d = Q.qw_repack_query(wfmt | Q.QW_W_SCALE2, 3, 200, 512)
        assert d.wfmt == wfmt | Q.QW_W_SCALE2 and d.N_pad == base.N_pad
        assert d.s_expert_stride == base.s_expert_stride and d.w_bytes == base.w_bytes
        assert d.s_bytes == base.s_bytes + (3 * base.N_pad * 4 + 255) // 256 * 256
    with pytest.raises(Q.QwError):
        Q.qw_repack_query(0x200, 1, 16, 128)
    plain = Q.qw_repack_query(Q.QW_W_INT4_G128_BF16, 1, 16, 128)
    good = 1 << 20
    for call in (lambda: Q.qw_repack_scale2(plain, good, good, stream=0),
                 lambda: Q.qw_unpack_scale2(plain, good, good, stream=0)):
        with pytest.raises(Q.QwError) as e:
            call()
        assert e.value.status == Q.QW_ERR_INVALID_ARG


def test_stream_read_validates_on_the_host(Q):
    """The diagnostic streaming read rejects a missing sink and unaligned sizes or
    addresses before launching anything; its sink length is the header's."""
    src = open(os.path.join(ROOT, "include", "qw.h")).read()
    m = re.search(r"#define\s+QW_STREAM_READ_SINK_WORDS\s+(\d+)", src)
    assert m and Q.QW_STREAM_READ_SINK_WORDS == int(m.group(1))
    fake = 1 << 20  # never dereferenced
    assert Q.LIB.qw_stream_read(fake, 64, None, 0, None) == Q.QW_ERR_INVALID_ARG
    assert Q.LIB.qw_stream_read(fake, 40, fake, 0, None) == Q.QW_ERR_ALIGNMENT
    assert Q.LIB.qw_stream_read(fake + 8, 64, fake, 0, None) == Q.QW_ERR_ALIGNMENT


def test_grouped_workspace_covers_every_smaller_call(Q):
    """A workspace sized for max_rows serves every grouped call of at most max_rows rows:
    the size never decreases as max_rows grows, across the switches of the GEMV's token
    tile (8 -> 16 rows at 8 rows per expert) and of the tensor-core path (16 rows per
    expert), for the W4A16 and W4A8 formats."""
    for wfmt, afmt in ((Q.QW_W_INT4_G128_BF16, Q.QW_A_BF16), (Q.QW_W_INT3_G128_BF16, Q.QW_A_BF16),
                       (Q.QW_W_MXFP4_G32, Q.QW_A_MXFP8_G32)):
        for E in (8, 128):
            d = Q.qw_repack_query(wfmt, E, 1280, 4096)
            prev = 0
            for rows in range(0, 40 * E + 1, max(1, E // 16)):
                n = Q.qgemm_workspace_size(d, afmt, rows)
                assert n >= prev, (wfmt, E, rows, n, prev)
                prev = n


def test_binding_fails_loudly_without_the_library(tmp_path):
    """No fallback: with the shared library absent, importing the binding raises ImportError
    naming the missing file (run in a fresh interpreter so this process keeps its library)."""
    import subprocess
    import sys
    missing = tmp_path / "libqw.so"
    code = ("import moe_qw_repack_gb300.build as b; b.LIB = %r\n"
            "try:\n"
            "    import moe_qw_repack_gb300.qw\n"
            "except ImportError as e:\n"
            "    print('IMPORT-ERROR', e)\n"
            "else:\n"
            "    print('LOADED')\n" % str(missing))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       timeout=300)
    assert "IMPORT-ERROR" in r.stdout and str(missing) in r.stdout, r.stdout + r.stderr


def test_mma_rate_probe_validates_on_the_host(Q):
    """The MMA-rate diagnostic takes only the shapes the GEMMs issue; nothing launches."""
    out = ctypes.c_void_p(64)
    err = ctypes.c_void_p(64)
    bad = [(16, 256, 4096), (24, 256, 4096), (32, 128, 4096), (-1, 128, 4096),  # unknown mode
           (Q.QW_MMA_PROBE_RANDOM | 16, 128, 4096), (Q.QW_MMA_PROBE_MXF4NVF4, 128, 4096),
           (Q.QW_MMA_PROBE_MXF4NVF4_CP | Q.QW_MMA_PROBE_RANDOM, 64, 4096),
           (Q.QW_MMA_PROBE_F16_TMEM_A, 96, 4096), (Q.QW_MMA_PROBE_F16_SMEM, 512, 4096),
           (Q.QW_MMA_PROBE_MXF8F6F4, 128, 4096), (Q.QW_MMA_PROBE_MXF8F6F4_CP, 64, 4096),
           (Q.QW_MMA_PROBE_MXF8F6F4_CP_AHEAD, 128, 4096),
           (Q.QW_MMA_PROBE_MXF8F6F4_CP_WIDE | Q.QW_MMA_PROBE_RANDOM, 64, 4096),
           (Q.QW_MMA_PROBE_F16_SMEM, 128, 63), (Q.QW_MMA_PROBE_F16_SMEM, 128, (1 << 20) + 1)]
    for mode, n, iters in bad:
        assert Q.LIB.qw_mma_rate_probe(mode, n, iters, out, err, None) == Q.QW_ERR_INVALID_ARG
    assert Q.LIB.qw_mma_rate_probe(0, 128, 4096, None, err, None) == Q.QW_ERR_INVALID_ARG
    assert Q.LIB.qw_mma_rate_probe(0, 128, 4096, out, None, None) == Q.QW_ERR_INVALID_ARG
    assert Q.LIB.qw_mma_rate_probe(0, 128, 4096, ctypes.c_void_p(68), err, None) == \
        Q.QW_ERR_ALIGNMENT
