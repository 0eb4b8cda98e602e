"""CPU-side checks of the C ABI: the library loads, exports every declared entry point,
and its host logic (descriptor validation, sizes, argument errors) behaves as documented.
No test here launches a kernel."""
import ctypes
import os
import re

import pytest

import quantized_weight_gemm_gb300 as qg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    with open(os.path.join(ROOT, "include", "qgemm.h"), encoding="utf-8") as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return set(re.findall(r"\b(qgemm_[a-z0-9_]+)\s*\(", text))


@pytest.fixture(scope="module")
def L():
    from quantized_weight_gemm_gb300 import build
    build.build()
    return qg.lib()


def test_exports_match_header(L):
    declared = _declared_functions()
    assert declared == set(qg.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings(L):
    for s in range(10):
        assert L.qgemm_status_str(s)
    assert L.qgemm_version() >= 100


@pytest.mark.parametrize("wfmt,group,afmt,ok", [
    ("int4_sym", 128, "bf16", True), ("uint4_zp", 128, "bf16", True),
    ("int4_sym", 32, "bf16", True), ("uint4_zp", 64, "bf16", True),
    ("mxfp4", 32, "bf16", True), ("mxfp4", 32, "fp8", True),
    ("int4_sym", 48, "bf16", False), ("mxfp4", 64, "bf16", False),
    ("int4_sym", 128, "fp8", False),
    ("mxint4", 32, "bf16", True), ("nvfp4", 16, "bf16", True),
    ("mxint4", 64, "bf16", False), ("nvfp4", 32, "bf16", False),
    ("mxint4", 32, "fp8", False), ("nvfp4", 16, "fp8", False),
    ("mxfp4", 32, "fp8n", True), ("uint4_zp", 128, "fp8n", False), ("mxint4", 32, "fp8n", False),
])
def test_check_desc(L, wfmt, group, afmt, ok):
    d = qg.WeightDesc(wfmt, 256, 512, group, afmt)
    assert (qg.check_desc(d) == 0) == ok


def test_packed_bytes_accounting(L):
    # INT4 asym 28672 x 8192, group 128: codes + scales + packed uint4 zero points
    d = qg.WeightDesc("uint4_zp", 28672, 8192, 128)
    n = qg.packed_bytes(d)
    codes, scales, zeros = 28672 * 8192 // 2, 28672 * 64 * 2, 28672 * 64 // 2
    assert n >= codes + scales + zeros
    assert n - (codes + scales + zeros) < 4096
    assert n % 256 == 0
    # MXFP4 4096 x 7168: codes + one E8M0 byte per 32
    d = qg.WeightDesc("mxfp4", 4096, 7168, 32)
    assert qg.packed_bytes(d) - (4096 * 7168 // 2 + 4096 * 7168 // 32) < 4096
    # ragged N and K pad to the tile
    d = qg.WeightDesc("int4_sym", 130, 96, 32)
    assert qg.packed_bytes(d) >= 256 * 128 // 2
    # MXINT4 packs like MXFP4; NVFP4: codes + one E4M3 byte per 16
    assert qg.packed_bytes(qg.WeightDesc("mxint4", 4096, 7168, 32)) == \
        qg.packed_bytes(qg.WeightDesc("mxfp4", 4096, 7168, 32))
    n = qg.packed_bytes(qg.WeightDesc("nvfp4", 4096, 7168, 16))
    assert 0 <= n - (4096 * 7168 // 2 + 4096 * 7168 // 16) < 4096


def test_batch_invariant_plan(L):
    """QGEMM_FLAG_BATCH_INVARIANT: one schedule for every M (128-token tiles, no cut, no
    stream-K, so no workspace); other flag bits are invalid."""
    d = qg.WeightDesc("uint4_zp", 28672, 8192, 128, batch_invariant=True)
    assert qg.check_desc(d) == 0
    for M in (1, 16, 100, 1000, 8192):
        p = qg.plan(d, M)
        assert (p["token_tile"], p["splits"], p["sk_tiles"], p["max_contrib"]) == (128, 1, 0, 0)
        assert p["grid"] == min(-(-M // 128) * 224, 152)
    # nothing is cut: the workspace is just the FP16 activation copy of INT4 with BF16 scales
    assert qg.workspace_bytes(d, 8192) == qg.act_copy_bytes(d, 8192)
    raw = qg.WeightDesc("uint4_zp", 256, 512, 128).c()
    raw.flags = 2
    assert L.qgemm_check_desc(ctypes.byref(raw)) != 0
    assert L.qgemm_packed_bytes(ctypes.byref(raw)) == 0


def test_repack_scaled_argument_errors(L):
    """The per-tensor scale belongs to NVFP4 and must be finite; checked before any launch."""
    P = ctypes.c_void_p
    buf = P(1 << 20)                       # never dereferenced: the calls fail first
    for wfmt, group, g, want in [("mxfp4", 32, 2.0, 2), ("int4_sym", 128, 0.5, 2),
                                 ("nvfp4", 16, float("nan"), 1), ("nvfp4", 16, float("inf"), 1),
                                 ("nvfp4", 16, 3.0e38, 1)]:
        d = qg.WeightDesc(wfmt, 256, 512, group).c()
        st = L.qgemm_repack_scaled(ctypes.byref(d), buf, buf, None, ctypes.c_float(g), buf, None)
        assert st == want, (wfmt, g, st)


def test_bad_descriptors_give_zero(L):
    for d in [qg.WeightDesc("int4_sym", 0, 512), qg.WeightDesc("int4_sym", 16, 500),
              qg.WeightDesc("int4_sym", 16, 512, 100)]:
        assert L.qgemm_packed_bytes(ctypes.byref(d.c())) == 0


def test_workspace_bytes(L):
    d = qg.WeightDesc("uint4_zp", 28672, 8192, 128)
    assert qg.workspace_bytes(d, 1) > 0                # decode-sized M splits K
    big = qg.workspace_bytes(d, 8192)
    assert big >= qg.workspace_bytes(d, 1)
    assert big < 256 * 1024 * 1024


def test_argument_errors_before_any_launch(L):
    d = qg.WeightDesc("int4_sym", 256, 512, 128).c()
    P = ctypes.c_void_p
    # null X, null packed, negative M, ldx < K, misaligned X
    assert L.qgemm_w4a16(ctypes.byref(d), None, P(256), 16, 512, None, None, P(256), 256, None, 0, None) == 1
    assert L.qgemm_w4a16(ctypes.byref(d), P(256), None, 16, 512, None, None, P(256), 256, None, 0, None) == 1
    assert L.qgemm_w4a16(ctypes.byref(d), P(256), P(256), -1, 512, None, None, P(256), 256, None, 0, None) == 1
    assert L.qgemm_w4a16(ctypes.byref(d), P(256), P(256), 16, 256, None, None, P(256), 256, None, 0, None) == 1
    assert L.qgemm_w4a16(ctypes.byref(d), P(256), P(258), 16, 512, None, None, P(256), 256, None, 0, None) == 3
    assert L.qgemm_w4a16(ctypes.byref(d), P(256), P(256), 16, 516, None, None, P(256), 256, None, 0, None) == 3
    # misaligned bias
    assert L.qgemm_w4a16(ctypes.byref(d), P(256), P(256), 16, 512, None, P(258), P(256), 256, None, 0,
                         None) == 3
    # M = 0 is a no-op (returns before touching any device)
    assert L.qgemm_w4a16(ctypes.byref(d), P(256), P(256), 0, 512, None, None, P(256), 256, None, 0, None) == 0
    # FP8 entry point with a BF16-activation descriptor
    assert L.qgemm_w4a8(ctypes.byref(d), P(256), P(256), 4, 512, P(256), None, None, P(256), 256, None, 0, None) == 1
    assert L.qgemm_force_config(48, 0) == 1
    assert L.qgemm_force_config(0, -2) == 1
    assert L.qgemm_force_config(0, 0) == 0


def test_host_staging_bytes(L):
    """Staging of the host-buffer call: two X and two Y chunk buffers; chunks are all rows up
    to 512, else M/16 rounded up to 256 rows (at least 512), so the size never shrinks as M
    grows (a buffer sized for M_max serves every smaller M)."""
    d = qg.WeightDesc("uint4_zp", 8192, 28672, 128)
    K, N = 28672, 8192

    def rows(M):
        if M <= 512:
            return M
        return max(512, -(-(-(-M // 16)) // 256) * 256)

    def rup(v):
        return -(-v // 256) * 256

    prev = 0
    for M in (1, 2, 100, 511, 512, 513, 1000, 4096, 8191, 8192, 8193, 20000):
        n = qg.host_staging_bytes(d, M)
        r = rows(M)
        assert n == 2 * (rup(r * K * 2) + rup(r * N * 2)), M
        assert n >= prev
        prev = n
    assert qg.host_staging_bytes(d, 0) == 0
    assert qg.host_staging_bytes(qg.WeightDesc("int4_sym", 0, 512), 16) == 0


def test_moe_argument_errors_before_any_launch(L):
    """The MoE calls check their arguments on the host, before any device is touched."""
    P = ctypes.c_void_p
    d = qg.WeightDesc("mxfp4", 256, 512, 32).c()
    bf16, fp8 = 0, 1
    buf, off = P(1 << 20), P(1 << 21)

    def grouped(E=4, afmt=bf16, X=buf, R=8, ldx=512, ts=None, offs=off, Y=buf, ldy=256, packed=buf,
                bias=None):
        return L.qgemm_moe_grouped(ctypes.byref(d), packed, E, afmt, X, R, ldx, ts, bias, offs, Y,
                                   ldy, None, 0, None)

    def indexed(T=8, R=8, idx=P(1 << 22), E=4):
        return L.qgemm_moe_indexed(ctypes.byref(d), buf, E, bf16, buf, T, 512, None, None, off, idx,
                                   R, buf, 256, None, 0, None)

    assert grouped(E=0) == 1 and grouped(E=1025) == 1           # expert count
    assert grouped(afmt=fp8) == 1                                # descriptor is BF16
    assert grouped(R=-1) == 1 and grouped(offs=None) == 1 and grouped(packed=None) == 1
    assert grouped(packed=P((1 << 20) + 16)) == 3                # packed not 256-byte aligned
    assert grouped(offs=P((1 << 21) + 2)) == 3                   # offsets not 4-byte aligned
    assert grouped(bias=P((1 << 21) + 2)) == 3                   # bias not 4-byte aligned
    assert grouped(ldx=256) == 1                                 # ldx < K
    assert grouped(X=P((1 << 20) + 2)) == 3                      # X not 16-byte aligned
    assert grouped(ldy=128) == 1                                 # ldy < N
    assert grouped(R=0) == 0                                     # empty: a no-op
    assert indexed(T=0) == 1                                     # rows to gather from none
    assert indexed(idx=P((1 << 22) + 2)) == 3                    # index not 4-byte aligned
    assert indexed(R=0) == 0
    d8 = qg.WeightDesc("mxfp4", 256, 512, 32, "fp8").c()
    assert L.qgemm_moe_grouped(ctypes.byref(d8), buf, 4, fp8, buf, 8, 512, None, None, off, buf,
                               256, None, 0, None) == 1          # FP8 without token scales


def test_product_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "quantized_weight_gemm_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "oracle" not in text.replace("the oracle", ""), f


def _sk_contributors(T, kb, P):
    """Stream-K as the header defines it, walked record by record: CTA i takes records
    [floor(i S / P), floor((i + 1) S / P)) of the S = T kb records of the cut tiles."""
    S = T * kb
    owners = [set() for _ in range(T)]
    covered = 0
    for i in range(P):
        lo, hi = i * S // P, (i + 1) * S // P
        for x in range(lo, hi):
            owners[x // kb].add(i)
        covered += hi - lo
    assert covered == S
    if S >= P:
        # every CTA holds a record: a tile's owners are consecutive CTAs, and contributor j
        # of tile t uses partial-sum slot t + min(owners) + j
        for o in owners:
            assert o == set(range(min(o), max(o) + 1))
        top = max(t + min(o) + len(o) - 1 for t, o in enumerate(owners))
        assert top < T + P
    else:
        # at most one record per CTA: kb owners per tile, a record's slot is its index (< S)
        assert all(len(o) == kb for o in owners)
    return max(len(o) for o in owners)


@pytest.mark.parametrize("N,K,M,tt", [(28672, 1152, 16, 16), (28672, 8192, 100, 16),
                                      (8192, 28672, 16, 16), (4096, 7168, 1, 16),
                                      (384, 1024, 100, 16), (7168, 2048, 48, 16),
                                      (384, 1024, 100, 32), (384, 1024, 150, 32),
                                      (6400, 256, 16, 16), (19968, 512, 16, 16)])
def test_stream_k_plan(L, N, K, M, tt):
    """The forced stream-K plan of the dense path: leftover tiles = T mod P (all T when
    T < P), and partial-sum slots = the most CTAs whose record ranges meet one tile (also
    when the cut tiles hold fewer records than there are CTAs)."""
    d = qg.WeightDesc("uint4_zp", N, K, 128)
    P = 152
    qg.force_config(tt, -1)
    try:
        p = qg.plan(d, M)
        ws = qg.workspace_bytes(d, M)
    finally:
        qg.force_config(0, 0)
    T = -(-M // tt) * -(-N // 128)
    kb = -(-K // 128)
    sk = T if T < P else T % P
    assert p["token_tile"] == tt and p["splits"] == 1 and p["grid"] == P
    assert p["sk_tiles"] == sk
    c = _sk_contributors(sk, kb, P)
    assert p["max_contrib"] == (c if c > 1 else 0)
    if c > 1:
        assert ws >= (sk + P) * 128 * tt * 4 + 4 * sk


def test_default_plans_match_the_contributor_model(L):
    """Over a grid of shapes, every default plan that cuts tiles agrees with the record-walk
    model of stream-K (leftover tiles, contributors per tile, at most 8 unforced), uniform
    cuts keep at least two K blocks per part, and a workspace sized for M covers the plan."""
    P = 152
    for N in (128, 384, 4096, 19968, 28672):
        for K in (128, 256, 512, 1024, 8192):
            d = qg.WeightDesc("uint4_zp", N, K, 128)
            kb = -(-K // 128)
            for M in (1, 2, 7, 16, 33, 100, 300, 1024):
                p = qg.plan(d, M)
                tt = p["token_tile"]
                T = -(-M // tt) * -(-N // 128)
                assert 1 <= p["grid"] <= P
                if p["sk_tiles"] > 0:
                    assert p["splits"] == 1
                    assert p["sk_tiles"] == (T if T < P else T % P), (N, K, M, p)
                    c = _sk_contributors(p["sk_tiles"], kb, P)
                    assert p["max_contrib"] == (c if c > 1 else 0), (N, K, M, p, c)
                    assert c <= 8
                    if c > 1:
                        need = (p["sk_tiles"] + p["grid"]) * 128 * tt * 4
                        assert qg.workspace_bytes(d, M) >= need
                elif p["splits"] > 1:
                    assert kb // p["splits"] >= 2
                    assert qg.workspace_bytes(d, M) >= T * p["splits"] * 128 * tt * 4


def test_large_m_stream_k_plans_and_workspace(L):
    """Above M = 1024, stream-K is planned only for K >= 16384 (128 blocks), agrees with the
    record-walk model, and a workspace sized for M_max covers the plan of every M <= M_max."""
    P = 152
    for (N, K) in [(8192, 28672), (4096, 16384), (28672, 8192), (4096, 7168)]:
        d = qg.WeightDesc("uint4_zp", N, K, 128)
        kb = -(-K // 128)
        copy = qg.act_copy_bytes(d, 4096)
        ws = qg.workspace_bytes(d, 4096)
        seen = 0
        for M in range(1025, 4097, 7):
            p = qg.plan(d, M)
            if kb < 128:
                assert p["sk_tiles"] == 0 and p["splits"] == 1, (N, K, M, p)
                continue
            assert p["splits"] == 1
            if p["sk_tiles"] > 0:
                seen += 1
                tt = p["token_tile"]
                T = -(-M // tt) * -(-N // 128)
                assert p["sk_tiles"] == T % P
                c = _sk_contributors(p["sk_tiles"], kb, P)
                assert p["max_contrib"] == (c if c > 1 else 0) and c <= 8
                assert ws - copy >= (p["sk_tiles"] + p["grid"]) * 128 * tt * 4 + 4 * p["sk_tiles"]
        assert kb < 128 or seen > 0


def test_plan_defaults_are_valid(L):
    for (N, K) in [(28672, 8192), (8192, 28672), (4096, 7168), (7168, 2048)]:
        d = qg.WeightDesc("uint4_zp", N, K, 128)
        for M in (1, 16, 64, 256, 1024, 8192):
            p = qg.plan(d, M)
            assert p["token_tile"] in (16, 32, 64, 128, 256)
            assert p["splits"] >= 1 and 0 < p["grid"] <= 152
            assert p["sk_tiles"] == 0 or p["splits"] == 1
            assert (p["max_contrib"] > 0) == (p["splits"] > 1 or p["sk_tiles"] > 0)
            assert qg.workspace_bytes(d, M) >= (4 if p["max_contrib"] else 0)


def test_moe_workspace_bytes(L):
    d = qg.WeightDesc("mxfp4", 4096, 7168, 32)
    # 16-row tiles, counters rounded up to 256 B; narrow MXFP4 tiles also hold the FP16
    # activation copy of the 8 rows (7168 x 2 bytes each, then 8 row scales, each part
    # rounded up to 256 B) that lets them run on FP16 operands
    copy8 = 8 * 7168 * 2 + 256
    assert qg.moe_workspace_bytes(d, 256, 8) == 2 * 152 * 128 * 16 * 4 + 768 + copy8
    # 128-token tiles up to 192 rows per expert, 256-token tiles above
    assert qg.moe_workspace_bytes(d, 8, 8 * 150) == 2 * 152 * 128 * 128 * 4 + 768
    assert qg.moe_workspace_bytes(d, 8, 8 * 200) == 2 * 152 * 128 * 256 * 4 + 768
    assert qg.moe_workspace_bytes(d, 0, 8) == 0
    assert qg.moe_workspace_bytes(d, 8, 0) == 0


def test_moe_indexed_workspace_holds_the_copy_from_256_rows(L):
    """The indexed MoE call gathers its rows into the workspace from 256 sorted rows on: the
    workspace it asks for grows by exactly the sorted copy of the rows and their scales
    there, and not below."""
    d = qg.WeightDesc("mxfp4", 4096, 7168, 32)
    for fp8, esz in ((False, 2), (True, 1)):
        dd = qg.WeightDesc("mxfp4", 4096, 7168, 32, afmt="fp8") if fp8 else d
        below = qg.moe_indexed_workspace_bytes(dd, 256, 40, 255, fp8=fp8)
        at = qg.moe_indexed_workspace_bytes(dd, 256, 40, 256, fp8=fp8)
        copy = -(-256 * 7168 * esz // 256) * 256 + -(-256 * 4 // 256) * 256
        assert at - below == copy, (fp8, at, below)
        assert qg.moe_indexed_workspace_bytes(dd, 256, 40, 200, fp8=fp8) == below


def test_act_copy_bytes():
    """INT4 with BF16 scales runs on FP16 operands: the workspace leads with an FP16 copy of
    X ([rows][K], 256-byte rounded) and one FP32 row scale per row (256-byte rounded); no
    other layout has one."""
    for wfmt, group in [("int4_sym", 128), ("uint4_zp", 64), ("int4_sym", 32)]:
        d = qg.WeightDesc(wfmt, 1000, 4096, group)
        for rows in (1, 3, 100, 8192):
            want = -(-rows * 4096 * 2 // 256) * 256 + -(-rows * 4 // 256) * 256
            assert qg.act_copy_bytes(d, rows) == want
        assert qg.act_copy_bytes(d, 0) == 0
        assert qg.workspace_bytes(d, 8192) >= qg.act_copy_bytes(d, 8192)
        assert qg.moe_workspace_bytes(d, 8, 1000) > qg.act_copy_bytes(d, 1000)
    for wfmt, group, afmt in [("mxfp4", 32, "bf16"), ("mxint4", 32, "bf16"), ("nvfp4", 16, "bf16"),
                              ("mxfp4", 32, "fp8")]:
        d = qg.WeightDesc(wfmt, 1000, 4096, group, afmt)
        assert qg.act_copy_bytes(d, 100) == 0


def test_w4a4_argument_errors_before_any_launch(L):
    """W4A4 descriptors pair MXFP4 weights with MXFP4 activations only; the GEMM and the
    activation quantization check their arguments on the host first."""
    P = ctypes.c_void_p
    assert qg.check_desc(qg.WeightDesc("mxfp4", 256, 512, 32, "mxfp4")) == 0
    assert qg.check_desc(qg.WeightDesc("uint4_zp", 256, 512, 128, "mxfp4")) != 0
    assert qg.check_desc(qg.WeightDesc("nvfp4", 256, 512, 16, "mxfp4")) != 0
    d = qg.WeightDesc("mxfp4", 256, 512, 32, "mxfp4").c()
    buf, ex = P(1 << 20), P(1 << 21)

    def w4a4(packed=buf, X=buf, M=8, ldq=256, E=ex, lde=16, Y=buf, ldy=256, desc=d):
        return L.qgemm_w4a4(ctypes.byref(desc), packed, X, M, ldq, E, lde, None, None, Y, ldy,
                            None, 0, None)

    assert w4a4(M=-1) == 1 and w4a4(E=None) == 1 and w4a4(packed=None) == 1
    assert w4a4(ldq=240) == 1                       # ldq < K / 2
    assert w4a4(lde=12) == 1                        # lde < ceil(K / 128) * 4
    assert w4a4(X=P((1 << 20) + 8)) == 3            # codes not 16-byte aligned
    assert w4a4(E=P((1 << 21) + 8)) == 3            # exponents not 16-byte aligned
    assert w4a4(lde=24) == 3                        # exponent rows not a multiple of 16
    assert w4a4(M=0) == 0
    bf = qg.WeightDesc("mxfp4", 256, 512, 32, "bf16").c()
    assert w4a4(desc=bf) == 1                       # a BF16-activation packing
    q = L.qgemm_quant_act_mxfp4
    assert q(buf, 4, 500, 512, buf, 256, ex, 16, None) == 1     # K % 32 != 0
    assert q(buf, 4, 512, 512, buf, 255, ex, 16, None) == 1     # ldq < K / 2
    assert q(buf, 4, 512, 512, buf, 256, ex, 15, None) == 1     # lde too small
    assert q(buf, 0, 512, 512, buf, 256, ex, 16, None) == 0     # empty: a no-op
