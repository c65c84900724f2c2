"""Host-side tests of the C ABI: the library builds, loads and exports every
declared entry point; argument checks return the documented codes without
touching a GPU; workspace sizes follow the documented layout."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def L():
    from io_aware_exact_05_gb300 import attn
    from io_aware_exact_05_gb300.build import build

    if not os.path.exists(attn.lib_path()):
        build()
    return attn.lib()


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", txt)))


def test_header_declares_entry_points():
    names = _declared()
    for n in ("attn_fwd", "attn_bwd", "attn_fwd_gqa", "attn_bwd_gqa", "attn_bwd_workspace_size",
              "attn_status",
              "attn_strerror", "attn_mat_fwd", "attn_mat_bwd", "attn_gemm_bf16"):
        assert n in names


def test_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_strerror_and_version(L):
    from io_aware_exact_05_gb300 import attn

    assert attn.attn_strerror(0) == "success"
    for c in range(1, 6):
        assert attn.attn_strerror(c) not in ("", "unknown status code")
    assert attn.attn_strerror(99) == "unknown status code"
    assert "sm_103a" in attn.attn_version()


FAKE = ctypes.c_void_p(1 << 20)          # aligned, never dereferenced
MIS = ctypes.c_void_p((1 << 20) + 8)     # misaligned


def _fwd(L, *, p=FAKE, B=1, H=1, n=128, d=64, dt=0, scale=0.125, causal=0):
    return L.attn_fwd(p, FAKE, FAKE, FAKE, FAKE, B, H, n, d, dt, scale, causal, None)


def test_fwd_argument_checks(L):
    assert _fwd(L, p=ctypes.c_void_p(0)) == 1
    assert _fwd(L, p=MIS) == 1
    assert _fwd(L, B=0) == 1
    assert _fwd(L, n=0) == 1
    assert _fwd(L, d=0) == 1
    assert _fwd(L, causal=2) == 1
    assert _fwd(L, scale=float("nan")) == 1
    assert _fwd(L, n=65535 * 128 + 1) == 2     # 128-row tiles map to a 65535-wide grid dimension
    assert _fwd(L, scale=float("inf")) == 1
    assert _fwd(L, dt=7) == 1
    assert _fwd(L, d=96) == 2                # bf16 head dims are 64, 128, 256
    assert _fwd(L, d=512, dt=1) == 2         # fp32 path: d <= 256
    assert _fwd(L, B=300, H=300) == 2        # B*H beyond the grid's head axis


def _ws(L, B, H, n, d, dt, causal, mode):
    return L.attn_bwd_workspace_size(B, H, n, d, dt, causal, mode)


def _rup(x, a=256):
    return (x + a - 1) // a * a


def test_workspace_sizes(L):
    B, H, n, d = 2, 3, 1000, 128
    BH, n_pad = B * H, 1024
    stats = 2 * _rup(BH * n_pad * 4)
    assert _ws(L, B, H, n, d, 0, 1, 1) == stats + _rup(BH * n * d * 4)   # atomic
    assert _ws(L, B, H, n, d, 0, 1, 2) == stats                          # pass
    assert _ws(L, B, H, n, d, 0, 1, 0) == _ws(L, B, H, n, d, 0, 1, 1)    # auto = atomic
    assert _ws(L, B, H, n, 256, 0, 1, 0) == stats                        # d=256 causal: pass
    assert _ws(L, B, H, n, 256, 0, 0, 2) == stats
    assert _ws(L, B, H, n, 256, 0, 0, 0) == stats + _rup(BH * n * 1000 * 2)   # spill: dS^T
    assert _ws(L, B, H, n, 256, 0, 0, 1) == 0                            # not supported
    assert _ws(L, B, H, n, 100, 1, 0, 0) == _rup(BH * n * 4)             # fp32: D only
    assert _ws(L, B, H, n, 96, 0, 0, 0) == 0
    assert _ws(L, 0, H, n, d, 0, 0, 0) == 0
    # materialise-P: S/dP fp32 + P/dS bf16 + D + LSE2
    nn = BH * 1024 * 1024
    assert L.attn_mat_workspace_size(B, H, 1024, 64) == (
        _rup(nn * 4) + _rup(nn * 2) + 2 * _rup(BH * 1024 * 4))
    assert L.attn_mat_workspace_size(B, H, 1001, 64) == 0               # n % 8 != 0


def test_bwd_argument_checks(L):
    ws = ctypes.c_void_p(1 << 24)
    args = [FAKE] * 9

    def call(*, d=128, dt=0, mode=0, wsb=1 << 30, wsp=ws, scale=0.1):
        return L.attn_bwd(*args, 1, 2, 256, d, dt, scale, 1, mode, wsp, wsb, None)

    assert call(mode=9) == 1
    assert call(d=96) == 2
    assert call(d=256, mode=1) == 2
    assert call(wsb=16) == 3                       # workspace too small
    assert call(wsp=ctypes.c_void_p(0)) == 3       # no workspace
    assert call(wsp=ctypes.c_void_p((1 << 24) + 16)) == 3   # not 256-byte aligned
    assert call(scale=float("nan")) == 1
    bad = [FAKE] * 8 + [ctypes.c_void_p(0)]
    assert L.attn_bwd(*bad, 1, 2, 256, 128, 0, 0.1, 1, 0, ws, 1 << 30, None) == 1


def test_backward_stage_argument_checks(L):
    """attn_bwd_preprocess / attn_bwd_dkdv / attn_bwd_dq check like attn_bwd,
    before any launch, and a rejected call enqueues nothing."""
    ws = ctypes.c_void_p(1 << 24)
    before = L.attn_launch_count()

    def pre(*, d=128, dt=0, mode=0, wsb=1 << 30, wsp=ws, causal=1, ptr=FAKE):
        return L.attn_bwd_preprocess(ptr, FAKE, FAKE, 1, 2, 256, d, dt, causal, mode, wsp, wsb,
                                     None)

    def kv(*, d=128, dt=0, mode=0, wsb=1 << 30, wsp=ws, scale=0.1, ptr=FAKE):
        return L.attn_bwd_dkdv(ptr, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, d, dt, scale, 1,
                               mode, wsp, wsb, None)

    def dq(*, d=128, dt=0, mode=0, wsb=1 << 30, wsp=ws, scale=0.1, ptr=FAKE, qptr=FAKE):
        # ptr: dQ (always used); qptr: Q (read only by the dQ pass)
        return L.attn_bwd_dq(qptr, FAKE, FAKE, FAKE, ptr, 1, 2, 256, d, dt, scale, 1, mode, wsp,
                             wsb, None)

    for f in (pre, kv, dq):
        assert f(ptr=ctypes.c_void_p(0)) == 1                 # null tensor
        assert f(ptr=ctypes.c_void_p((1 << 20) + 8)) == 1     # not 16-byte aligned
        assert f(mode=9) == 1
        assert f(dt=5) == 1
        assert f(d=96) == 2                                   # bf16 head dims: 64, 128, 256
        assert f(d=256, mode=1) == 2                          # atomic dQ needs d <= 128
        assert f(dt=1, d=300) == 2                            # fp32: d <= 256
        assert f(wsb=16) == 3
        assert f(wsp=ctypes.c_void_p(0)) == 3
        assert f(wsp=ctypes.c_void_p((1 << 24) + 16)) == 3    # not 256-byte aligned
    assert pre(causal=2) == 1
    assert kv(scale=float("inf")) == 1 and dq(scale=float("nan")) == 1
    assert dq(mode=2, qptr=ctypes.c_void_p(0)) == 1          # the dQ pass reads Q
    assert dq(dt=1) == 1 and kv(dt=1) == 1                   # fp32: attn_bwd only
    assert L.attn_launch_count() == before


def test_key_rows_study_argument_checks(L):
    """attn_bwd_dkdv_keys checks like attn_bwd_dkdv, plus the key tile size
    and the dQ mode its instances exist for; nothing is launched."""
    ws = ctypes.c_void_p(1 << 24)
    before = L.attn_launch_count()

    def kv(*, d=128, dt=0, mode=0, rows=64, wsb=1 << 30, ptr=FAKE):
        return L.attn_bwd_dkdv_keys(ptr, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, d, dt, 0.1, 0,
                                    mode, rows, ws, wsb, None)

    for rows in (0, 16, 48, 96, 256):
        assert kv(rows=rows) == 1
    assert kv(ptr=ctypes.c_void_p(0)) == 1
    assert kv(dt=1) == 1                                   # bf16 only
    assert kv(d=96) == 2
    assert kv(mode=2) == 2 and kv(d=64, mode=2) == 2       # d <= 128: atomic dQ only
    assert kv(d=256, mode=1) == 2                          # d = 256: the dQ pass only
    assert kv(wsb=16) == 3
    assert L.attn_launch_count() == before


def test_dq_spill_mode_checks(L):
    """ATTN_DQ_SPILL (3): d = 256, non-causal, dense, one key/value head per
    query head; its workspace adds a bf16 n x round_up(n, 8) dS^T per head."""
    ws = ctypes.c_void_p(1 << 24)
    B, H, n = 1, 2, 300
    pas = L.attn_bwd_workspace_size(B, H, n, 256, 0, 0, 2)
    spill = L.attn_bwd_workspace_size(B, H, n, 256, 0, 0, 3)
    ld = (n + 7) // 8 * 8
    assert spill >= pas + B * H * n * ld * 2 and spill - pas < B * H * n * ld * 2 + 512
    assert L.attn_bwd_workspace_size(B, H, n, 256, 0, 1, 3) == 0      # causal
    # the automatic mode: spill where it applies and its buffer is <= 4 GiB
    assert L.attn_bwd_workspace_size(B, H, n, 256, 0, 0, 0) == spill
    assert L.attn_bwd_workspace_size(B, H, n, 256, 0, 1, 0) == L.attn_bwd_workspace_size(B, H, n, 256, 0, 1, 2)
    assert L.attn_bwd_workspace_size(16, 8, 32768, 256, 0, 0, 0) == \
        L.attn_bwd_workspace_size(16, 8, 32768, 256, 0, 0, 2)             # 274 GB: the pass
    assert L.attn_bwd_gqa_workspace_size(B, 4, 2, n, 256, 0, 0, 0) == \
        L.attn_bwd_gqa_workspace_size(B, 4, 2, n, 256, 0, 0, 2)
    lists = L.attn_bwd_sparse_workspace_size(B, H, n, 256, 0, 0, 2) - pas
    assert L.attn_bwd_sparse_workspace_size(B, H, n, 256, 0, 0, 0) == pas + lists
    assert L.attn_bwd_workspace_size(B, H, n, 128, 0, 0, 3) == 0      # d <= 128
    assert L.attn_bwd_workspace_size(B, H, n, 256, 1, 0, 3) == 0      # fp32
    assert L.attn_bwd_gqa_workspace_size(B, 4, 2, n, 256, 0, 0, 3) == 0
    before = L.attn_launch_count()

    def bwd(*, d=256, causal=0, mode=3, dt=0):
        return L.attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, H, n, d, dt,
                          0.1, causal, mode, ws, 1 << 30, None)

    assert bwd(causal=1) == 2 and bwd(d=128) == 2 and bwd(dt=1) == 2
    assert bwd(mode=4) == 1
    assert L.attn_bwd_gqa(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, 4, 2, n, 256, 0,
                          0.1, 0, 3, ws, 1 << 30, None) == 2
    assert L.attn_bwd_sparse(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, H, n, 256, 0,
                             0.1, 0, 3, FAKE, ws, 1 << 30, None) == 2
    assert L.attn_launch_count() == before


def test_gqa_argument_checks(L):
    def fwd(H=4, Hkv=2, d=64):
        return L.attn_fwd_gqa(FAKE, FAKE, FAKE, FAKE, FAKE, 1, H, Hkv, 128, d, 0, 0.125, 0, None)

    assert fwd(Hkv=3) == 1       # does not divide H
    assert fwd(Hkv=0) == 1
    assert fwd(Hkv=8) == 1       # more key/value heads than query heads
    assert fwd(d=96) == 2
    ws = ctypes.c_void_p(1 << 24)
    assert L.attn_bwd_gqa(*([FAKE] * 9), 1, 4, 3, 256, 128, 0, 0.1, 1, 0, ws, 1 << 30, None) == 1
    assert L.attn_bwd_gqa(*([FAKE] * 9), 1, 4, 2, 256, 96, 0, 0.1, 1, 0, ws, 1 << 30, None) == 2
    assert L.attn_bwd_gqa_workspace_size(1, 4, 3, 256, 128, 0, 1, 0) == 0
    mha = L.attn_bwd_workspace_size(2, 16, 8192, 128, 0, 1, 0)
    assert L.attn_bwd_gqa_workspace_size(2, 16, 16, 8192, 128, 0, 1, 0) == mha
    assert L.attn_bwd_gqa_workspace_size(2, 16, 4, 8192, 128, 0, 1, 0) == mha   # no split needed
    # one key/value head for 32 query heads at n = 4096: the group is split, and the
    # fp32 dK and dV accumulators (2 x 4096 x 128 x 4 bytes) are added
    mqa = L.attn_bwd_gqa_workspace_size(1, 32, 1, 4096, 128, 0, 1, 0)
    assert mqa == L.attn_bwd_workspace_size(1, 32, 4096, 128, 0, 1, 0) + 2 * 4096 * 128 * 4


def test_sparse_argument_checks(L):
    ws = ctypes.c_void_p(1 << 24)
    # null block mask
    assert L.attn_fwd_sparse(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, 128, 0, 0.1, 0, None, ws,
                             1 << 20, None) == 1
    # list workspace too small
    assert L.attn_fwd_sparse(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, 128, 0, 0.1, 0, FAKE, ws,
                             16, None) == 3
    assert L.attn_fwd_sparse_workspace_size(0, 128) == 0
    assert L.attn_fwd_sparse_workspace_size(256, 128) > 0
    dense = L.attn_bwd_workspace_size(1, 2, 4096, 128, 0, 1, 0)
    assert L.attn_bwd_sparse_workspace_size(1, 2, 4096, 128, 0, 1, 0) > dense
    assert L.attn_bwd_sparse(*([FAKE] * 9), 1, 2, 256, 128, 0, 0.1, 1, 0, None, ws, 1 << 30,
                             None) == 1


def test_fp8_argument_checks(L):
    MIS4 = ctypes.c_void_p((1 << 20) + 2)

    def call(d=128, n=256, scale=0.1, dsq=None, q=FAKE, causal=0):
        return L.attn_fwd_fp8(q, FAKE, FAKE, FAKE, FAKE, 1, 2, n, d, scale, dsq, FAKE, None,
                              causal, None)
    assert call(d=64) == 2
    assert call(n=100) == 2
    assert call(scale=float("nan")) == 1
    assert call(causal=3) == 1
    assert call(dsq=MIS4) == 1
    assert call(q=MIS) == 1
    assert call(q=ctypes.c_void_p(0)) == 1


def test_quantize_fp8_argument_checks(L):
    MIS4 = ctypes.c_void_p((1 << 20) + 2)
    ws = L.attn_quantize_fp8_workspace_size(4, 1000, 128)
    assert ws == 4 * 8 * 4                              # one float per 128-row block
    assert L.attn_quantize_fp8_workspace_size(4, 1000, 64) == 0

    def call(n=1024, d=128, tr=0, signs=None, x=FAKE, desc=FAKE, ws_p=FAKE, ws_b=ws):
        return L.attn_quantize_fp8(x, FAKE, desc, 4, n, d, tr, signs, ws_p, ws_b, None)
    assert call(d=64) == 2
    assert call(n=1000, tr=1) == 2                      # transposed rows of n bytes
    assert call(tr=1, signs=FAKE) == 1                  # V is never rotated
    assert call(tr=2) == 1
    assert call(n=0) == 1
    assert call(x=MIS) == 1
    assert call(desc=ctypes.c_void_p(0)) == 1
    assert call(desc=MIS4) == 1
    assert call(signs=MIS4) == 1
    assert call(ws_p=ctypes.c_void_p(0)) == 3
    assert call(ws_b=ws - 1) == 3


def test_selftest_argument_checks(L):
    assert L.attn_selftest_wait_timeout(0, None) == 1          # below 1 us
    assert L.attn_selftest_wait_timeout(10**11, None) == 1     # above 10 s


def test_gemm_argument_checks(L):
    g = L.attn_gemm_bf16
    assert g(FAKE, FAKE, FAKE, 1, 128, 128, 60, 1, 1, 1, 1.0, None) == 2   # K % 8
    assert g(FAKE, FAKE, FAKE, 1, 100, 128, 64, 0, 1, 1, 1.0, None) == 2   # MN-major A, M % 8
    assert g(FAKE, FAKE, FAKE, 1, 128, 100, 64, 1, 0, 1, 1.0, None) == 2   # MN-major B, N % 8
    assert g(FAKE, FAKE, FAKE, 0, 128, 128, 64, 1, 1, 1, 1.0, None) == 1
    assert g(ctypes.c_void_p(0), FAKE, FAKE, 1, 128, 128, 64, 1, 1, 1, 1.0, None) == 1


def test_flop_counts():
    from io_aware_exact_05_gb300.flops import attention_flops

    f = attention_flops(2, 16, 8192, 128, causal=True)
    assert f["fwd"] == 4 * 2 * 16 * 8192 ** 2 * 128 // 2
    assert f["bwd"] == 10 * 2 * 16 * 8192 ** 2 * 128 // 2
    assert abs(f["bwd"] / 1e12 - 1.374) < 1e-3


def test_kept_entries_counts_the_pattern():
    # the FLOP count of a block pattern: brute-force count of kept (i, j) pairs
    import numpy as np

    from io_aware_exact_05_gb300.flops import kept_entries

    rng = np.random.default_rng(3)
    for n, causal in ((300, False), (300, True), (129, True), (520, False)):
        nb = (n + 127) // 128
        m = rng.random((nb, nb)) < 0.5
        i = np.arange(n)[:, None]
        j = np.arange(n)[None, :]
        keep = m[i // 128, j // 128] & ((j <= i) if causal else True)
        assert kept_entries(m, n, causal) == int(keep.sum())


def test_io_study_summary_sums_backward_launches(tmp_path, capsys):
    # two synthetic ncu CSVs: the fused file's backward is every launch after
    # fwd_tc_kernel, the materialise file's every launch after three
    from io_aware_exact_05_gb300 import io_study

    hdr = '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",' \
          '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",' \
          '"Metric Value"\n'

    def write(path, launches):
        with open(path, "w") as f:
            f.write(hdr)
            for i, (name, dr, dw, l2) in enumerate(launches):
                for m, v in (("dram__bytes_read.sum", dr), ("dram__bytes_write.sum", dw),
                             ("lts__t_bytes.sum", l2)):
                    f.write('"%d","1","p","h","void unnamed>::%s<1, 2>(int)","1","7","(1, 1, 1)",'
                            '"(1, 1, 1)","0","10.3","","%s","byte","%d"\n' % (i, name, m, v))

    fused = tmp_path / "io_fused_n2048_d64.csv"
    mat = tmp_path / "io_mat_n2048_d64.csv"
    write(fused, [("fwd_tc_kernel", 7, 7, 7), ("delta_kernel", 1, 2, 30), ("bwd_kv_kernel", 3, 4, 50)])
    write(mat, [("gemm_bf16_kernel", 9, 9, 9), ("mat_softmax_kernel", 9, 9, 9),
                ("gemm_bf16_kernel", 9, 9, 9), ("gemm_bf16_kernel", 5e6, 5e6, 1e7)])
    io_study.main(["summarize", str(fused), str(mat)])
    line = [l for l in capsys.readouterr().out.splitlines() if l.startswith("| 2048 |")][0]
    cells = [c.strip() for c in line.strip("|").split("|")]
    assert cells[2] == "0.0" and cells[3] == "0.0"        # 10 bytes, 80 bytes in MB
    assert cells[4] == "10.0" and cells[5] == "10.0"      # materialise backward: 1e7 bytes each
