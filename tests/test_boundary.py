"""C ABI boundary checks that need no GPU: the library loads, exports every
function declared in include/*.h, and rejects bad arguments synchronously
(before touching CUDA) with the documented status codes."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def declared_functions():
    names = set()
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(kda_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("kda_fwd", "kda_fwd_ws", "kda_workspace_size", "kda_device_status",
              "kda_status_string", "kda_last_error_message", "kda_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(kda_lib):
    L = ctypes.CDLL(kda_lib.library_path())
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, f"not exported: {missing}"
    assert L.kda_abi_version() == 1


def call(kda_lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, scale=0.088, out=FAKE, A_log=FAKE,
             dt_bias=FAKE, lb=-5.0, h0=None, h0d=0, hT=None, hTd=0, cu=None, ns=0, B=1, T=64,
             H=2, K=128, V=128)
    a.update(over)
    L = kda_lib.lib()
    rc = L.kda_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["out"], a["A_log"],
                   a["dt_bias"], a["lb"], a["h0"], a["h0d"], a["hT"], a["hTd"], a["cu"], a["ns"],
                   a["B"], a["T"], a["H"], a["K"], a["V"], None)
    return rc, L.kda_last_error_message().decode()


@pytest.mark.parametrize("over,code", [
    (dict(K=64), 1), (dict(V=256), 1), (dict(H=0), 1), (dict(T=-1), 1), (dict(B=0), 1),
    (dict(B=2, cu=FAKE, ns=2), 1),                        # cu_seqlens needs B == 1
    (dict(h0=FAKE, h0d=1, hT=FAKE + (1 << 24), hTd=2), 1),  # state dtypes differ
    (dict(h0=FAKE, h0d=3), 1),                            # bad dtype code
    (dict(h0=FAKE, h0d=0), 1),                            # pointer without dtype
    (dict(h0=None, h0d=2), 1),                            # dtype without pointer
    (dict(lb=0.5), 1), (dict(lb=float("nan")), 1), (dict(lb=float("-inf")), 1),
    (dict(lb=-10.5), 2),                                  # outside the supported range
    (dict(scale=float("inf")), 1),
    (dict(q=None), 1), (dict(out=None), 1), (dict(A_log=None), 1),
    (dict(q=FAKE + 8), 1),                                # misaligned
    (dict(h0=FAKE, h0d=2, hT=FAKE + 4096, hTd=2), 1),     # partial overlap of the states
    (dict(cu=FAKE + 2, ns=1), 1),                         # misaligned cu_seqlens
    (dict(cu=FAKE, ns=-1), 1),
])
def test_invalid_arguments_rejected(kda_lib, over, code):
    rc, msg = call(kda_lib, **over)
    assert rc == code, (rc, msg)
    assert msg


def test_status_strings(kda_lib):
    L = kda_lib.lib()
    assert L.kda_status_string(0) == b"KDA_OK"
    assert L.kda_status_string(2) == b"KDA_ERR_UNSUPPORTED"
    assert L.kda_status_string(99) == b"KDA_ERR_UNKNOWN"


def test_workspace_size(kda_lib):
    L = kda_lib.lib()
    rec = 82432
    # dense: N * ceil(T/64) chunks bound = (B*T + 63 B) / 64
    n = L.kda_workspace_size(8, 2048, 16, 0, 0)
    assert n >= 8 * 32 * 16 * rec
    assert n < 8 * 33 * 16 * rec + 1 << 20
    assert L.kda_workspace_size(2, 64, 1, 3, 1) == 0   # cu_seqlens needs B == 1
    assert L.kda_workspace_size(1, 100, 2, 3, 1) > 0


def test_stage_events_validation(kda_lib):
    L = kda_lib.lib()
    assert L.kda_set_stage_events(None, 0) == 0
    arr = (ctypes.c_void_p * 3)()
    assert L.kda_set_stage_events(arr, 3) == 1
    arr6 = (ctypes.c_void_p * 6)()
    assert L.kda_set_stage_events(arr6, 6) == 1   # null events
    assert L.kda_set_stage_events(arr6, 5) == 1   # count neither 4 nor 6
    assert L.kda_set_stage_events(None, 0) == 0


def test_workspace_size_follows_segmented_selection(kda_lib):
    """Few long sequences take the segmented path (automatically or forced): the
    workspace adds the segment offsets and 3 fp32 128x128 tiles per (segment, head)
    for 4..32 segments per sequence; the other kernels need none of it."""
    L = kda_lib.lib()
    try:
        kda_lib.set_recurrence_kernel("sliced")
        base = L.kda_workspace_size(1, 65536, 4, 0, 0)
        kda_lib.set_recurrence_kernel("auto")
        auto = L.kda_workspace_size(1, 65536, 4, 0, 0)
        kda_lib.set_recurrence_kernel("segmented")
        forced = L.kda_workspace_size(1, 65536, 4, 0, 0)
        # four one-chunk sequences: no segment area under automatic selection, 2 segments forced
        forced_short = L.kda_workspace_size(1, 64 * 4, 4, 4, 1)
        kda_lib.set_recurrence_kernel("auto")
        auto_short = L.kda_workspace_size(1, 64 * 4, 4, 4, 1)
    finally:
        kda_lib.set_recurrence_kernel("auto")

    def area(P, N=1, H=4):
        return ((N * P + 1) * 4 + 255) // 256 * 256 + N * P * H * 3 * 128 * 128 * 4

    assert auto == forced
    assert any(auto - base == area(P) for P in range(4, 33)), auto - base
    assert auto_short < forced_short
    assert forced_short - auto_short == area(2, N=4)


def test_recurrence_selection_validation(kda_lib):
    L = ctypes.CDLL(kda_lib.library_path())
    L.kda_set_recurrence_kernel.argtypes = [ctypes.c_int32]
    for kind in (-1, 5, 99):
        assert L.kda_set_recurrence_kernel(kind) == 1  # KDA_ERR_INVALID_ARGUMENT
    for kind in (4, 3, 2, 1, 0):
        assert L.kda_set_recurrence_kernel(kind) == 0
    with pytest.raises(ValueError):
        kda_lib.set_recurrence_kernel("bogus")
    # no forward pass has run on this thread
    assert L.kda_last_path() == 0 and kda_lib.last_path() is None


def test_python_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import gated_delta_rule_30_gb300 as kda
    monkeypatch.setattr(kda, "_lib", None)
    monkeypatch.setattr(kda, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        kda.lib()


def test_fwd_ex_rejects_unknown_flags(kda_lib):
    """kda_fwd_ex: flag bits other than KDA_FWD_QK_L2NORM are an argument error,
    and its other arguments are validated like kda_fwd's (nothing launched)."""
    L = kda_lib.lib()

    def ex(flags, K=128):
        rc = L.kda_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 0.088, FAKE, FAKE, FAKE, -5.0, None, 0,
                          None, 0, None, 0, 1, 64, 2, K, 128, flags, None, 0, None)
        return rc, L.kda_last_error_message().decode()

    for bad in (2, 4, 0x80000000, 3):
        rc, msg = ex(bad)
        assert rc == 1 and "flag" in msg, (bad, rc, msg)
    rc, msg = ex(1, K=64)   # a valid flag does not skip the shape checks
    assert rc == 1 and "128" in msg


def test_workspace_size_single_token_step(kda_lib):
    """Single-token problems take the step that uses no scratch: the answer is the
    minimum (256 bytes) under automatic selection, the chunked size otherwise."""
    L = kda_lib.lib()
    try:
        kda_lib.set_recurrence_kernel("auto")
        assert L.kda_workspace_size(1024, 1, 32, 0, 0) == 256
        assert L.kda_workspace_size(1, 1024, 32, 1024, 1) > 256   # packed: chunked path
        kda_lib.set_recurrence_kernel("transposed")
        assert L.kda_workspace_size(1024, 1, 32, 0, 0) > 64 << 20
    finally:
        kda_lib.set_recurrence_kernel("auto")


def call_bwd(kda_lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, scale=0.088, A_log=FAKE, dt_bias=FAKE,
             lb=-5.0, h0=None, h0d=0, dout=FAKE, dhT=None, cu=None, ns=0, B=1, T=64, H=2, K=128,
             V=128, dq=FAKE, dk=FAKE, dv=FAKE, dg=FAKE, dbeta=FAKE, dA=FAKE, ddt=FAKE, dh0=None,
             flags=0, ws=FAKE, wsb=0)
    a.update(over)
    L = kda_lib.lib()
    rc = L.kda_bwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["A_log"],
                   a["dt_bias"], a["lb"], a["h0"], a["h0d"], a["dout"], a["dhT"], a["cu"], a["ns"],
                   a["B"], a["T"], a["H"], a["K"], a["V"], a["dq"], a["dk"], a["dv"], a["dg"],
                   a["dbeta"], a["dA"], a["ddt"], a["dh0"], a["flags"], a["ws"], a["wsb"], None)
    return rc, L.kda_last_error_message().decode()


@pytest.mark.parametrize("over", [
    dict(K=64), dict(V=64), dict(H=0), dict(T=-1), dict(B=0), dict(B=2, cu=FAKE, ns=2),
    dict(h0=FAKE, h0d=3), dict(h0=FAKE, h0d=0), dict(h0=None, h0d=2),
    dict(lb=0.5), dict(lb=float("nan")), dict(scale=float("nan")),
    dict(dout=None), dict(dq=None), dict(dA=None), dict(ddt=None), dict(A_log=None),
    dict(dout=FAKE + 8), dict(dv=FAKE + 4), dict(dbeta=FAKE + 2), dict(dhT=FAKE + 8),
    dict(dh0=FAKE + 8), dict(cu=FAKE + 2, ns=1), dict(cu=FAKE, ns=-1),
    dict(wsb=1),                      # caller workspace smaller than kda_bwd_workspace_size
    dict(flags=4), dict(flags=0x80000000),  # unknown flag bits
    dict(flags=2),                    # low memory: the workspace (0 bytes) is too small
])
def test_bwd_invalid_arguments_rejected(kda_lib, over):
    rc, msg = call_bwd(kda_lib, **over)
    assert rc == 1, (rc, msg)
    assert msg


def test_bwd_workspace_size(kda_lib):
    """Per-pair partial sums plus two fp32 states (128 x 128) per head for each of
    floor(total / 16) + N + 1 checkpoint slots (states entering tokens 0 and 8)."""
    L = kda_lib.lib()
    n = L.kda_bwd_workspace_size(8, 2048, 16, 0, 0, 0)
    slots = 8 * 2048 // 16 + 8 + 1
    ckpt = slots * 16 * 2 * 128 * 128 * 4
    assert ckpt <= n <= ckpt + 8 * 16 * (4 + 128) * 4 + 512
    assert L.kda_bwd_workspace_size(2, 64, 1, 3, 1, 0) == 0
    assert L.kda_bwd_workspace_size(1, 100, 2, 3, 1, 0) > 0
    assert L.kda_bwd_workspace_size(1, 100, 2, 3, 1, 4) == 0   # unknown flag bit
    # low memory: one state per 64 tokens, plus 256 replay slots of 8 states
    lo = L.kda_bwd_workspace_size(8, 2048, 16, 0, 0, 2)
    slots64 = 8 * 2048 // 64 + 8 + 1
    ckpt64 = slots64 * 16 * 128 * 128 * 4
    replay = 256 * 8 * 32 * 128 * 4
    assert ckpt64 + replay <= lo <= ckpt64 + replay + 8 * 16 * (4 + 128) * 4 + 2048
    long_ctx = L.kda_bwd_workspace_size(1, 65536, 32, 0, 0, 0)
    assert L.kda_bwd_workspace_size(1, 65536, 32, 0, 0, 2) * 7 < long_ctx
