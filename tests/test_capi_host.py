"""Host-side tests of the C ABI: the library builds and loads without a GPU, exports every
function include/attn_gb300.h declares, and rejects invalid arguments before launching
anything (no CUDA call is reached in these tests)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def capi():
    from attention_flash_attn_gb300 import build as b
    b.build()
    from attention_flash_attn_gb300 import _capi
    return _capi


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[\w\s\*]+?\b(attn_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_function(capi):
    names = declared_functions()
    assert names, "no declarations found"
    L = capi.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(capi.EXPORTS) == names


def valid_args(capi, dtype=1, B=1, S=16, H=2, D=64, **kw):
    a = capi.AttnArgs()
    a.dtype, a.B, a.Sq, a.Sk, a.Hq, a.Hkv, a.D = dtype, B, S, S, H, H, D
    fake = 0x10000  # never dereferenced: only validation runs in these tests
    a.q = a.k = a.v = fake
    a.q_stride_b = a.k_stride_b = a.v_stride_b = S * H * D
    a.q_stride_s = a.k_stride_s = a.v_stride_s = H * D
    a.q_stride_h = a.k_stride_h = a.v_stride_h = D
    a.scale = D ** -0.5
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,status", [
    ("dtype", 3, 1), ("Hq", 3, 1), ("Hkv", 0, 1), ("D", 60, 1), ("D", 520, 2),
    ("softcap", -1.0, 1), ("softcap", float("nan"), 1), ("softcap", float("inf"), 1),
    ("scale", float("inf"), 1), ("q", None, 1), ("q", 0x10008, 1), ("q_stride_s", 12, 1),
    ("Sq", -1, 1), ("seg_q", 0x20000, 1), ("softmax_type", 2, 1), ("softmax_type", -1, 1),
    ("kv_splits", -1, 1), ("kv_splits", 65, 1),
])
def test_invalid_arguments_rejected_before_launch(capi, field, value, status):
    L = capi.lib()
    a = valid_args(capi, **{field: value})
    assert L.attn_fwd_workspace_size(ctypes.byref(a)) == 0
    assert L.attn_fwd(ctypes.byref(a), 0x30000, 0x40000, 0x50000, 1 << 20, None) == status
    n = L.attn_launch_counter()
    assert L.attn_bwd(ctypes.byref(a), 0x30000, 0x40000, 0x30000, 0x30000, 0x30000, 0x30000,
                      None, None, 0x50000, 1 << 20, None) == status
    assert L.attn_launch_counter() == n
    assert L.attn_path_name(ctypes.byref(a)) == b""


def test_off_by_one_softmax_arguments(capi):
    """The off-by-one column replaces the sink array: valid alone, invalid with a sink; its
    backward takes no dsink (there is no sink array to differentiate)."""
    L = capi.lib()
    a = valid_args(capi, softmax_type=capi.ATTN_SOFTMAX_OFF_BY_ONE)
    assert L.attn_fwd_workspace_size(ctypes.byref(a)) >= 256
    assert L.attn_bwd_workspace_size(ctypes.byref(a)) >= 256
    need = L.attn_bwd_workspace_size(ctypes.byref(a))
    n = L.attn_launch_counter()
    assert L.attn_bwd(ctypes.byref(a), 0x30000, 0x40000, 0x30000, 0x30000, 0x30000, 0x30000,
                      None, 0x60000, 0x50000, need, None) == 1
    assert L.attn_launch_counter() == n
    a = valid_args(capi, softmax_type=capi.ATTN_SOFTMAX_OFF_BY_ONE, sink=0x60000)
    assert L.attn_fwd_workspace_size(ctypes.byref(a)) == 0
    assert L.attn_fwd(ctypes.byref(a), 0x30000, 0x40000, 0x50000, 1 << 20, None) == 1


def test_kv_splits_workspace(capi):
    """A split-KV forward adds n * B * Hq * Sq * (D + 1) floats of partials to the forward's
    workspace (tensor-core path: bf16 without a bias); the backward's is unchanged, and the
    FFMA path (fp32) computes unsplit."""
    L = capi.lib()
    ws = lambda **kw: L.attn_fwd_workspace_size(ctypes.byref(valid_args(capi, S=100, **kw)))
    base = ws()
    for n in (2, 7, 64):
        assert ws(kv_splits=n) >= base + n * 1 * 2 * 100 * (64 + 1) * 4
    assert ws(kv_splits=1) == base
    bw = lambda **kw: L.attn_bwd_workspace_size(ctypes.byref(valid_args(capi, S=100, **kw)))
    assert bw(kv_splits=7) == bw()
    f32 = lambda **kw: L.attn_fwd_workspace_size(ctypes.byref(valid_args(capi, dtype=2, S=100, **kw)))
    assert f32(kv_splits=7) == f32()


def test_backward_workspace_regions(capi):
    """The backward's workspace: a 256-byte status word, then 256-byte-aligned regions for D
    (fp32 per padded query row, rows padded to 128), LSE*log2(e) and the fp32 dQ accumulator
    on the tensor-core path, and -- for its one-pass form (head dim 64 or 128), which starts
    dP^T at -D -- one 16-byte row of -D's bf16 parts per padded query row."""
    L = capi.lib()
    up = lambda x: (x + 255) // 256 * 256
    B, S, H = 1, 100, 2
    rows = B * H * 128  # Sq = 100 padded to 128
    bw = lambda **kw: L.attn_bwd_workspace_size(ctypes.byref(valid_args(capi, B=B, S=S, H=H, **kw)))
    for D in (64, 128):  # one-pass form
        assert bw(D=D) == 256 + up(rows * 4) * 2 + up(rows * 16) + up(B * S * H * D * 4)
    assert bw(D=256) == 256 + up(rows * 4) * 2 + up(B * S * H * 256 * 4)  # two-pass form
    assert bw(D=64, dtype=2) == 256 + up(rows * 4)  # fp32: FFMA kernels, D only


def test_cu_seqlens_with_segments_unsupported_and_shape_rules(capi):
    L = capi.lib()
    # separate key boundaries: need cu_seqlens; lift the Sq == Sk rule; B stays 1
    a = valid_args(capi, cu_seqlens_k=0x22000, nseq=2)
    assert L.attn_fwd(ctypes.byref(a), 0x30000, 0x40000, 0x50000, 1 << 20, None) == 1
    a = valid_args(capi, cu_seqlens=0x21000, cu_seqlens_k=0x22000, nseq=2)
    a.Sk = 40
    assert L.attn_fwd_workspace_size(ctypes.byref(a)) >= 256
    a.Sk = 16
    a.Sq = 40
    assert L.attn_fwd_workspace_size(ctypes.byref(a)) >= 256
    a = valid_args(capi, B=2, cu_seqlens=0x21000, cu_seqlens_k=0x22000, nseq=2)
    assert L.attn_fwd_workspace_size(ctypes.byref(a)) == 0
    a = valid_args(capi, cu_seqlens=0x21000, nseq=2)
    a.Sk = 40
    assert L.attn_fwd_workspace_size(ctypes.byref(a)) == 0
    a = valid_args(capi, seg_q=0x20000, seg_k=0x20000, cu_seqlens=0x21000, nseq=2)
    assert L.attn_fwd(ctypes.byref(a), 0x30000, 0x40000, 0x50000, 1 << 20, None) == 2
    a = valid_args(capi, B=2, cu_seqlens=0x21000, nseq=2)
    assert L.attn_fwd(ctypes.byref(a), 0x30000, 0x40000, 0x50000, 1 << 20, None) == 1


def test_missing_outputs_and_workspace(capi):
    L = capi.lib()
    a = valid_args(capi)
    need = L.attn_fwd_workspace_size(ctypes.byref(a))
    assert need >= 256 and need % 256 == 0
    assert L.attn_fwd(ctypes.byref(a), None, 0x40000, 0x50000, need, None) == 1
    assert L.attn_fwd(ctypes.byref(a), 0x30000, 0x40000, None, need, None) == 3
    assert L.attn_fwd(ctypes.byref(a), 0x30000, 0x40000, 0x50000, need - 1, None) == 3
    assert L.attn_fwd(ctypes.byref(a), 0x30000, 0x40000, 0x50010, need, None) == 3
    # dbias required iff bias; dsink iff sink
    a = valid_args(capi, sink=0x60000)
    nb = L.attn_bwd_workspace_size(ctypes.byref(a))
    assert L.attn_bwd(ctypes.byref(a), 0x30000, 0x40000, 0x30000, 0x30000, 0x30000, 0x30000,
                      None, None, 0x50000, nb, None) == 1
    a = valid_args(capi, bias=0x70000)
    assert L.attn_bwd(ctypes.byref(a), 0x30000, 0x40000, 0x30000, 0x30000, 0x30000, 0x30000,
                      None, None, 0x50000, 1 << 30, None) == 1


def test_empty_problem_is_a_no_op(capi):
    L = capi.lib()
    for kw in ({"B": 0}, {"Sq": 0}):
        a = valid_args(capi, **kw)
        n = L.attn_launch_counter()
        assert L.attn_fwd(ctypes.byref(a), 0x30000, 0x40000, 0x50000, 1 << 20, None) == 0
        assert L.attn_launch_counter() == n


def test_workspace_grows_with_backward_needs(capi):
    L = capi.lib()
    a = valid_args(capi, S=4096, H=8, D=128)
    f = L.attn_fwd_workspace_size(ctypes.byref(a))
    b = L.attn_bwd_workspace_size(ctypes.byref(a))
    assert b >= f + 4 * 8 * 4096  # at least D = rowsum(dO*O)
    a2 = valid_args(capi, S=4096, H=8, D=128, seg_q=0x20000, seg_k=0x20000)
    assert L.attn_fwd_workspace_size(ctypes.byref(a2)) > f


def test_status_strings(capi):
    L = capi.lib()
    for s in range(7):
        assert L.attn_status_string(s)


def test_noalloc_answers_like_attn_fwd_before_its_size_limit(capi):
    """attn_fwd_noalloc makes attn_fwd's checks first, in attn_fwd's order: invalid arguments
    and missing or misaligned outputs are ATTN_ERR_INVALID even when the request would also
    exceed its 4 MiB array, and a problem without query rows is ATTN_OK whatever its key axis
    would need.  None of these reaches a CUDA call."""
    L = capi.lib()
    S = 1 << 20  # per-token key metadata alone needs more than 4 MiB
    a = valid_args(capi, S=S, H=1, cu_seqlens=0x21000, cu_seqlens_k=0x22000, nseq=1)
    assert L.attn_fwd_workspace_size(ctypes.byref(a)) > (4 << 20)
    n = L.attn_launch_counter()
    assert L.attn_fwd_noalloc(ctypes.byref(a), None, 0x40000, None) == 1
    assert L.attn_fwd_noalloc(ctypes.byref(a), 0x30000, None, None) == 1
    assert L.attn_fwd_noalloc(ctypes.byref(a), 0x30008, 0x40000, None) == 1
    bad = valid_args(capi, S=S, H=1, cu_seqlens=0x21000, cu_seqlens_k=0x22000, nseq=1, softcap=-1.0)
    assert L.attn_fwd_noalloc(ctypes.byref(bad), 0x30000, 0x40000, None) == 1
    a.Sq = 0
    assert L.attn_fwd(ctypes.byref(a), None, None, None, 0, None) == 0
    assert L.attn_fwd_noalloc(ctypes.byref(a), None, None, None) == 0
    b0 = valid_args(capi, B=0)
    assert L.attn_fwd_noalloc(ctypes.byref(b0), None, None, None) == 0
    assert L.attn_launch_counter() == n


def test_selftest_wait_expiry_rejects_bad_arguments(capi):
    """The failure-path self-test checks its workspace and its limit before launching."""
    L = capi.lib()
    n = L.attn_launch_counter()
    assert L.attn_selftest_wait_expiry(None, 256, 10 ** 6, None) == 3
    assert L.attn_selftest_wait_expiry(0x50000, 255, 10 ** 6, None) == 3
    assert L.attn_selftest_wait_expiry(0x50010, 256, 10 ** 6, None) == 3
    assert L.attn_selftest_wait_expiry(0x50000, 256, 999, None) == 1
    assert L.attn_selftest_wait_expiry(0x50000, 256, 2 * 10 ** 9 + 1, None) == 1
    assert L.attn_launch_counter() == n
