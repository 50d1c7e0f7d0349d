"""Host-side tests of the Python binding's argument checks: a request the kernels could not
serve safely (tensors off the GPU, shapes that disagree, a metadata buffer too small for its
arguments) is refused with ValueError before any pointer reaches the library, so that it fails
the call instead of faulting the GPU (TransformerEngine PR #3391, "What changed": fail
closed).  No CUDA call is made here."""
import pytest
import torch

import attention_flash_attn_gb300 as fa


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_flash_attn_gb300 import build as b
    b.build()


def qkv(B=1, Sq=16, Sk=16, Hq=2, Hkv=1, D=64):
    q = torch.zeros(B, Sq, Hq, D, dtype=torch.bfloat16)
    k = torch.zeros(B, Sk, Hkv, D, dtype=torch.bfloat16)
    return q, k, k.clone()


def test_host_tensors_refused_by_every_entry_point():
    q, k, v = qkv()
    for f in (fa.attn_fwd, fa.attn_fwd_noalloc, fa.attn_meta):
        with pytest.raises(ValueError, match="CUDA"):
            f(q, k, v, causal=True)
    O, LSE = torch.zeros_like(q), torch.zeros(1, 2, 16)
    with pytest.raises(ValueError, match="CUDA"):
        fa.attn_bwd(q, k, v, O, LSE, O, causal=True)


@pytest.mark.parametrize("kshape,vshape", [
    ((2, 16, 1, 64), (2, 16, 1, 64)),   # batch differs from q's
    ((1, 16, 1, 32), (1, 16, 1, 32)),   # head dim differs from q's
    ((1, 16, 1, 64), (1, 12, 1, 64)),   # v's rows differ from k's
    ((1, 16, 1, 64), (1, 16, 2, 64)),   # v's heads differ from k's
])
def test_key_and_value_shapes_must_agree_with_the_query(kshape, vshape):
    q = torch.zeros(1, 16, 2, 64, dtype=torch.bfloat16)
    k, v = torch.zeros(kshape, dtype=torch.bfloat16), torch.zeros(vshape, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="k and v"):
        fa.build_args(q, k, v)


def test_segment_ids_shapes():
    q, k, v = qkv(B=2, Sq=16, Sk=24)
    seg_q = torch.zeros(2, 16, dtype=torch.int32)
    with pytest.raises(ValueError, match="seg_k"):  # one id array serves both axes only if Sq == Sk
        fa.build_args(q, k, v, seg_q=seg_q)
    with pytest.raises(ValueError, match="seg_q must be"):
        fa.build_args(q, k, v, seg_q=seg_q, seg_k=torch.zeros(2, 16, dtype=torch.int32))
    with pytest.raises(ValueError, match="seg_q must be"):
        fa.build_args(q, k, v, seg_q=torch.zeros(1, 16, dtype=torch.int32), seg_k=torch.zeros(2, 24, dtype=torch.int32))
    with pytest.raises(ValueError, match="needs seg_q"):
        fa.build_args(q, k, v, seg_k=torch.zeros(2, 24, dtype=torch.int32))
    a, keep = fa.build_args(q, k, v, seg_q=seg_q, seg_k=torch.zeros(2, 24, dtype=torch.int32))
    assert a.seg_q and a.seg_k and a.seg_q != a.seg_k


def test_sink_and_cu_seqlens_shapes():
    q, k, v = qkv(Hq=4, Hkv=2)
    with pytest.raises(ValueError, match="sink"):
        fa.build_args(q, k, v, sink=torch.zeros(2))
    with pytest.raises(ValueError, match="cu_seqlens"):
        fa.build_args(q, k, v, cu_seqlens=torch.zeros(2, 2, dtype=torch.int32))
    a, keep = fa.build_args(q, k, v, sink=torch.zeros(4), cu_seqlens=torch.tensor([0, 5, 16], dtype=torch.int32))
    assert a.nseq == 2 and a.sink


def test_metadata_buffer_must_hold_what_its_arguments_need():
    import ctypes
    q, k, v = qkv(B=2, Sq=300, Sk=300)
    seg = torch.zeros(2, 300, dtype=torch.int32)
    a, keep = fa.build_args(q, k, v, causal=True, seg_q=seg)
    need = fa.lib().attn_meta_size(ctypes.byref(a))
    assert need > 256
    buf = torch.zeros(need + 256, dtype=torch.uint8)[256:]  # dtype and size right (alignment is the library's check)
    a2, keep2 = fa.build_args(q, k, v, causal=True, seg_q=seg, meta=buf)
    assert a2.meta == buf.data_ptr()
    with pytest.raises(ValueError, match="need"):
        fa.build_args(q, k, v, causal=True, seg_q=seg, meta=buf[: need - 1])
    with pytest.raises(ValueError, match="uint8"):
        fa.build_args(q, k, v, causal=True, seg_q=seg, meta=torch.zeros(need, dtype=torch.int32))


@pytest.mark.parametrize("shape", [(3, 1, 16, 16), (1, 3, 16, 16), (1, 1, 16, 15), (2, 16, 16)])
def test_bias_shape_must_broadcast_over_batch_and_heads(shape):
    q, k, v = qkv(B=2, Hq=2)
    with pytest.raises(ValueError, match="bias"):
        fa.build_args(q, k, v, bias=torch.zeros(shape, dtype=torch.bfloat16))
    for ok in [(1, 1, 16, 16), (2, 1, 16, 16), (1, 2, 16, 16), (2, 2, 16, 16)]:
        a, keep = fa.build_args(q, k, v, bias=torch.zeros(ok, dtype=torch.bfloat16))
        assert a.bias and (a.bias_stride_b != 0) == (ok[0] == 2) and (a.bias_stride_h != 0) == (ok[1] == 2)
