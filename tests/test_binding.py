"""The Python binding without a GPU: argument checks that run before any CUDA call.

The binding marshals tensors into the C ABI; it refuses wrong dtypes, unknown keywords,
missing companions and tensors that are not contiguous CUDA tensors on the current device,
so that no bad pointer reaches a kernel.
"""
import pytest

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def q8():
    import __graft_entry__ as g
    g.build()
    import q8_int8_block_gb300 as m
    return m


def _cpu(shape, dtype):
    return torch.zeros(shape, dtype=dtype)


def test_keywords_are_checked_first(q8):
    x = _cpu((2, 64), torch.bfloat16)
    Wq, Wd = _cpu((4, 64), torch.int8), _cpu((4, 2), torch.int16)
    with pytest.raises(ValueError, match="epi"):
        q8.q8_linear_fused(x, Wq, Wd, epi="gelu")
    with pytest.raises(ValueError, match="path"):
        q8.q8_linear_fused(x, Wq, Wd, path="cublas")
    with pytest.raises(ValueError, match="needs aux"):
        q8.q8_linear_fused(x, Wq, Wd, epi="add")
    with pytest.raises(TypeError, match="out_dtype"):
        q8.q8_linear_fused(x, Wq, Wd, out_dtype=torch.float16)
    with pytest.raises(ValueError, match="path"):
        q8.q8_linear_ex(x, Wq, Wd, path="fast")
    with pytest.raises(ValueError, match="path"):
        q8.q8_linear_workspace_size(2, 4, 64, path="fast")
    with pytest.raises(ValueError, match="path"):
        q8.q8_block_sums(_cpu((2, 64), torch.int8), Wq, path="slow")
    with pytest.raises(ValueError, match="epi"):
        q8.q8_linear_prepared(x, _cpu((4, 64), torch.int16), Wd, epi="relu")


def test_dtypes_are_checked(q8):
    with pytest.raises(TypeError, match="W"):
        q8.q8_quantize_weights(_cpu((4, 64), torch.float64))
    with pytest.raises(TypeError, match="x"):
        q8.q8_quantize_act(_cpu((2, 64), torch.float16))
    with pytest.raises(TypeError, match="x"):
        q8.q8_linear(_cpu((2, 64), torch.float32), _cpu((4, 64), torch.int8), _cpu((4, 2), torch.int16))
    with pytest.raises(TypeError, match="x"):
        q8.q8_kv3_encode(_cpu((4, 128), torch.int32))
    with pytest.raises(TypeError, match="q"):
        q8.q8_bsa_attention(_cpu((2, 64, 128), torch.float32), _cpu((1, 64, 128), torch.bfloat16),
                            _cpu((1, 64, 128), torch.bfloat16), _cpu((3,), torch.int32),
                            _cpu((2,), torch.int32))


def test_host_tensors_never_reach_the_library(q8):
    with pytest.raises(ValueError, match="CUDA"):
        q8.q8_quantize_weights(_cpu((4, 64), torch.float32))
    with pytest.raises(ValueError, match="CUDA"):
        q8.q8_linear(_cpu((2, 64), torch.bfloat16), _cpu((4, 64), torch.int8), _cpu((4, 2), torch.int16))
    with pytest.raises(ValueError, match="CUDA"):
        q8.q8_kv3_encode(_cpu((4, 128), torch.bfloat16))
    with pytest.raises(ValueError, match="whole 128-element groups"):
        q8.q8_kv3_encode(_cpu((4, 100), torch.bfloat16))
    with pytest.raises(ValueError, match="CUDA"):
        q8.q8_bsa_attention(*(_cpu((2, 64, 128), torch.bfloat16) for _ in range(3)),
                            _cpu((3,), torch.int32), _cpu((2,), torch.int32))

