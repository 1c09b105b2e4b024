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



def test_every_tensor_argument_is_checked_before_the_call(q8):
    """The per-call check refuses host tensors and strided views, including a caller's
    workspace (which no shape check covers), and skips absent optional tensors."""
    q8._on_device(aux=None, norm_weight=None)
    with pytest.raises(ValueError, match="workspace"):
        q8._on_device(workspace=torch.zeros(1024, dtype=torch.uint8))
    with pytest.raises(ValueError, match="y"):
        q8._on_device(y=torch.zeros((4, 8))[:, ::2])


def test_keywords_reach_the_abi_as_their_enum_values(q8, monkeypatch):
    """With the library replaced by a recorder (and the device checks off), every keyword
    arrives at its C ABI argument as the value include/q8.h gives it."""
    calls = {}

    class Recorder:
        def __getattr__(self, name):
            def f(*args):
                calls[name] = args
                return 0
            return f
    monkeypatch.setattr(q8, "_L", Recorder())
    monkeypatch.setattr(q8, "_need", lambda t, dtype, shape, name: None)
    monkeypatch.setattr(q8, "_on_device", lambda **tensors: None)
    monkeypatch.setattr(q8, "_stream", lambda s: None)
    monkeypatch.setattr(q8, "_ptr", lambda t: None if t is None else 1)
    x = _cpu((2, 64), torch.bfloat16)
    Wq, Wd, aux = _cpu((4, 64), torch.int8), _cpu((4, 2), torch.int16), _cpu((2, 4), torch.float32)
    q8.q8_linear_fused(x, Wq, Wd, epi="silu_mul", aux=aux, path="tensor", out_dtype=torch.bfloat16)
    a = calls["q8_linear_fused"]
    assert (a[1], a[6], a[9], a[13]) == (1, 2, 1, 2)   # xtype bf16, SILU_MUL, ytype bf16, TENSOR
    q8.q8_linear_prepared(x, _cpu((4, 64), torch.int16), Wd, epi="add", aux=aux)
    assert calls["q8_linear_prepared"][6] == 1          # Q8_EPI_ADD
    q8.q8_linear_ex(x.float(), Wq, Wd, path="batch")
    assert calls["q8_linear_ex"][1] == 0 and calls["q8_linear_ex"][8] == 3   # f32 x, Q8_PATH_BATCH
    q8.q8_block_sums(_cpu((2, 64), torch.int8), Wq, path="dp4a")
    assert calls["q8_block_sums"][6] == 4               # Q8_PATH_DP4A
    q8.q8_linear_workspace_size(2, 4, 64, "decode")
    assert calls["q8_linear_workspace_size"] == (2, 4, 64, 1)
