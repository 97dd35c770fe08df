"""The Python binding's argument checks, on the CPU: tensors of the wrong type
or on the wrong device are refused before anything reaches the library."""
import pytest
import torch

import cascade_paged_attention_gb300 as cpa


def _cpu(shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def test_verify_refuses_host_tensors():
    q = _cpu((12, 8, 128))
    kv = _cpu((4, 16, 2, 128))
    i2 = _cpu((2, 4), torch.int32)
    i1 = _cpu((2,), torch.int32)
    with pytest.raises(ValueError, match="CUDA device"):
        cpa.cpa_cascade_verify(q, kv, kv, i2, i2, i1, 2, 3)
    with pytest.raises(ValueError, match="CUDA device"):
        cpa.cpa_tree_verify(q, kv, kv, i2, i2, i1, _cpu((2, 6), torch.int32))
    with pytest.raises(ValueError, match="CUDA device"):
        cpa.cpa_cascade_verify_shared(q, kv, kv, _cpu((1, 4), torch.int32), 32, i2, i2, i1, 2, 3)


def test_verify_refuses_wrong_dtypes():
    kv = _cpu((4, 16, 2, 128))
    i2 = _cpu((2, 4), torch.int32)
    i1 = _cpu((2,), torch.int32)
    with pytest.raises(TypeError, match="bfloat16"):
        cpa.cpa_cascade_verify(_cpu((12, 8, 128), torch.float16), kv, kv, i2, i2, i1, 2, 3)
    with pytest.raises(TypeError, match="bfloat16"):
        cpa.cpa_tree_pass_b(_cpu((12, 8, 128), torch.float32), kv, kv, i2,
                            _cpu((2, 6), torch.int32))
    with pytest.raises(TypeError, match="float32"):
        cpa.cpa_merge_state(_cpu((4, 2, 128), torch.float16), _cpu((4, 2), torch.float32),
                            _cpu((4, 2, 128), torch.float32), _cpu((4, 2), torch.float32))
    with pytest.raises(TypeError, match="torch.Tensor"):
        cpa.cpa_prefill_hit([0], kv, kv, i2, 1, 4, 0)
