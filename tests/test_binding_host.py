"""Argument checks of the Python binding that run before the library is
called: wrong types and host tensors are refused with an exception, never
passed on as pointers."""

import pytest
import torch

import paged_kv_cache_pkv_gb300 as pkv


def _attend_args(**over):
    a = dict(q=torch.zeros(4, 8, 128, dtype=torch.bfloat16),
             k_cache=torch.zeros(8, 2, 16, 128, dtype=torch.bfloat16),
             v_cache=torch.zeros(8, 2, 16, 128, dtype=torch.bfloat16),
             block_tables=torch.zeros(4, 2, dtype=torch.int32),
             seq_lens=torch.ones(4, dtype=torch.int32),
             query_start_loc=torch.arange(5, dtype=torch.int32), scale=0.088)
    a.update(over)
    return a


def test_attend_refuses_wrong_types():
    # arguments are checked in order, so on a host without a GPU only the
    # first one's type check is reached before the device check
    with pytest.raises(TypeError, match="q must be"):
        pkv.attend(**_attend_args(q=torch.zeros(4, 8, 128, dtype=torch.float32)))
    with pytest.raises(TypeError, match="q must be a torch.Tensor"):
        pkv.attend(**_attend_args(q=[[0.0]]))


def test_attend_refuses_host_tensors():
    with pytest.raises(ValueError, match="CUDA"):
        pkv.attend(**_attend_args())


def test_write_refuses_wrong_types_and_host_tensors():
    kn = torch.zeros(4, 2, 128, dtype=torch.bfloat16)
    pool = torch.zeros(8, 2, 16, 128, dtype=torch.bfloat16)
    with pytest.raises(TypeError, match="k_new"):
        pkv.write(kn.float(), kn, torch.zeros(4, dtype=torch.int64), pool, pool)
    with pytest.raises(ValueError, match="CUDA"):
        pkv.write(kn, kn, torch.zeros(4, dtype=torch.int64), pool, pool)


def test_fp8_calls_refuse_bf16_pools():
    kn = torch.zeros(4, 2, 128, dtype=torch.bfloat16)
    pool = torch.zeros(8, 2, 16, 128, dtype=torch.bfloat16)
    scales = torch.zeros(8, 2, 16, dtype=torch.uint8)
    with pytest.raises((TypeError, ValueError)):
        pkv.write_fp8(kn, kn, torch.zeros(4, dtype=torch.int64), pool, pool, scales, scales)
    a = _attend_args()
    with pytest.raises((TypeError, ValueError)):
        pkv.attend_fp8(a["q"], pool, pool, scales, scales, a["block_tables"], a["seq_lens"],
                       a["query_start_loc"], a["scale"])
