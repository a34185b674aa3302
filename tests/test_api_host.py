"""The tensor API's marshalling on the CPU: how a tensor's strides map to
the stored layout and pitch the C ABI receives, and the argument errors the
Python layer raises before any library call."""

import pytest
import torch

import dense_gemm_02_gb300 as g
from dense_gemm_02_gb300 import api


def test_layout_of_row_major_and_transposed_views():
    W = torch.zeros(5, 7)
    assert api._layout(W, "A") == (0, 7)             # row-major, pitch 7
    assert api._layout(W.t(), "A") == (1, 7)         # stored 5 x 7: A = W^T is 7 x 5
    P = torch.zeros(5, 12)[:, :7]                    # pitched rows
    assert api._layout(P, "A") == (0, 12)
    assert api._layout(P.t(), "A") == (1, 12)
    assert api._layout(torch.zeros(1, 7), "A") == (0, 7)   # one row: pitch = row length
    assert api._layout(torch.zeros(5, 1), "A") == (0, 1)   # one column
    with pytest.raises(ValueError, match="transpose of a row-major"):
        api._layout(torch.zeros(6, 8)[::2, ::2], "A")
    with pytest.raises(ValueError, match="2-D"):
        api._layout(torch.zeros(2, 3, 4), "A")


def test_row_major_pitch_and_rejections():
    assert api._row_major(torch.zeros(4, 6), "C") == 6
    assert api._row_major(torch.zeros(4, 16)[:, :6], "C") == 16
    assert api._row_major(torch.zeros(0, 6), "C") == 6        # empty: any valid pitch
    assert api._row_major(torch.zeros(1, 6), "C") == 6
    with pytest.raises(ValueError, match="unit column stride"):
        api._row_major(torch.zeros(6, 4).t(), "C")
    with pytest.raises(ValueError, match="2-D"):
        api._row_major(torch.zeros(6), "C")


def test_shape_checks():
    assert api._shapes(torch.zeros(3, 4), torch.zeros(4, 5), None) == (3, 5, 4)
    with pytest.raises(ValueError, match="inner dimensions"):
        api._shapes(torch.zeros(3, 4), torch.zeros(5, 5), None)
    with pytest.raises(ValueError, match="C must be"):
        api._shapes(torch.zeros(3, 4), torch.zeros(4, 5), torch.zeros(5, 3))


def test_device_entry_points_reject_host_or_wrong_dtype_tensors():
    a32, b32 = torch.zeros(4, 4), torch.zeros(4, 4)
    a16, b16 = a32.bfloat16(), b32.bfloat16()
    with pytest.raises(TypeError, match="float32 CUDA"):
        g.sgemm(a32, b32)
    with pytest.raises(TypeError, match="bfloat16 CUDA"):
        g.gemm_bf16(a16, b16)
    with pytest.raises(TypeError, match="float32 or both bfloat16"):
        g.gemm_ex(a32, b16)
    with pytest.raises(TypeError, match="CUDA tensors"):
        g.gemm_ex(a16, b16)
    with pytest.raises(ValueError, match="3-D"):
        g.gemm_batched(a16, b16)


def test_host_buffer_call_argument_errors():
    a, b = torch.zeros(4, 6), torch.zeros(6, 5)
    with pytest.raises(TypeError, match="float32 or both bfloat16"):
        g.gemm(a, b.bfloat16())
    with pytest.raises(TypeError, match="float32 or both bfloat16"):
        g.gemm(a.double(), b.double())
    with pytest.raises(ValueError, match="out must be"):
        g.gemm(a, b, out=torch.zeros(4, 6))
    with pytest.raises(ValueError, match="out must be"):
        g.gemm(a, b, out=torch.zeros(4, 5, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="inner dimensions"):
        g.gemm(a, torch.zeros(5, 5))
    with pytest.raises(TypeError, match="output must be float32 or bfloat16"):
        g.gemm(a.bfloat16(), b.bfloat16(), out_dtype=torch.float16)
