"""The Python binding turns the library's host-side refusals into DGError with
the status name; the arguments here are rejected before any device access, so
these run without a GPU."""
import types

import pytest
import torch

from block_scaled_fp8_gb300 import binding

NO_STREAM = types.SimpleNamespace(cuda_stream=0)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from block_scaled_fp8_gb300 import build
    build.build()
    binding.lib()


def test_fp4_k_not_multiple_of_128_raises():
    a = torch.zeros(128, 192, dtype=torch.float8_e4m3fn)
    b = torch.zeros(128, 96, dtype=torch.uint8)
    sf = torch.zeros(64, dtype=torch.int32)
    d = torch.zeros(128, 128, dtype=torch.bfloat16)
    with pytest.raises(binding.DGError) as e:
        binding.dg_fp8_fp4_gemm_nt(a, sf, b, sf, d, stream=NO_STREAM)
    assert e.value.name == "DG_ERR_ALIGNMENT"


def test_k_grouped_bad_group_size_raises():
    a = torch.zeros(256, 128, dtype=torch.float8_e4m3fn)
    b = torch.zeros(256, 128, dtype=torch.float8_e4m3fn)
    sf = torch.zeros(8, 128, dtype=torch.int32)
    c = torch.zeros(1, 128, 128, dtype=torch.float32)
    with pytest.raises(binding.DGError) as e:
        binding.dg_k_grouped_fp8_gemm_tn_contiguous(a, sf, b, sf, c, [130], c=c, stream=NO_STREAM)
    assert e.value.name == "DG_ERR_INVALID_ARG"


def test_k_grouped_transform_needs_mn_multiple_of_4():
    sf = torch.ones(2, 6, dtype=torch.float32)
    out = torch.zeros(1, 6, dtype=torch.int32)
    with pytest.raises(binding.DGError) as e:
        binding.dg_transform_sf_k_grouped(sf, [256], out=out, stream=NO_STREAM)
    assert e.value.name == "DG_ERR_LAYOUT"


def test_k_grouped_packed_rows_helper():
    assert binding.k_grouped_packed_sf_rows([256, 640, 0, 128]) == 4
    assert binding.k_grouped_packed_sf_rows([100]) == -1
