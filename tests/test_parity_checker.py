"""The GPU-vs-oracle comparator (tests/parity.py::compare) on the CPU: it
accepts the oracle's own result rounded as the GPU path rounds it (O to
bf16, LSE to fp32) and rejects results with a planted mistake -- one output
element or one LSE off by more than the bounds, a row's LSE turned into
-inf or a -inf into a number, a NaN, two heads swapped, a wrong shape."""
import numpy as np
import pytest
import torch

from exact_attention_62_gb300.inputs import make_qkv
from parity import compare


@pytest.fixture(scope="module")
def case(oracle_mod):
    # causal with Nq > Nk: the first rows have no allowed key (LSE = -inf)
    q, k, v = make_qkv(2, 4, 2, 40, 33, 64, seed=17)
    o_ref, l_ref = oracle_mod.attn_fwd(q, k, v, True, 0.125)
    o_gpu = torch.from_numpy(o_ref).to(torch.bfloat16)
    l_gpu = torch.from_numpy(l_ref).to(torch.float32)
    return o_gpu, l_gpu, o_ref, l_ref


def test_accepts_the_oracle_rounded_as_the_gpu_rounds(case):
    o_gpu, l_gpu, o_ref, l_ref = case
    d_o, d_l = compare(o_gpu, l_gpu, o_ref, l_ref, torch.bfloat16, "rounded oracle")
    assert d_o > 0.0  # the bf16 rounding is seen, and is within the bound


def _planted(case, kind):
    o_gpu, l_gpu, o_ref, l_ref = case
    o, l = o_gpu.clone(), l_gpu.clone()
    fin = torch.isfinite(l)
    b, h, i = [int(x) for x in torch.nonzero(fin)[5]]
    if kind == "o_element":
        o[b, i, h, 3] += 0.03
    elif kind == "lse_element":
        l[b, h, i] += 2e-3
    elif kind == "lse_to_minus_inf":
        l[b, h, i] = float("-inf")
    elif kind == "minus_inf_to_number":
        b0, h0, i0 = [int(x) for x in torch.nonzero(~fin)[0]]
        l[b0, h0, i0] = 0.0
    elif kind == "nan":
        o[b, i, h, 0] = float("nan")
    elif kind == "heads_swapped":
        o = o[:, :, [1, 0, 2, 3]].contiguous()
    elif kind == "shape":
        o = o[:, :-1]
    return o, l, o_ref, l_ref


@pytest.mark.parametrize("kind", ["o_element", "lse_element", "lse_to_minus_inf", "minus_inf_to_number", "nan",
                                  "heads_swapped", "shape"])
def test_rejects_a_planted_mistake(case, kind):
    o, l, o_ref, l_ref = _planted(case, kind)
    with pytest.raises(AssertionError):
        compare(o, l, o_ref, l_ref, torch.bfloat16, kind)


def test_fp32_bound_is_the_tighter_one(case):
    _, _, o_ref, l_ref = case
    o = torch.from_numpy(o_ref).to(torch.float32)
    l = torch.from_numpy(l_ref).to(torch.float32)
    compare(o, l, o_ref, l_ref, torch.float32, "fp32 rounding")
    o[0, -1, 0, 0] += 3e-5
    with pytest.raises(AssertionError):
        compare(o, l, o_ref, l_ref, torch.float32, "fp32 planted")
