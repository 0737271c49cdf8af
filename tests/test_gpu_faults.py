"""Failure paths on the GPU without faulting it.

The tensor-core kernel bounds every wait; the testing-only `debug=1` knob withholds the V tiles
so the MMA issuer's wait runs out of its (shortened) budget.  The kernel must report
CP_ERR_TIMEOUT in the error word, drain its own copies and MMAs, free TMEM and return, leaving
the context usable: a normal call right after must still match the oracle.
"""
import math

import pytest
import torch

from oracle import cp_oracle as orc
import workloads as wl
from tests.parity_util import check_partials

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("impl", ["tc", "tc1"])
def test_wait_timeout_is_reported_and_context_survives(lib, impl):
    lens, Hq, Hkv, d, cp = [640], 8, 2, 128, 2
    x = wl.prefill_inputs(lens, Hq, Hkv, d, torch.bfloat16, seed=77)
    q, k, v, cu = (x[n].cuda() for n in ("q", "k", "v", "cu_seqlens"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    code = {"tc": lib.CP_IMPL_TCGEN05, "tc1": lib.CP_IMPL_TCGEN05_SINGLE}[impl]
    lib.cp_partial_attn_prefill(q, cu, cp, k=k, v=v, max_seqlen_q=640, impl=code, err=err,
                                debug=1)
    torch.cuda.synchronize()
    assert int(err.item()) == 4          # CP_ERR_TIMEOUT
    err.zero_()
    out, lse = lib.cp_partial_attn_prefill(q, cu, cp, k=k, v=v, max_seqlen_q=640, impl=code,
                                           err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    O, L = orc.pass_kv_partials(x["q"], x["k"], x["v"], x["cu_seqlens"], cp, 1 / math.sqrt(d))
    check_partials(out, lse, O, L, what="after timeout")


def test_host_rejects_before_launch(lib):
    q = torch.zeros(10, 8, 96, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 10], dtype=torch.int32, device="cuda")
    with pytest.raises(lib.CPError) as e:
        lib.cp_partial_attn_prefill(q, cu, 2, k=q[:, :2].contiguous(), v=q[:, :2].contiguous())
    assert e.value.status == 2       # head_dim 96 unsupported
