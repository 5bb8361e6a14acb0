"""Failure detection on the GPU without a fault: a pipeline wait that runs out.

FA_FLAG_TEST_SKIP_KV_LOAD makes the tensor-core kernel's loader skip one key
tile, so the waits that depend on it run out (20 ms under the flag).  The
kernel must report FA_ERR_TIMEOUT through fa_check_device_error, leave the
context usable, and the next call must be correct.  Nothing traps or hangs.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_online_softmax_attn_gb300 as fa
from parity import compare

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,causal", [(128, False), (64, True)])
def test_skipped_load_times_out_and_the_next_call_works(d, causal):
    w = synth.Workload("t", 1, 1, 512, d, "bf16", causal, seed=4000 + d)
    q, k, v = w.inputs()
    qd, kd, vd = (torch.from_numpy(x).cuda().to(torch.bfloat16) for x in (q, k, v))
    assert fa.check_device_error() == fa.FA_OK
    fa.fa_forward(qd, kd, vd, scale=w.scale, causal=causal, flags=fa.FA_FLAG_TEST_SKIP_KV_LOAD)
    st = fa.check_device_error()
    assert st == fa.FA_ERR_TIMEOUT, fa.last_error()
    assert "gave up" in fa.last_error()
    # the error word was cleared and the context still works
    assert fa.check_device_error() == fa.FA_OK
    o, lse = fa.fa_forward(qd, kd, vd, scale=w.scale, causal=causal)
    assert fa.check_device_error() == fa.FA_OK
    o_ref, l_ref = oracle.attention(q, k, v, w.scale, causal)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "bf16", "bf16")


def test_flag_has_no_effect_on_a_single_key_tile():
    w = synth.Workload("t", 1, 2, 100, 128, "bf16", False, seed=4100)
    q, k, v = w.inputs()
    qd, kd, vd = (torch.from_numpy(x).cuda().to(torch.bfloat16) for x in (q, k, v))
    o, lse = fa.fa_forward(qd, kd, vd, scale=w.scale, flags=fa.FA_FLAG_TEST_SKIP_KV_LOAD)
    assert fa.check_device_error() == fa.FA_OK
    o_ref, l_ref = oracle.attention(q, k, v, w.scale, False)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "bf16", "bf16")
