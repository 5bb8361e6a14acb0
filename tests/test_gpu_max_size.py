"""Problems whose tensors hold more than 2^31 elements (4 GiB of bf16).

"The Details of Flash Attention" works through one head of N x d (its kernels
section: N = d = 1024); a batched library addresses B*H*N*d elements, and past
2^31 elements a 32-bit offset would wrap.  These tests fill Q, K, V (and dO)
from 61 seeded base heads, head h taking base h mod 61, so that a wrapped
offset reads or writes a head with other data (61 is prime and the wrap
distance, 2^31 elements, is not a multiple of 61 heads), and check:

* sampled heads on both sides of the 2^31-element boundary, and the last
  ones, against the oracle run on their base head;
* that every sampled head is bit-identical to the low head with the same
  base (the kernels are deterministic and position-independent).

Every kernel computes element offsets in 64-bit arithmetic; these tests run
the paths that batched problems of this size take: the tensor-core forward
at d = 128 and 64, the CUDA-core forward (d = 40 forced onto it) and the
tensor-core backward.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_online_softmax_attn_gb300 as fa

pytestmark = pytest.mark.gpu

PERIOD = 61          # distinct base heads
B, N = 2, 129        # N ragged: a full and a one-row query tile per head


def heads_for(d):
    """H such that B*H*N*d is about 2.3e9 elements, 7 % past 2^31."""
    return -(-int(1.07 * (1 << 31)) // (B * N * d))


def _base(d, seed, causal=False):
    w = synth.Workload("max-size base", 1, PERIOD, N, d, "bf16", causal, seed=seed)
    return w, w.inputs()


def _expand(x):
    """[1, PERIOD, N, d] host array -> [B, H, N, d] bf16 device tensor, head
    h = base h mod PERIOD."""
    base = torch.from_numpy(x[0]).to(torch.bfloat16).cuda()
    H = heads_for(base.shape[-1])
    idx = torch.arange(B * H, device="cuda") % PERIOD
    return base.index_select(0, idx).view(B, H, N, base.shape[-1])


def _heads(d):
    """Flat head indices to check: the first ones, those on both sides of the
    2^31-element boundary, and the last ones."""
    n_heads = B * heads_for(d)
    edge = (1 << 31) // (N * d)
    cand = [0, 1, PERIOD, edge - 2, edge - 1, edge, edge + 1, edge + 2, n_heads // 2, n_heads - 2, n_heads - 1]
    assert edge + 2 < n_heads
    return sorted({h for h in cand if 0 <= h < n_heads})


def _flat(t):
    return t.view(-1, N, t.shape[-1])


def _check_forward(o, lse, ref, d, tol_o):
    o_f, l_f = _flat(o), lse.view(-1, N)
    for h in _heads(d):
        b = h % PERIOD
        o_h = o_f[h].float().cpu().numpy()
        err = np.abs(o_h - ref[0][0, b]).max()
        assert err <= tol_o, f"head {h}: O max error {err}"
        lerr = np.abs(l_f[h].cpu().numpy() - ref[1][0, b]).max()
        assert lerr <= 1e-3, f"head {h}: LSE max error {lerr}"
        # the same base head, far below the boundary: bit-identical
        assert torch.equal(o_f[h], o_f[b]), f"head {h} differs from head {b}"
        assert torch.equal(l_f[h], l_f[b])


@pytest.mark.parametrize("d,flags", [(128, 0), (64, 0), (40, fa.FA_FLAG_GENERAL_PATH)])
def test_forward_beyond_2_31_elements(d, flags):
    w, (q, k, v) = _base(d, seed=9100 + d)
    ref = oracle.attention(q, k, v, w.scale, False)
    qd, kd, vd = _expand(q), _expand(k), _expand(v)
    assert qd.numel() > (1 << 31)
    o, lse = fa.fa_forward(qd, kd, vd, scale=w.scale, flags=flags)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    # bf16 O: the stated 1e-2 bound plus half a bf16 ulp of |O| <= 4
    _check_forward(o, lse, ref, d, 1e-2 + 2.0 ** -7)


def test_backward_beyond_2_31_elements():
    d = 128
    w, (q, k, v) = _base(d, seed=9200, causal=True)
    dout = synth.tensor(3 * 9200 + 9, (1, PERIOD, N, d), "bf16")
    ref = oracle.attention_backward(q, k, v, dout, w.scale, True)
    qd, kd, vd, gd = _expand(q), _expand(k), _expand(v), _expand(dout)
    assert qd.numel() > (1 << 31)
    o, lse = fa.fa_forward(qd, kd, vd, scale=w.scale, causal=True)
    assert fa.backward_plan(*qd.shape, torch.bfloat16, True)[1] == "tensor-core"
    grads = fa.fa_backward(qd, kd, vd, o, gd, lse, scale=w.scale, causal=True)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        g_f = _flat(g)
        bound = 2e-2 * np.abs(r).max()
        for h in _heads(d):
            b = h % PERIOD
            err = np.abs(g_f[h].float().cpu().numpy() - r[0, b]).max()
            assert err <= bound + 2.0 ** -8 * np.abs(r[0, b]).max(), f"{name} head {h}: max error {err}"
            assert torch.equal(g_f[h], g_f[b]), f"{name}: head {h} differs from head {b}"
