"""GPU parity: the CUDA kernels (through the C ABI) against the CPU fp64 oracle.

Small shapes are compared element by element on every output.  At full
size the multi-head (4x32x4096x128) and causal (1x32x16384x128) workloads
are compared on every row, and the very-long peaked one (1x8x65536x64) on
16384 seeded rows plus the first, second, 128th, 129th, middle and last two
rows of every head, each against the full key range.  Both kernels are
covered: the tensor-core kernel (bf16, d of 64 or 128) through the default
dispatch and the general-d kernel through FA_FLAG_GENERAL_PATH.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_online_softmax_attn_gb300 as fa
from conftest import read_golden
from parity import compare, sample_rows

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "fp32": torch.float32}
PATHS = {"auto": 0, "general": fa.FA_FLAG_GENERAL_PATH}


def to_dev(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(TORCH_DT[dtype])


def run(q, k, v, dtype, scale, causal, o_dtype=None, flags=0):
    qd, kd, vd = (to_dev(x, dtype) for x in (q, k, v))
    o, lse = fa.fa_forward(qd, kd, vd, scale=scale, causal=causal,
                           o_dtype=TORCH_DT[o_dtype or dtype], flags=flags)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def full_check(w, path, o_dtype=None):
    q, k, v = w.inputs()
    o, lse = run(q, k, v, w.dtype, w.scale, w.causal, o_dtype, PATHS[path])
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, w.causal)
    return compare(o, lse, o_ref, lse_ref, w.dtype, o_dtype or w.dtype,
                   label=f"{w.name} {w.B}x{w.H}x{w.N}x{w.d} {w.dtype}{' causal' if w.causal else ''} {path} "
                         f"O {o_dtype or w.dtype}")


SMALL = [
    # (B, H, N, d, dtype, causal): several tiles plus ragged tails
    (1, 2, 256, 64, "bf16", False),
    (1, 2, 256, 64, "bf16", True),
    (2, 3, 200, 64, "bf16", True),
    (1, 2, 77, 128, "bf16", False),
    (2, 1, 129, 128, "bf16", False),
    (1, 2, 300, 128, "bf16", True),
    (1, 1, 513, 64, "bf16", True),
    (1, 1, 640, 128, "bf16", False),
    (1, 1, 1, 64, "bf16", False),
    (1, 1, 1, 128, "bf16", True),
    (3, 2, 96, 128, "fp32", False),
]


@pytest.mark.parametrize("path", ["auto", "general"])
@pytest.mark.parametrize("B,H,N,d,dtype,causal", SMALL)
def test_small_shapes_full(B, H, N, d, dtype, causal, path):
    w = synth.Workload("t", B, H, N, d, dtype, causal, seed=1000 + N + d)
    full_check(w, path)


@pytest.mark.parametrize("d", [1, 3, 16, 40, 100, 200, 257])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("causal", [False, True])
def test_general_head_dims(d, dtype, causal):
    w = synth.Workload("t", 1, 2, 150, d, dtype, causal, seed=2000 + d)
    full_check(w, "general")


@pytest.mark.parametrize("d", [8, 16, 24, 40, 56, 72, 80, 96, 112, 120])
@pytest.mark.parametrize("causal", [False, True])
def test_narrow_head_dims_on_tensor_cores(d, causal):
    """Head dimensions below 128 that are multiples of 8 run on the tensor-core
    kernel padded to 64 or 128: the tensor maps keep the real width, so the
    missing columns load as zeros (no effect on S) and O's padding columns are
    not stored."""
    w = synth.Workload("t", 1, 3, 200, d, "bf16", causal, seed=2500 + d)
    assert fa.plan(w.B, w.H, w.N, d, torch.bfloat16, torch.bfloat16, causal)[1].startswith(f"tensor-core d={d}")
    full_check(w, "auto")


@pytest.mark.parametrize("path", ["auto", "general"])
@pytest.mark.parametrize("o_dtype", ["bf16", "fp32"])
def test_tiny_workload(path, o_dtype):
    full_check(synth.WORKLOADS["tiny"], path, o_dtype)


def test_large_d_fp32_workload():
    stats = full_check(synth.WORKLOADS["large_d"], "auto")
    assert stats["o_max"] <= 2e-4


def _sampled(w, o_dtype=None, flags=0, nrows=384):
    q, k, v = w.inputs()
    o, lse = run(q, k, v, w.dtype, w.scale, w.causal, o_dtype, flags)
    rows = sample_rows(w.B, w.H, w.N, nrows, seed=w.seed)
    o_ref, lse_ref = oracle.attention_rows(q, k, v, w.scale, w.causal, rows)
    return compare(o.reshape(-1, w.d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref,
                   w.dtype, o_dtype or w.dtype, label=f"{w.name} {rows.size} rows O {o_dtype or w.dtype}")


@pytest.mark.parametrize("name", ["multihead", "causal"])
def test_full_size_workloads_every_row(name):
    """Every element of O and LSE of the full-size workload against the
    oracle's three passes over the full key range."""
    w = synth.WORKLOADS[name]
    q, k, v = w.inputs()
    o, lse = run(q, k, v, w.dtype, w.scale, w.causal)
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, w.causal)
    del q, k, v
    compare(o, lse, o_ref, lse_ref, w.dtype, w.dtype, label=f"{w.name} every row O {w.dtype}")


@pytest.mark.parametrize("o_dtype", ["bf16", "fp32"])
def test_peaked_workload_rows(o_dtype):
    """The 1x8x65536x64 peaked workload on 16384 seeded rows plus each head's
    edge rows; with fp32 O the plain bounds hold without the bf16 floor."""
    _sampled(synth.WORKLOADS["peaked"], o_dtype=o_dtype, nrows=16384)


@pytest.mark.parametrize("d", [64, 128])
def test_persistent_ctas_with_ragged_rows(d):
    """More items (256-row query blocks x heads) than SMs, few key tiles and a
    ragged N: CTAs loop over several items each, so the per-item barrier
    phases and the release of O between items are exercised; every row of the
    last, partial query block is checked too."""
    w = synth.Workload("persistent", 2, 40, 1000, d, "bf16", False, seed=7100 + d)
    q, k, v = w.inputs()
    o, lse = run(q, k, v, w.dtype, w.scale, w.causal)
    rows = np.unique(np.concatenate([sample_rows(w.B, w.H, w.N, 512, seed=w.seed),
                                     np.arange(w.N - 232, w.N, dtype=np.int64) + (w.B * w.H - 1) * w.N]))
    o_ref, lse_ref = oracle.attention_rows(q, k, v, w.scale, w.causal, rows)
    compare(o.reshape(-1, w.d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, w.dtype, w.dtype)


@pytest.mark.parametrize("d,N", [(64, 1000), (128, 300), (128, 2048)])
def test_persistent_ctas_causal_short_items(d, N):
    """Causal items short enough to run on persistent CTAs (at most 2048
    key-tile columns, more items than SMs): every CTA loops over items of
    unequal length, longest first in rounds of alternating direction.  Every
    row against the oracle."""
    w = synth.Workload("persistent causal", 2, 80 if N < 2048 else 40, N, d, "bf16", True, seed=7200 + d + N)
    q, k, v = w.inputs()
    o, lse = run(q, k, v, w.dtype, w.scale, w.causal)
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, w.causal)
    compare(o, lse, o_ref, lse_ref, w.dtype, w.dtype, label=f"persistent causal {w.B}x{w.H}x{N}x{d}")


def test_repeat_runs_are_bitwise_identical():
    w = synth.WORKLOADS["tiny"].scaled(N=333, causal=True)
    q, k, v = w.inputs()
    a = run(q, k, v, w.dtype, w.scale, w.causal)
    b = run(q, k, v, w.dtype, w.scale, w.causal)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_side_stream_and_no_lse():
    w = synth.WORKLOADS["tiny"]
    q, k, v = (to_dev(x, "bf16") for x in w.inputs())
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fa.fa_forward(q, k, v, return_lse=False, stream=s)
    s.synchronize()
    assert lse is None
    o_ref, _ = oracle.attention(*w.inputs(), w.scale, False)
    compare(o.float().cpu().numpy(), None, o_ref, None, "bf16", "bf16")


def test_uniform_scores_give_mean_of_values_on_gpu():
    """Q = 0: every causal row i is the mean of v_0..v_i (closed form)."""
    N, d = 300, 128
    v = synth.tensor(77, (1, 1, N, d), "bf16")
    q = np.zeros_like(v)
    k = synth.tensor(78, (1, 1, N, d), "bf16")
    for flags in PATHS.values():
        o, lse = run(q, k, v, "bf16", 0.1, True, "fp32", flags)
        ref = np.cumsum(v[0, 0].astype(np.float64), axis=0) / np.arange(1, N + 1)[:, None]
        assert np.abs(o[0, 0] - ref).max() < 1e-3
        assert np.abs(lse[0, 0] - np.log(np.arange(1, N + 1))).max() < 1e-4


def test_worked_example_on_gpu():
    """The 4x4 worked example of "Deep Learning - Flash Attention" ("An
    Example"), zero-padded to d = 64 (the padding adds nothing to q . k and V's
    padding columns are 0), with the page's scale passed explicitly: rows 1
    and 2 of O are the probability rows the page prints to four decimals.  The
    general kernel keeps fp32 weights, so it must agree to the printed digits;
    the tensor-core kernel feeds bf16 weights to the P V product (each rounded
    by up to 2^-8 of itself, and the normaliser, exact but for the top weight,
    differs from their sum by up to 2^-8 of the other weights' share), so it is
    allowed 2^-7 of each value more."""
    g = read_golden("worked_example_4x4.txt")
    Q = np.array([[1, 2, 3, 4], [2, 1, 0, -1], [4, 3, 2, 1], [-1, 0, 1, 2]], dtype=np.float32)
    d = 64
    q, k, v = (np.zeros((1, 1, 4, d), dtype=np.float32) for _ in range(3))
    q[0, 0, :, :4] = Q
    k[0, 0, :, :4] = 2.0 * np.eye(4)
    v[0, 0, :, :4] = np.eye(4)
    scale = g["scale"][0]
    printed = np.array([g["O_row1"], g["O_row2"]])
    half_digit = 0.5 * 10.0 ** -int(g["decimals"][0])
    # S = scale Q (2 I) = Q, so the natural-log LSE of each row is logsumexp(Q_i)
    lse_exact = np.log(np.exp(Q.astype(np.float64)).sum(axis=1))
    for dtype, flags, rel in (("bf16", 0, 2.0 ** -7), ("bf16", fa.FA_FLAG_GENERAL_PATH, 0.0),
                              ("fp32", 0, 0.0)):
        o, lse = run(q, k, v, dtype, scale, False, "fp32", flags)
        err = np.abs(o[0, 0, :2, :4] - printed)
        assert np.all(err <= half_digit + rel * printed + 1e-5), (dtype, flags, err.max())
        assert np.all(o[0, 0, :, 4:] == 0)
        assert np.abs(lse[0, 0] - lse_exact).max() < 1e-4


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("direction", ["rising", "falling"])
def test_scores_ramping_across_key_tiles(d, causal, direction):
    """Every query is one +-1 vector u and key j is t_j u, with t_j rising (or
    falling) along the keys, so the scores climb by 14-20 (natural units) per
    128-key tile.  Rising scores move every row's maximum on every tile, past
    the lazy-rescale margin each time, so O is rescaled on each one; falling
    scores keep the maximum in the first tile and drive the later weights to
    exact zeros."""
    N = 1024
    u = np.where(synth.tensor(501, (d,), "bf16") < 0, -1.0, 1.0).astype(np.float32)
    t = synth.round_to_bf16((14.0 * np.arange(N) / N).astype(np.float32))
    if direction == "falling":
        t = t[::-1].copy()
    q = np.broadcast_to(u, (1, 2, N, d)).astype(np.float32)
    # t_j is bf16 and u is +-1, so every key element is exact in bf16
    k = np.broadcast_to(t[:, None] * u[None, :], (1, 2, N, d)).astype(np.float32)
    v = synth.tensor(502, (1, 2, N, d), "bf16")
    scale = 1.0 / np.sqrt(d)
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal)
    for flags in PATHS.values():
        o, lse = run(q, k, v, "bf16", scale, causal, None, flags)
        compare(o, lse, o_ref, l_ref, "bf16", "bf16")


def test_invalid_arguments_are_rejected_before_launch():
    q = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    st = fa.forward_raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), None,
                        1, 1, 8, 64, float("nan"), 0, fa.FA_BF16, fa.FA_BF16)
    assert st == fa.FA_ERR_INVALID_ARG
    st = fa.forward_raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), None,
                        1, 1, 8, 64, 1.0, 0, fa.FA_BF16, fa.FA_BF16)
    assert st == fa.FA_ERR_INVALID_ARG and "overlap" in fa.last_error()
    st = fa.forward_raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), None,
                        1, 1, 8, 2048, 1.0, 0, fa.FA_BF16, fa.FA_BF16)
    assert st == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("B,H,N,d,dtype,causal", [(2, 5, 300, 128, "bf16", True), (2, 8, 1024, 128, "bf16", True),
                                                  (1, 3, 200, 64, "bf16", False),
                                                  (1, 2, 100, 40, "fp32", False)])
def test_host_buffer_entry_point_matches_device_path(B, H, N, d, dtype, causal):
    """fa_forward_host (pinned host buffers, pipelined chunks of heads) gives
    the same bits as fa_forward on device buffers, and both match the oracle."""
    w = synth.Workload("t", B, H, N, d, dtype, causal, seed=3000 + N)
    q, k, v = w.inputs()
    tdt = TORCH_DT[dtype]
    qh, kh, vh = (torch.from_numpy(x).to(tdt).pin_memory() for x in (q, k, v))
    oh = torch.empty(w.shape, dtype=tdt).pin_memory()
    lh = torch.empty(w.shape[:3], dtype=torch.float32).pin_memory()
    ws = torch.empty(fa.host_workspace_size(B, H, N, d, tdt, tdt), dtype=torch.uint8, device="cuda")
    for _ in range(2):   # repeated calls reuse the cached streams and events
        fa.forward_host(qh, kh, vh, oh, lh, ws, scale=w.scale, causal=causal)
    od, ld = fa.fa_forward(qh.cuda(), kh.cuda(), vh.cuda(), scale=w.scale, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(oh, od.cpu()) and torch.equal(lh, ld.cpu())
    o_ref, l_ref = oracle.attention(q, k, v, w.scale, causal)
    compare(oh.float().numpy(), lh.numpy(), o_ref, l_ref, dtype, dtype)


def test_host_buffer_chunks_keep_the_whole_problems_item_shape():
    """A problem whose two-tile items fill more than half of the SMs runs
    two-tile items; the head chunks of fa_forward_host, each alone small enough
    for single-tile items, still run the whole problem's item shape, so the
    result is the device-buffer call's bit for bit."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, N, d = 1, 512, 64
    H = sms // 2 + 8                        # 2 items per head: more than half of the SMs
    assert "one query tile" not in fa.plan(B, H, N, d, torch.bfloat16, torch.bfloat16, False)[1]
    assert "one query tile" in fa.plan(B, H // 4, N, d, torch.bfloat16, torch.bfloat16, False)[1]
    w = synth.Workload("t", B, H, N, d, "bf16", False, seed=3200)
    q, k, v = w.inputs()
    qh, kh, vh = (torch.from_numpy(x).to(torch.bfloat16).pin_memory() for x in (q, k, v))
    oh = torch.empty(w.shape, dtype=torch.bfloat16).pin_memory()
    lh = torch.empty(w.shape[:3], dtype=torch.float32).pin_memory()
    ws = torch.empty(fa.host_workspace_size(B, H, N, d, torch.bfloat16, torch.bfloat16), dtype=torch.uint8, device="cuda")
    fa.forward_host(qh, kh, vh, oh, lh, ws, scale=w.scale)
    od, ld = fa.fa_forward(qh.cuda(), kh.cuda(), vh.cuda(), scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(oh, od.cpu()) and torch.equal(lh, ld.cpu())
    o_ref, l_ref = oracle.attention(q[:, :4], k[:, :4], v[:, :4], w.scale, False)  # the first 4 heads
    compare(oh[:, :4].float().numpy(), lh[:, :4].numpy(), o_ref, l_ref, "bf16", "bf16")


def test_host_buffer_entry_point_from_two_threads():
    """Two host threads call fa_forward_host at once on one device (the call
    releases the interpreter lock): the shared pipeline streams are taken in
    turn, and each result equals the device-buffer path bit for bit."""
    import threading
    cases = [synth.Workload("t", 2, 8, 2048, 128, "bf16", c, seed=3100 + c) for c in (0, 1)]
    bufs, errors = [], []
    for w in cases:
        q, k, v = w.inputs()
        qh, kh, vh = (torch.from_numpy(x).to(torch.bfloat16).pin_memory() for x in (q, k, v))
        oh = torch.empty(w.shape, dtype=torch.bfloat16).pin_memory()
        lh = torch.empty(w.shape[:3], dtype=torch.float32).pin_memory()
        ws = torch.empty(fa.host_workspace_size(*w.shape, torch.bfloat16, torch.bfloat16),
                         dtype=torch.uint8, device="cuda")
        bufs.append((w, qh, kh, vh, oh, lh, ws))

    def run(b):
        w, qh, kh, vh, oh, lh, ws = b
        try:
            for _ in range(4):
                fa.forward_host(qh, kh, vh, oh, lh, ws, scale=w.scale, causal=w.causal)
        except Exception as e:  # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(b,)) for b in bufs]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for w, qh, kh, vh, oh, lh, ws in bufs:
        od, ld = fa.fa_forward(qh.cuda(), kh.cuda(), vh.cuda(), scale=w.scale, causal=w.causal)
        torch.cuda.synchronize()
        assert torch.equal(oh, od.cpu()) and torch.equal(lh, ld.cpu())


def test_host_buffer_entry_point_rejects_small_workspace():
    x = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.forward_host(x, x, x, torch.empty_like(x), None, ws)
    assert e.value.status == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("B,H,N,causal", [(1, 2, 256, False), (1, 2, 100, False), (4, 32, 4096, False),
                                          (1, 2, 256, True), (1, 38, 512, False), (1, 39, 512, False)])
def test_item_shape_follows_the_fill(B, H, N, causal):
    """Unmasked problems of at most 128 query rows, or whose two-tile items
    (256 rows) would fill at most half of the SMs, run items of one query tile;
    the rest, and every causal problem, two-tile items."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    items2 = -(-N // 256) * B * H
    one = not causal and (N <= 128 or 2 * items2 <= sms)
    desc = fa.plan(B, H, N, 64, torch.bfloat16, torch.bfloat16, causal)[1]
    assert desc.startswith("tensor-core d=64")
    assert ("one query tile per item" in desc) == one, desc
