"""GPU parity of dit_attn_fwd (through the C ABI) against the fp64 oracle.

Small cases are compared element by element on every row; they span several
256-row query blocks and 128-key tiles with ragged tails in both.  The
model-shaped workloads are compared on >= 1024 sampled query rows per head
against all keys, in the launch configuration the benchmark times.
"""
import math

import numpy as np
import pytest
import torch

from dit_long_sequence_gb300 import workloads as wl
import parity

pytestmark = pytest.mark.gpu


def _dev():
    return torch.device("cuda:0")


def _attn(q, k, v, **kw):
    import dit_long_sequence_gb300 as dl
    return dl.attn_fwd(q, k, v, **kw)


@pytest.mark.parametrize("B,Nq,Nkv,H,D,kvl,seed", [
    (1, 1024, 1024, 2, 64, None, 0),      # the tiny workload, whole
    (1, 256, 256, 1, 128, None, 1),       # exactly one block, two key tiles
    (1, 300, 300, 2, 128, None, 2),       # ragged query block and key tile
    (2, 257, 383, 3, 64, None, 3),        # cross lengths, D = 64
    (1, 520, 700, 2, 128, 555, 4),        # key mask inside a tile
    (1, 129, 260, 1, 128, 256, 5),        # mask exactly on a tile edge
    (1, 64, 300, 2, 128, 1, 6),           # one valid key
    (1, 1, 1, 1, 128, None, 7),           # single query, single key
    (3, 700, 129, 2, 64, None, 8),        # one key past a tile
])
def test_attn_matches_oracle_small(B, Nq, Nkv, H, D, kvl, seed):
    q, k, v, _ = wl.make_qkv(B, Nq, H, D, seed, device=_dev(), Nkv=Nkv)
    O, L = _attn(q, k, v, key_valid_len=kvl)
    torch.cuda.synchronize()
    Or, Lr = parity.oracle_full(q, k, v, key_valid_len=kvl)
    parity.compare(O.double().cpu().numpy(), L.double().cpu().numpy(), Or, Lr, head_axes=(0, 2))


def test_fused_strided_views_and_bf16_out():
    B, N, H, D = 2, 600, 4, 128
    q, k, v, buf = wl.make_qkv(B, N, H, D, seed=9, device=_dev(), fused=True)
    assert q.stride(1) == 3 * H * D
    O, L = _attn(q, k, v)
    Ob, Lb = _attn(q, k, v, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    Or, Lr = parity.oracle_full(q, k, v)
    parity.compare(O.double().cpu().numpy(), L.double().cpu().numpy(), Or, Lr, head_axes=(0, 2))
    # bf16 output only adds its own rounding (<= 2^-9 relative)
    parity.compare(Ob.double().cpu().numpy(), Lb.double().cpu().numpy(), Or, Lr, head_axes=(0, 2))
    assert torch.equal(L, Lb)


def test_strided_output():
    B, N, H, D = 1, 384, 2, 128
    q, k, v, _ = wl.make_qkv(B, N, H, D, seed=10, device=_dev())
    big = torch.full((B, N, H, 2 * D), float("nan"), device=_dev())
    out = big[..., :D]                     # row stride 2*D, not contiguous
    O, L = _attn(q, k, v, out=out)
    torch.cuda.synchronize()
    assert torch.isnan(big[..., D:]).all(), "wrote outside the output view"
    Or, Lr = parity.oracle_full(q, k, v)
    parity.compare(O.double().cpu().numpy(), L.double().cpu().numpy(), Or, Lr, head_axes=(0, 2))


def test_peaky_attention_large_outputs():
    # Q and K share a strong rank-1 component: attention concentrates on few keys
    # and |O| ~ 1, so the absolute gates are tight relative to the values.
    B, N, H, D = 1, 640, 2, 128
    g = wl.generator(_dev(), 11)
    base = torch.randn(B, N, H, D, generator=g, device=_dev())
    u = torch.randn(1, 1, H, D, generator=g, device=_dev())
    w = torch.randn(B, N, H, 1, generator=g, device=_dev())
    q = (0.3 * base + 2.0 * u).to(torch.bfloat16)
    k = (0.3 * torch.randn(B, N, H, D, generator=g, device=_dev()) + 2.0 * w * u).to(torch.bfloat16)
    v = torch.randn(B, N, H, D, generator=g, device=_dev()).to(torch.bfloat16)
    O, L = _attn(q, k, v)
    torch.cuda.synchronize()
    Or, Lr = parity.oracle_full(q, k, v)
    assert np.abs(Or).max() > 0.5
    parity.compare(O.double().cpu().numpy(), L.double().cpu().numpy(), Or, Lr, head_axes=(0, 2))


@pytest.mark.parametrize("D", [64, 128])
def test_large_score_jumps_exercise_the_rescale_paths(D):
    # Key tiles after the first hold scores far above its max: key 200 lifts P to
    # about 2^23 (kept without a rescale), keys 450 and 600 push the row sum past
    # 2^39 (the running max moves twice).  The oracle is exact for all of them.
    B, N, H = 1, 640, 2
    g = wl.generator(_dev(), 21)
    q = torch.randn(B, N, H, D, generator=g, device=_dev()) * 0.1 + 0.5
    k = torch.randn(B, N, H, D, generator=g, device=_dev()) * 0.1
    v = torch.randn(B, N, H, D, generator=g, device=_dev())
    scale = 8.0 / D        # 64-channel dot products of 0.5 * c land near 8c/D * 32 = 4c at D = 64
    k[:, 200] += 4.0 * (64.0 / D)
    k[:, 450] += 9.0 * (64.0 / D)
    k[:, 600] += 20.0 * (64.0 / D)
    q, k, v = (x.to(torch.bfloat16) for x in (q, k, v))
    O, L = _attn(q, k, v, scale=scale)
    torch.cuda.synchronize()
    Or, Lr = parity.oracle_full(q, k, v, scale=scale)
    parity.compare(O.double().cpu().numpy(), L.double().cpu().numpy(), Or, Lr, head_axes=(0, 2))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("masked", [False, True])
def test_score_jumps_by_warp_exercise_every_rescale_order(D, masked):
    # Each 32-row warp of queries is tied to one of four keys: channel c of
    # warp w's rows (c = w mod 4) is raised, and key_c carries a large value in
    # channel c.  Those rows see their scores jump by ~60 in log2 units at key_c,
    # far past the 2^39 row-sum limit, while the other warps' rows barely move.
    # key_0 and key_2 sit in the second 64-key half of their tile and key_1 and
    # key_3 in the first (the softmax takes a tile's scores in two halves), so
    # the rescale is triggered from either half, in some warps of a query tile
    # while the others take none.
    B, N, H = 1, 1024, 2
    g = wl.generator(_dev(), 22)
    q = torch.randn(B, N, H, D, generator=g, device=_dev()) * 0.5
    k = torch.randn(B, N, H, D, generator=g, device=_dev()) * 0.5
    v = torch.randn(B, N, H, D, generator=g, device=_dev())
    keys = (200, 300, 470, 530)      # (tile, key within the tile): (1, 72), (2, 44), (3, 86), (4, 18)
    rows = torch.arange(N, device=_dev())
    for c, key in enumerate(keys):
        q[:, (rows // 32) % 4 == c, :, c] += 6.0
        k[:, key, :, c] += 7.0 * math.sqrt(D)
    q, k, v = (x.to(torch.bfloat16) for x in (q, k, v))
    if masked:
        import dit_long_sequence_gb300 as dl
        allow = torch.ones((1, N, N), dtype=torch.bool)
        allow[0, ::7, 100:260] = False       # some rows miss key 200
        bits = wl.pack_mask_bits(allow).to(_dev())
        O, L = dl.attn_fwd_masked(q, k, v, bits)
    else:
        O, L = _attn(q, k, v)
    torch.cuda.synchronize()
    if masked:
        import oracle
        Or, Lr = oracle.attn(parity.host_bits(q), parity.host_bits(k), parity.host_bits(v),
                             allow=oracle.expand_mask(allow.numpy(), N))
    else:
        Or, Lr = parity.oracle_full(q, k, v)
    # the jumps really are large: nearly every row's LSE sits more than 27
    # (2^39 in log2 units) above the ln N that keys without a jump would give
    assert np.mean(Lr > np.log(N) + 27.0) > 0.9
    parity.compare(O.double().cpu().numpy(), L.double().cpu().numpy(), Or, Lr, head_axes=(0, 2))


def test_pad_keys_never_read_and_deterministic():
    B, N, H, D, kvl = 1, 700, 2, 128, 515
    q, k, v, _ = wl.make_qkv(B, N, H, D, seed=12, device=_dev())
    O1, L1 = _attn(q, k, v, key_valid_len=kvl)
    O1b, L1b = _attn(q, k, v, key_valid_len=kvl)
    k2, v2 = k.clone(), v.clone()
    k2[:, kvl:] = float("inf")
    v2[:, kvl:] = float("nan")
    O2, L2 = _attn(q, k2, v2, key_valid_len=kvl)
    torch.cuda.synchronize()
    assert torch.equal(O1, O1b) and torch.equal(L1, L1b), "not run-to-run deterministic"
    assert torch.equal(O1, O2) and torch.equal(L1, L2), "pad keys changed the result"


def test_zero_valid_keys():
    B, N, H, D = 1, 300, 2, 128
    q, k, v, _ = wl.make_qkv(B, N, H, D, seed=13, device=_dev())
    O, L = _attn(q, k, v, key_valid_len=0)
    torch.cuda.synchronize()
    assert (O == 0).all() and torch.isneginf(L).all()


def test_scale_is_honoured():
    B, N, H, D = 1, 256, 2, 64
    q, k, v, _ = wl.make_qkv(B, N, H, D, seed=14, device=_dev())
    for scale in (0.01, 0.3):
        O, L = _attn(q, k, v, scale=scale)
        torch.cuda.synchronize()
        Or, Lr = parity.oracle_full(q, k, v, scale=scale)
        parity.compare(O.double().cpu().numpy(), L.double().cpu().numpy(), Or, Lr, head_axes=(0, 2))


def test_watchdog_clean_after_runs():
    import dit_long_sequence_gb300 as dl
    rc, info = dl.check_watchdog()
    assert rc == 0, info


def _sampled_check(w, rows_per_head=1024):
    """The workload in the benchmark's launch configuration: dit_attn_fwd_ws,
    whose last partial wave of work items runs as key-range pieces; the sample
    includes the first split item's edge rows."""
    import dit_long_sequence_gb300 as dl
    q, k, v, buf = wl.make_workload_inputs(w, device=_dev())
    O, L = dl.attn_fwd_ws(q, k, v, key_valid_len=w.key_valid_len)
    torch.cuda.synchronize()
    must = [w.N - 80, w.N - 1]
    if w.key_valid_len is not None:
        must += [w.key_valid_len - 1, w.key_valid_len, w.N - 1]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nqb = (w.N + 255) // 256
    tail = (w.B * w.H * nqb) % sms
    if tail:
        qb0 = (w.B * w.H * nqb - tail) % nqb      # block of the first split item
        must += [qb0 * 256, qb0 * 256 + 127, qb0 * 256 + 128, min(w.N - 1, qb0 * 256 + 255)]
    rows = wl.sample_rows(w.B, w.H, w.N, rows_per_head, seed=w.seed, must=must)
    Og, Lg = parity.gather_rows(O, L, rows)
    Or, Lr = parity.oracle_rows(q, k, v, rows, key_valid_len=w.key_valid_len)
    res = parity.compare(Og, Lg, Or, Lr, head_axes=(0, 1))
    # statistical smoke check: LSE ~ ln(valid keys) + 1/2 for N(0,1) inputs
    assert abs(float(Lr.mean()) - (math.log(w.kv_len) + 0.5)) < 0.2
    return res


@pytest.mark.parametrize("name", ["ltx2_padded", "cosmos3_nano", "wan22_a14b"])
def test_workload_sampled_rows(name):
    _sampled_check(wl.WORKLOADS[name])


# ---------------------------------------------------- streaming accumulation

@pytest.mark.parametrize("bounds,D", [([0, 100, 257, 300, 512, 700], 128), ([0, 128, 129, 400], 64)])
def test_accumulate_over_key_chunks_equals_single_pass(bounds, D):
    import dit_long_sequence_gb300 as dl
    B, N, H = 1, 700 if D == 128 else 400, 2
    q, k, v, _ = wl.make_qkv(B, N, H, D, seed=15, device=_dev())
    out = torch.full((B, N, H, D), float("nan"), device=_dev())   # never read while lse = -inf
    lse = torch.full((B, H, N), float("-inf"), device=_dev())
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        dl.attn_fwd_accumulate(q, k[:, lo:hi], v[:, lo:hi], out, lse)
    dl.attn_fwd_accumulate(q, k[:, :0], v[:, :0], out, lse)          # an empty chunk changes nothing
    O1, L1 = _attn(q, k, v)
    torch.cuda.synchronize()
    assert (out - O1).abs().max().item() <= 2e-3
    assert (lse - L1).abs().max().item() <= 1e-4
    Or, Lr = parity.oracle_full(q, k, v)
    parity.compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), Or, Lr, head_axes=(0, 2))


def test_accumulate_ring_workload_sampled():
    import dit_long_sequence_gb300 as dl
    w = wl.WORKLOADS["ring9"]
    q, k, v, _ = wl.make_workload_inputs(w, device=_dev())
    cl = w.N // w.kv_chunks
    out = torch.empty(w.B, w.N, w.H, w.D, device=_dev())
    lse = torch.full((w.B, w.H, w.N), float("-inf"), device=_dev())
    for c in range(w.kv_chunks):
        dl.attn_fwd_accumulate(q, k[:, c * cl:(c + 1) * cl], v[:, c * cl:(c + 1) * cl], out, lse)
    torch.cuda.synchronize()
    rows = wl.sample_rows(w.B, w.H, w.N, 1024, seed=w.seed, must=[cl - 1, cl, w.N - 1])
    Og, Lg = parity.gather_rows(out, lse, rows)
    Or, Lr = parity.oracle_rows(q, k, v, rows)
    parity.compare(Og, Lg, Or, Lr, head_axes=(0, 1))
