"""GPU checks of dit_attn_fwd_ws: the work items of the grid's last partial
wave split over key ranges, their partial (O, LSE) merged by a second kernel.

- the plan (pieces per split item) follows its rule for this GPU's SM count;
- shapes where every item is split (f = 2, 3, 8; ragged query blocks and key
  tiles; D = 64 and 128; fp32 and bf16 output) match the fp64 oracle whole;
- items that are not split are bit-identical to dit_attn_fwd; split ones
  differ from it by the bf16 rounding of P (a piece rounds its probabilities
  against its own running max, so they round differently: about
  2^-8 * |v| / sqrt(keys) per element, a few 1e-4 at most at 8k keys; the
  LSE only by fp32 rounding);
- a NULL workspace is exactly dit_attn_fwd; a short one is refused before
  anything is enqueued;
- the LTX-2-shaped workload in the benchmark's configuration (32 items of
  head 31 split 4 ways on a 152-SM GB300) matches the oracle on sampled rows
  that include the split rows.
"""
import ctypes

import numpy as np
import pytest
import torch

from dit_long_sequence_gb300 import workloads as wl
import parity

pytestmark = pytest.mark.gpu

SPLIT_VS_SINGLE_O = 2e-3      # ~10x the largest difference seen at 8k keys
SPLIT_VS_SINGLE_LSE = 5e-5


def _dev():
    return torch.device("cuda:0")


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _plan(B, Nq, H, kvl):
    """Pieces per split item and the index of the first split item: the tail
    of items mod SMs, cut into f = min(SMs // tail, 8, key tiles // 16) ranges
    (SMs // tail raised to 2 behind whole waves) when f >= 2."""
    items = B * H * ((Nq + 255) // 256)
    tiles = (kvl + 127) // 128
    tail = items % _sms()
    if tail == 0 or tiles == 0:
        return 1, items
    f = _sms() // tail
    if items > _sms():
        f = max(f, 2)
    f = min(f, 8, tiles // 16)
    return (f, items - tail) if f >= 2 else (1, items)


def _expected_bytes(B, Nq, H, D, kvl):
    f, first = _plan(B, Nq, H, kvl)
    items = B * H * ((Nq + 255) // 256)
    pieces = (items - first) * f
    if f == 1:
        return 0
    return pieces * 256 * D * 4 + (pieces * 256 * 4 + 255) // 256 * 256


def _split_rows_mask(B, Nq, H, kvl):
    """[B, H, Nq] bool: rows that belong to split items."""
    f, first = _plan(B, Nq, H, kvl)
    nqb = (Nq + 255) // 256
    m = np.zeros((B, H, Nq), dtype=bool)
    for item in range(first, B * H * nqb):
        qb, h, b = item % nqb, (item // nqb) % H, item // nqb // H
        m[b, h, qb * 256:min(Nq, qb * 256 + 256)] = True
    return m


@pytest.mark.parametrize("shape", [
    (1, 24576, 32, 128, 24200),    # LTX-2-shaped
    (2, 44160, 16, 128, 44160),    # Cosmos-shaped
    (2, 75600, 40, 128, 75600),    # Wan-shaped
    (1, 60000, 40, 128, 300),      # 3 key tiles: too few to split
    (1, 1024, 2, 64, 1024),        # tiny: too few key tiles
    (1, 8192, 2, 128, 8000),
    (1, 2048, 2, 128, 16384),
    (1, 6400, 2, 128, 6390),
    (1, 5000, 3, 64, 5999),
])
def test_workspace_bytes_follow_the_plan(shape):
    import dit_long_sequence_gb300 as dl
    B, Nq, H, D, kvl = shape
    assert dl.attn_fwd_workspace_bytes(B, Nq, H, D, kvl) == _expected_bytes(B, Nq, H, D, kvl)


def test_plan_on_a_152_sm_gb300():
    if _sms() != 152:
        pytest.skip("plan figures for 152 SMs")
    assert _plan(1, 24576, 32, 24200) == (4, 3040)      # 3,072 items: 32 left over, split 4 ways
    assert _plan(2, 44160, 16, 44160) == (2, 5472)      # 5,536 items: 64 left over, split 2 ways
    assert _plan(2, 75600, 40, 75600) == (2, 23560)     # 120 left over, split 2 ways


def _ws_call(q, k, v, kvl, out_dtype=torch.float32, workspace="auto"):
    import dit_long_sequence_gb300 as dl
    if workspace == "auto":
        return dl.attn_fwd_ws(q, k, v, key_valid_len=kvl, out_dtype=out_dtype)
    return dl.attn_fwd_ws(q, k, v, key_valid_len=kvl, out_dtype=out_dtype, workspace=workspace)


@pytest.mark.parametrize("B,Nq,Nkv,H,D,kvl,f_152,seed", [
    (1, 8192, 8192, 2, 128, 8000, 2, 21),     # 64 items, all split in two; ragged last key tile
    (1, 2048, 16384, 2, 128, None, 8, 22),    # 16 items split 8 ways, 16 tiles per piece
    (1, 6400, 6400, 2, 128, 6390, 3, 23),     # 50 tiles in 3 uneven ranges (16, 17, 17)
    (1, 5000, 6000, 3, 64, 5999, 2, 24),      # D = 64, ragged query block (5000 = 19*256 + 136)
    (2, 4500, 4500, 2, 128, 4400, 2, 25),     # B = 2: 72 items split in two, ragged query blocks
])
def test_split_matches_oracle_whole(B, Nq, Nkv, H, D, kvl, f_152, seed):
    import dit_long_sequence_gb300 as dl
    q, k, v, _ = wl.make_qkv(B, Nq, H, D, seed, device=_dev(), Nkv=Nkv)
    kv = Nkv if kvl is None else kvl
    f, first = _plan(B, Nq, H, kv)
    if _sms() == 152:
        assert f == f_152 and first == 0
    assert dl.attn_fwd_workspace_bytes(B, Nq, H, D, kv) > 0
    O, L = _ws_call(q, k, v, kvl)
    Ob, Lb = _ws_call(q, k, v, kvl, out_dtype=torch.bfloat16)
    O1, L1 = dl.attn_fwd(q, k, v, key_valid_len=kvl)
    torch.cuda.synchronize()
    Or, Lr = parity.oracle_full(q, k, v, key_valid_len=kvl)
    parity.compare(O.double().cpu().numpy(), L.double().cpu().numpy(), Or, Lr, head_axes=(0, 2))
    parity.compare(Ob.double().cpu().numpy(), Lb.double().cpu().numpy(), Or, Lr, head_axes=(0, 2))
    assert torch.equal(L, Lb)
    # against the single pass: P's bf16 rounding (O), fp32 rounding (LSE)
    assert (O - O1).abs().max().item() <= SPLIT_VS_SINGLE_O
    assert (L - L1).abs().max().item() <= SPLIT_VS_SINGLE_LSE
    rc, info = dl.check_watchdog()
    assert rc == 0, info


def test_unsplit_items_bit_identical_and_null_workspace_is_plain():
    import dit_long_sequence_gb300 as dl
    from dit_long_sequence_gb300 import binding
    w = wl.WORKLOADS["ltx2_padded"]
    q, k, v, _ = wl.make_workload_inputs(w, device=_dev())
    O, L = dl.attn_fwd_ws(q, k, v, key_valid_len=w.key_valid_len)
    O1, L1 = dl.attn_fwd(q, k, v, key_valid_len=w.key_valid_len)
    # NULL workspace through the C ABI: the plain kernel, bit for bit
    O0 = torch.empty_like(O1)
    L0 = torch.empty_like(L1)
    st = binding.AttnStrides(binding.Strides4(*q.stride()), binding.Strides4(*k.stride()),
                             binding.Strides4(*v.stride()), binding.Strides4(*O0.stride()))
    rc = binding.raw().dit_attn_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(st), w.B, w.N, w.N,
                                       w.H, w.D, w.key_valid_len, w.scale, O0.data_ptr(), binding.DIT_F32,
                                       L0.data_ptr(), None, 0, torch.cuda.current_stream().cuda_stream)
    assert rc == binding.DIT_OK
    torch.cuda.synchronize()
    assert torch.equal(O0, O1) and torch.equal(L0, L1)
    split = torch.as_tensor(_split_rows_mask(w.B, w.N, w.H, w.kv_len), device=_dev())   # [B, H, N]
    if not split.any():
        pytest.skip("no split on this GPU for this shape")
    so = split.permute(0, 2, 1)                                                        # [B, N, H]
    assert torch.equal(O[~so], O1[~so]) and torch.equal(L[~split], L1[~split])
    assert (O[so] - O1[so]).abs().max().item() <= SPLIT_VS_SINGLE_O
    assert (L[split] - L1[split]).abs().max().item() <= SPLIT_VS_SINGLE_LSE


def test_short_workspace_refused_before_enqueue():
    import dit_long_sequence_gb300 as dl
    B, N, H, D = 1, 8192, 2, 128
    q, k, v, _ = wl.make_qkv(B, N, H, D, 25, device=_dev())
    need = dl.attn_fwd_workspace_bytes(B, N, H, D, N)
    assert need > 0
    ws = torch.empty(need - 16, dtype=torch.uint8, device=_dev())
    out = torch.full((B, N, H, D), float("nan"), device=_dev())
    lse = torch.full((B, H, N), float("nan"), device=_dev())
    with pytest.raises(dl.DitError) as e:
        dl.attn_fwd_ws(q, k, v, out=out, lse=lse, workspace=ws)
    assert e.value.status == 1        # DIT_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.isnan(out).all() and torch.isnan(lse).all()


def test_ltx_workload_sampled_rows_through_the_split():
    """The benchmark's call on the LTX-2-shaped workload: sampled rows of every
    head, with extra rows drawn from the split items."""
    import dit_long_sequence_gb300 as dl
    w = wl.WORKLOADS["ltx2_padded"]
    q, k, v, _ = wl.make_workload_inputs(w, device=_dev())
    O, L = dl.attn_fwd_ws(q, k, v, key_valid_len=w.key_valid_len)
    torch.cuda.synchronize()
    f, first = _plan(w.B, w.N, w.H, w.kv_len)
    nqb = (w.N + 255) // 256
    must = [w.key_valid_len - 1, w.key_valid_len, w.N - 1]
    if f > 1:
        # rows of the first split item and of the piece boundaries' neighbourhood
        qb0 = first % nqb
        must += [qb0 * 256, qb0 * 256 + 255, qb0 * 256 + 128]
    rows = wl.sample_rows(w.B, w.H, w.N, 1024, seed=w.seed, must=must)
    Og, Lg = parity.gather_rows(O, L, rows)
    Or, Lr = parity.oracle_rows(q, k, v, rows, key_valid_len=w.key_valid_len)
    parity.compare(Og, Lg, Or, Lr, head_axes=(0, 1))
    if f > 1:
        split = _split_rows_mask(w.B, w.N, w.H, w.kv_len)
        hit = split[np.arange(w.B)[:, None, None], np.arange(w.H)[None, :, None], rows]
        assert hit.sum() >= 256       # the split rows are well represented in the sample


# ------------------------------------------------------------------ FP8 path

def _fp8_vmax(v8) -> float:
    import oracle
    codes = np.asarray(parity.host_u8(v8))
    return float(oracle.e4m3_decode(np.array([int((codes & 0x7F).max())], dtype=np.uint8))[0])


@pytest.mark.parametrize("B,N,H,kvl,out_dtype,f_152,seed", [
    (1, 8192, 2, 8000, torch.float32, 2, 31),      # 64 items, all split in two, ragged last key tile
    (1, 8192, 2, 8000, torch.bfloat16, 2, 35),     # the same split with bf16 output
    (2, 4500, 2, 4400, torch.float32, 2, 36),      # B = 2, ragged query blocks: 72 items split in two
    (1, 2048, 2, 2000, torch.bfloat16, 0, 32),     # 16 items, 16 tiles: too few keys, no split
])
def test_fp8_split_matches_oracle_whole(B, N, H, kvl, out_dtype, f_152, seed):
    import dit_long_sequence_gb300 as dl
    import oracle
    D = 128
    qkv8 = wl.randn_e4m3((B, N, 3, H, D), seed, 64.0, _dev())
    q8, k8, v8 = dl.split_stacked_fp8(qkv8)
    desc = (1 / 64, 1 / 64, 1 / 64)
    f, first = _plan(B, N, H, kvl)
    if _sms() == 152 and f_152:
        assert f == f_152 and first == 0
    O, L = dl.attn_fwd_fp8_ws(q8, k8, v8, desc, key_valid_len=kvl, out_dtype=out_dtype)
    O1, L1 = dl.attn_fwd_fp8(q8, k8, v8, desc, key_valid_len=kvl, out_dtype=out_dtype)
    torch.cuda.synchronize()
    Oref, Lref = oracle.attn_fp8(*(parity.host_u8(t) for t in (q8, k8, v8)), scale=D ** -0.5, descale_q=desc[0],
                                 descale_k=desc[1], descale_v=desc[2], key_valid_len=kvl)
    vmax = _fp8_vmax(v8) * desc[2]
    parity.compare_fp8(O.double().permute(0, 2, 1, 3).cpu().numpy(), L.double().cpu().numpy(),
                       Oref.transpose(0, 2, 1, 3), Lref, vmax)
    # against the single pass: each is within the E4M3 bound of the oracle
    assert (O.float() - O1.float()).abs().max().item() <= 2 * (2.0 ** -4 * vmax + 1e-3)
    assert (L - L1).abs().max().item() <= SPLIT_VS_SINGLE_LSE
    if f == 1:
        assert torch.equal(O, O1) and torch.equal(L, L1)


def test_fp8_split_8_ways_matches_oracle():
    import dit_long_sequence_gb300 as dl
    import oracle
    B, N, Nkv, H, D = 1, 2048, 16384, 2, 128
    q8 = wl.randn_e4m3((B, N, H, D), 33, 64.0, _dev())
    kv8 = wl.randn_e4m3((B, Nkv, 2, H, D), 34, 64.0, _dev())
    k8, v8 = kv8[:, :, 0], kv8[:, :, 1]
    desc = (1 / 64, 1 / 64, 1 / 64)
    if _sms() == 152:
        assert _plan(B, N, H, Nkv) == (8, 0)
    O, L = dl.attn_fwd_fp8_ws(q8, k8, v8, desc)
    torch.cuda.synchronize()
    Oref, Lref = oracle.attn_fp8(*(parity.host_u8(t) for t in (q8, k8, v8)), scale=D ** -0.5, descale_q=desc[0],
                                 descale_k=desc[1], descale_v=desc[2])
    parity.compare_fp8(O.double().permute(0, 2, 1, 3).cpu().numpy(), L.double().cpu().numpy(),
                       Oref.transpose(0, 2, 1, 3), Lref, _fp8_vmax(v8) * desc[2])


def test_fp8_ltx_workload_through_the_split():
    """The benchmark's FP8 call on the LTX-2-shaped workload: unsplit items
    bit-identical to dit_attn_fwd_fp8, a NULL workspace exactly that call, and
    sampled rows of the split items (and every head) against the oracle."""
    import dit_long_sequence_gb300 as dl
    import oracle
    from dit_long_sequence_gb300 import binding
    w = wl.WORKLOADS["ltx2_padded_fp8"]
    buf = wl.randn_bf16((w.B, w.N, 3, w.H, w.D), w.seed, _dev())
    qkv8 = dl.qkv_cast_fp8(buf, wl.FP8_SCALES)
    q8, k8, v8 = dl.split_stacked_fp8(qkv8)
    desc = tuple(1.0 / s for s in wl.FP8_SCALES)
    O, L = dl.attn_fwd_fp8_ws(q8, k8, v8, desc, key_valid_len=w.key_valid_len)
    O1, L1 = dl.attn_fwd_fp8(q8, k8, v8, desc, key_valid_len=w.key_valid_len)
    O0, L0 = torch.empty_like(O1), torch.empty_like(L1)
    st = binding.AttnStrides(binding.Strides4(*q8.stride()), binding.Strides4(*k8.stride()),
                             binding.Strides4(*v8.stride()), binding.Strides4(*O0.stride()))
    rc = binding.raw().dit_attn_fwd_fp8_ws(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), ctypes.byref(st), w.B, w.N,
                                           w.N, w.H, w.D, w.key_valid_len, w.scale, *desc, O0.data_ptr(),
                                           binding.DIT_F32, L0.data_ptr(), None, 0,
                                           torch.cuda.current_stream().cuda_stream)
    assert rc == binding.DIT_OK
    torch.cuda.synchronize()
    assert torch.equal(O0, O1) and torch.equal(L0, L1)
    f, first = _plan(w.B, w.N, w.H, w.kv_len)
    split = torch.as_tensor(_split_rows_mask(w.B, w.N, w.H, w.kv_len), device=_dev())
    so = split.permute(0, 2, 1)
    assert torch.equal(O[~so], O1[~so]) and torch.equal(L[~split], L1[~split])
    must = [w.key_valid_len - 1, w.key_valid_len, w.N - 1]
    if f > 1:
        qb0 = first % ((w.N + 255) // 256)
        must += [qb0 * 256, qb0 * 256 + 255, qb0 * 256 + 128]
    rows = wl.sample_rows(w.B, w.H, w.N, 512, seed=w.seed, must=must)
    Og, Lg = parity.gather_rows(O, L, rows)
    Oref, Lref = oracle.attn_fp8(*(parity.host_u8(t) for t in (q8, k8, v8)), scale=w.scale, descale_q=desc[0],
                                 descale_k=desc[1], descale_v=desc[2], key_valid_len=w.key_valid_len, rows=rows)
    parity.compare_fp8(Og, Lg, Oref, Lref, _fp8_vmax(v8) * desc[2])


@pytest.mark.parametrize("fp8", [False, True])
def test_stream_order_covers_the_whole_call(fp8):
    """Work queued on the stream right after the call sees every output row:
    the piece launch completes only after the whole-item grid beside it, so a
    reader (a copy on the same side stream, with no host sync in between) never
    observes rows the whole-item grid has not written yet."""
    import dit_long_sequence_gb300 as dl
    w = wl.WORKLOADS["ltx2_padded"]
    side = torch.cuda.Stream()
    if fp8:
        qkv8 = wl.randn_e4m3((w.B, w.N, 3, w.H, w.D), w.seed, 64.0, _dev())
        q, k, v = dl.split_stacked_fp8(qkv8)
        d = (1 / 64, 1 / 64, 1 / 64)
        ref, ref_l = dl.attn_fwd_fp8(q, k, v, d, key_valid_len=w.key_valid_len)
        call = lambda o, l, s: dl.attn_fwd_fp8_ws(q, k, v, d, key_valid_len=w.key_valid_len, out=o, lse=l, stream=s)
    else:
        q, k, v, _ = wl.make_workload_inputs(w, device=_dev())
        ref, ref_l = dl.attn_fwd(q, k, v, key_valid_len=w.key_valid_len)
        call = lambda o, l, s: dl.attn_fwd_ws(q, k, v, key_valid_len=w.key_valid_len, out=o, lse=l, stream=s)
    torch.cuda.synchronize()
    split = torch.as_tensor(_split_rows_mask(w.B, w.N, w.H, w.kv_len), device=_dev())
    out = torch.empty_like(ref)
    lse = torch.empty_like(ref_l)
    side.wait_stream(torch.cuda.current_stream())
    for _ in range(4):
        with torch.cuda.stream(side):
            out.fill_(float("nan"))
            lse.fill_(float("nan"))
            call(out, lse, side)
            seen_o = out.clone()          # queued behind the call, no host sync in between
            seen_l = lse.clone()
        torch.cuda.synchronize()
        assert not torch.isnan(seen_o).any() and not torch.isnan(seen_l).any()
        so = split.permute(0, 2, 1)
        assert torch.equal(seen_o[~so], ref[~so]) and torch.equal(seen_l[~split], ref_l[~split])


@pytest.mark.parametrize("fp8", [False, True])
def test_split_reruns_are_bit_identical(fp8):
    """The pieces' partials are combined in a fixed order, so the split call is
    deterministic run to run, like the plain kernel."""
    import dit_long_sequence_gb300 as dl
    B, N, H, D, kvl = 1, 8192, 2, 128, 8000
    if fp8:
        q, k, v = dl.split_stacked_fp8(wl.randn_e4m3((B, N, 3, H, D), 41, 64.0, _dev()))
        run = lambda: dl.attn_fwd_fp8_ws(q, k, v, (1 / 64, 1 / 64, 1 / 64), key_valid_len=kvl)
    else:
        q, k, v, _ = wl.make_qkv(B, N, H, D, 41, device=_dev())
        run = lambda: dl.attn_fwd_ws(q, k, v, key_valid_len=kvl)
    O1, L1 = run()
    O2, L2 = run()
    torch.cuda.synchronize()
    assert dl.attn_fwd_workspace_bytes(B, N, H, D, kvl) > 0
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


# ------------------------------------------------------------ general mask
# dit_attn_fwd_masked splits the grid's last partial wave as dit_attn_fwd_ws
# does when its workspace has room past the occupancy map.  A piece's key
# range may hold no key a row may attend: its partial then has LSE = -inf and
# weight 0 in the merge, and a row with none in any piece ends with O = 0,
# LSE = -inf.

def _masked_oracle(q, k, v, m, T, Tp):
    import oracle
    return oracle.attn(parity.host_bits(q), parity.host_bits(k), parity.host_bits(v), key_valid_len=T,
                       allow=oracle.expand_mask(m.numpy(), Tp))


def _random_mask(B, T, density, seed, empty_rows=(), late_rows=()):
    g = torch.Generator().manual_seed(seed)
    m = torch.rand((B, T, T), generator=g) < density
    for bb, ii in empty_rows:
        m[bb, ii] = False
    for bb, ii, first_key in late_rows:            # no allowed key before first_key
        m[bb, ii, :first_key] = False
    return m


@pytest.mark.parametrize("B,T,Tp,H,D,f_152,first_152,seed,kind", [
    (1, 8000, 8192, 2, 128, 2, 0, 51, "random"),       # 64 items, all split in two
    (2, 4400, 4500, 2, 128, 2, 0, 52, "random"),       # B = 2, ragged query blocks
    (1, 4096, 4096, 4, 128, 2, 0, 53, "blocks"),       # block-diagonal: pieces with no allowed key
    (1, 4096, 4096, 10, 128, 2, 152, 54, "blocks"),    # 160 items: 152 whole, 8 split
])
def test_masked_split_matches_oracle_and_unsplit(B, T, Tp, H, D, f_152, first_152, seed, kind):
    import dit_long_sequence_gb300 as dl
    q, k, v, _ = wl.make_qkv(B, Tp, H, D, seed, device=_dev())
    if kind == "random":
        m = _random_mask(B, T, 0.3, seed, empty_rows=((0, 5), (B - 1, T - 1)),
                         late_rows=((0, 300, T // 2), (B - 1, 600, T - 10)))
    else:
        idx = torch.arange(T)
        m = ((idx[:, None] // 512) == (idx[None, :] // 512))[None].repeat(B, 1, 1)
        m[0, 1000] = False                          # one row attends nothing
    bits = wl.pack_mask_bits(m).to(_dev())
    f, first = _plan(B, Tp, H, T)
    if _sms() == 152:
        assert (f, first) == (f_152, first_152)
    need = dl.masked_split_workspace_bytes(B, Tp, H, D, T)
    occ = dl.masked_workspace_bytes(B, Tp, T)
    assert need == (occ + 255) // 256 * 256 + dl.attn_fwd_workspace_bytes(B, Tp, H, D, T)
    ws = torch.empty(need, dtype=torch.uint8, device=_dev())
    O, L = dl.attn_fwd_masked(q, k, v, bits, key_valid_len=T, workspace=ws)
    ws0 = torch.empty((occ + 15) // 16 * 16, dtype=torch.uint8, device=_dev())   # occupancy only: no split
    O0, L0 = dl.attn_fwd_masked(q, k, v, bits, key_valid_len=T, workspace=ws0)
    torch.cuda.synchronize()
    Or, Lr = _masked_oracle(q, k, v, m, T, Tp)
    parity.compare(O.double().permute(0, 2, 1, 3).cpu().numpy(), L.double().cpu().numpy(),
                   Or.transpose(0, 2, 1, 3), Lr)
    parity.compare(O0.double().permute(0, 2, 1, 3).cpu().numpy(), L0.double().cpu().numpy(),
                   Or.transpose(0, 2, 1, 3), Lr)
    assert torch.equal(torch.isneginf(L), torch.isneginf(L0))
    fin = torch.isfinite(L0)
    assert (O - O0).abs().max().item() <= SPLIT_VS_SINGLE_O
    assert (L[fin] - L0[fin]).abs().max().item() <= SPLIT_VS_SINGLE_LSE
    # items before the split are the unsplit kernel's, bit for bit
    split_rows = torch.from_numpy(_split_rows_mask(B, Tp, H, T)).to(_dev())   # [B, H, Nq]
    whole = ~split_rows
    assert torch.equal(L[whole], L0[whole])
    assert torch.equal(O.permute(0, 2, 1, 3)[whole], O0.permute(0, 2, 1, 3)[whole])
    if kind == "blocks":
        assert torch.all(O[0, 1000] == 0) and torch.all(torch.isneginf(L[0, :, 1000]))
    rc, info = dl.check_watchdog()
    assert rc == 0, info
