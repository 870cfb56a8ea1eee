"""GPU parity of cross-attention (Nq != Nkv) and of dit_attn_fwd_masked (a
general (B, T, T) bit mask, the pad-row rule, empty rows) against the oracle,
with the same tolerances as the unmasked kernel (tests/parity.py)."""
import numpy as np
import pytest
import torch

import oracle
from dit_long_sequence_gb300 import workloads as wl

from parity import compare, gather_rows, host_bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def dl():
    import dit_long_sequence_gb300 as m
    return m


def _full(O, L):
    return O.to(torch.float64).permute(0, 2, 1, 3).cpu().numpy(), L.double().cpu().numpy()


@pytest.mark.parametrize("B,Nq,Nkv,H,D", [(1, 300, 77, 2, 128), (2, 1000, 257, 3, 64), (1, 130, 2048, 2, 128),
                                          (1, 513, 1, 1, 128)])
def test_cross_attention(dl, B, Nq, Nkv, H, D):
    q, k, v, _ = wl.make_qkv(B, Nq, H, D, seed=Nq + Nkv, device=DEV, Nkv=Nkv)
    O, L = dl.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    Or, Lr = oracle.attn(host_bits(q), host_bits(k), host_bits(v))
    compare(*_full(O, L), Or.transpose(0, 2, 1, 3), Lr)


def test_cross_attention_cosmos_text_sampled(dl):
    """Cosmos-3-Nano-shaped video queries (2 x 44,160, 16 heads) over the
    2,992-token text path."""
    B, Nq, Nkv, H, D = 2, 44160, 2992, 16, 128
    q, k, v, _ = wl.make_qkv(B, Nq, H, D, seed=12, device=DEV, Nkv=Nkv)
    O, L = dl.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    rows = wl.sample_rows(B, H, Nq, 16, 12)
    Or, Lr = oracle.attn(host_bits(q), host_bits(k), host_bits(v), rows=rows)
    compare(*gather_rows(O, L, rows), Or, Lr)


@pytest.mark.parametrize("B,Nq,Nkv,kvl,H,D,density,rows", [
    (1, 700, 300, 290, 2, 128, 0.3, 700),     # more queries than keys, ragged key tile
    (2, 130, 2048, 2000, 2, 64, 0.05, 100),   # few queries over many keys, some rows unmasked
    (1, 2048, 4200, 4100, 3, 128, 0.5, 2048), # one partial wave, split over key ranges by the default workspace
])
def test_general_mask_on_cross_attention(dl, B, Nq, Nkv, kvl, H, D, density, rows):
    """A general mask with Nq != Nkv (video queries over a shorter or longer K/V):
    bit j of row i allows key j, rows >= mask_rows attend every valid key."""
    q, k, v, _ = wl.make_qkv(B, Nq, H, D, seed=Nq + 7 * Nkv, device=DEV, Nkv=Nkv)
    g = torch.Generator().manual_seed(Nq + Nkv)
    m = torch.rand((B, rows, kvl), generator=g) < density
    m[:, 0] = False                                    # a row with no allowed key
    bits = wl.pack_mask_bits(m).to(DEV)
    O, L = dl.attn_fwd_masked(q, k, v, bits, mask_rows=rows, key_valid_len=kvl)
    torch.cuda.synchronize()
    allow = np.ones((B, Nq, kvl), dtype=bool)
    allow[:, :rows] = m.numpy()
    Or, Lr = oracle.attn(host_bits(q), host_bits(k), host_bits(v), key_valid_len=kvl, allow=allow)
    compare(*_full(O, L), Or.transpose(0, 2, 1, 3), Lr)
    assert torch.all(O[:, 0] == 0) and torch.all(torch.isneginf(L[:, :, 0]))


def _masked_case(dl, B, T, Tp, H, D, density, seed, mask_rows=None, out_dtype=torch.float32, empty_rows=()):
    q, k, v, _ = wl.make_qkv(B, Tp, H, D, seed=seed, device=DEV)
    g = torch.Generator().manual_seed(seed)
    m = torch.rand((B, T, T), generator=g) < density
    for (bb, ii) in empty_rows:
        m[bb, ii] = False
    bits = wl.pack_mask_bits(m).to(DEV)
    O, L = dl.attn_fwd_masked(q, k, v, bits, mask_rows=T if mask_rows is None else mask_rows, key_valid_len=T,
                              out_dtype=out_dtype)
    torch.cuda.synchronize()
    allow = oracle.expand_mask(m.numpy(), Tp)
    Or, Lr = oracle.attn(host_bits(q), host_bits(k), host_bits(v), key_valid_len=T, allow=allow)
    return O, L, Or, Lr


@pytest.mark.parametrize("B,T,Tp,H,D,density", [(1, 300, 300, 2, 128, 0.5), (2, 700, 768, 2, 64, 0.1),
                                                (1, 1000, 1024, 1, 128, 0.9), (1, 129, 256, 2, 128, 0.02)])
def test_general_mask_with_padding_rule(dl, B, T, Tp, H, D, density):
    O, L, Or, Lr = _masked_case(dl, B, T, Tp, H, D, density, seed=T + Tp)
    compare(*_full(O, L), Or.transpose(0, 2, 1, 3), Lr)


def test_empty_rows_and_rows_empty_in_early_tiles(dl):
    """Rows with no allowed key give O = 0, LSE = -inf; rows whose first allowed
    key lies several tiles in exercise the m = -inf path and the rescale."""
    B, T, Tp, H, D = 1, 600, 640, 2, 128
    q, k, v, _ = wl.make_qkv(B, Tp, H, D, seed=4, device=DEV)
    m = torch.rand((B, T, T), generator=torch.Generator().manual_seed(4)) < 0.3
    m[0, 3] = False                     # empty
    m[0, 10, :400] = False              # nothing allowed in the first three key tiles
    m[0, 11, :] = False
    m[0, 11, 599] = True                # only the last key
    bits = wl.pack_mask_bits(m).to(DEV)
    O, L = dl.attn_fwd_masked(q, k, v, bits, key_valid_len=T, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    Or, Lr = oracle.attn(host_bits(q), host_bits(k), host_bits(v), key_valid_len=T,
                         allow=oracle.expand_mask(m.numpy(), Tp))
    compare(*_full(O, L), Or.transpose(0, 2, 1, 3), Lr)
    assert torch.all(O[0, 3] == 0) and torch.all(torch.isneginf(L[0, :, 3]))


def test_mask_shared_across_batch_and_no_mask_rows(dl):
    B, T, H, D = 2, 384, 2, 64
    q, k, v, _ = wl.make_qkv(B, T, H, D, seed=6, device=DEV)
    m = torch.rand((1, T, T), generator=torch.Generator().manual_seed(6)) < 0.4
    bits = wl.pack_mask_bits(m).to(DEV)
    O, L = dl.attn_fwd_masked(q, k, v, bits, key_valid_len=T)      # one mask for both batches
    O0, L0 = dl.attn_fwd_masked(q, k, v, bits, mask_rows=0)        # mask unread: plain attention
    P0, M0 = dl.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(O0, P0) and torch.equal(L0, M0)
    allow = np.broadcast_to(m.numpy(), (B, T, T)).copy()
    Or, Lr = oracle.attn(host_bits(q), host_bits(k), host_bits(v), allow=allow)
    compare(*_full(O, L), Or.transpose(0, 2, 1, 3), Lr)


def _ltx_mask_rows(rows: np.ndarray, T: int) -> np.ndarray:
    """Rows of a user mask over T = 24,200 valid tokens: frame-local blocks of
    1,512 tokens plus pseudo-random long-range links (a fixed hash, ~5%)."""
    cols = np.arange(T, dtype=np.int64)
    r = rows.astype(np.int64)[:, None]
    same_frame = (r // 1512) == (cols[None, :] // 1512)
    link = ((r * 1103515245 + cols[None, :] * 12345 + 7) >> 9) % 20 == 0
    return same_frame | link


@pytest.mark.slow
def test_masked_ltx_sized_sampled_rows(dl):
    """LTX-2-shaped padded sequence (24,200 valid of 24,576) with a user mask
    over the valid tokens; sampled rows, pad rows included."""
    B, T, Tp, H, D = 1, 24200, 24576, 8, 128
    q, k, v, _ = wl.make_qkv(B, Tp, H, D, seed=31, device=DEV)
    words = np.zeros((1, T, 4 * ((T + 127) // 128)), dtype=np.int32)
    for r0 in range(0, T, 2048):
        rr = np.arange(r0, min(T, r0 + 2048))
        words[0, r0:r0 + rr.size] = wl.pack_mask_bits(_ltx_mask_rows(rr, T)[None]).numpy()[0]
    bits = torch.from_numpy(words).to(DEV)
    O, L = dl.attn_fwd_masked(q, k, v, bits, key_valid_len=T)
    torch.cuda.synchronize()
    sel = np.sort(np.random.default_rng(31).choice(Tp, 24, replace=False)).astype(np.int32)
    sel[-1] = Tp - 1
    rows = np.broadcast_to(sel, (B, H, sel.size)).copy()
    allow = np.zeros((B, Tp, T), dtype=bool)
    valid = sel[sel < T]
    allow[0, valid] = _ltx_mask_rows(valid, T)
    allow[0, sel[sel >= T]] = True
    Or, Lr = oracle.attn(host_bits(q), host_bits(k), host_bits(v), key_valid_len=T, allow=allow, rows=rows)
    compare(*gather_rows(O, L, rows), Or, Lr)


@pytest.mark.parametrize("skip", [True, False])
def test_block_local_mask_skips_empty_tiles(dl, skip):
    """Frame-local blocks: most (256-row block, 128-key tile) pairs are empty and,
    with the workspace, skipped; a whole 256-row block with no allowed key
    (a CTA with nothing to do) ends with O = 0, LSE = -inf; pad rows past
    mask_rows attend every valid key.  Same results with and without skipping."""
    B, T, Tp, H, D = 2, 3000, 3072, 2, 128
    q, k, v, _ = wl.make_qkv(B, Tp, H, D, seed=41, device=DEV)
    idx = torch.arange(T)
    m = (idx[:, None] // 400) == (idx[None, :] // 400)
    m = m[None].repeat(B, 1, 1)
    m[1, 512:768] = False                      # one whole query block attends nothing
    bits = wl.pack_mask_bits(m).to(DEV)
    O, L = dl.attn_fwd_masked(q, k, v, bits, key_valid_len=T, skip_empty_tiles=skip)
    torch.cuda.synchronize()
    Or, Lr = oracle.attn(host_bits(q), host_bits(k), host_bits(v), key_valid_len=T,
                         allow=oracle.expand_mask(m.numpy(), Tp))
    compare(*_full(O, L), Or.transpose(0, 2, 1, 3), Lr)
    assert torch.all(O[1, 512:768] == 0) and torch.all(torch.isneginf(L[1, :, 512:768]))


def test_skipping_matches_full_walk_on_random_sparse_mask(dl):
    B, T, H, D = 1, 2048, 2, 64
    q, k, v, _ = wl.make_qkv(B, T, H, D, seed=43, device=DEV)
    g = torch.Generator().manual_seed(43)
    # sparse blocks of 128 x 128 kept at random, others empty
    keep = torch.rand((T // 128, T // 128), generator=g) < 0.2
    m = keep.repeat_interleave(128, 0).repeat_interleave(128, 1)[None]
    bits = wl.pack_mask_bits(m).to(DEV)
    O1, L1 = dl.attn_fwd_masked(q, k, v, bits, skip_empty_tiles=True)
    O0, L0 = dl.attn_fwd_masked(q, k, v, bits, skip_empty_tiles=False)
    torch.cuda.synchronize()
    Or, Lr = oracle.attn(host_bits(q), host_bits(k), host_bits(v), allow=m.numpy())
    compare(*_full(O1, L1), Or.transpose(0, 2, 1, 3), Lr)
    compare(*_full(O0, L0), Or.transpose(0, 2, 1, 3), Lr)
