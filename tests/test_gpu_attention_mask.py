"""GPU parity of the masked attention (boolean attn_mask, bf16 tensor-core path) against the
float64 oracle: packing bit-exact; forward and backward within the bf16 bounds of the other
attention tests (max-abs 1e-2, mean-abs 1e-3, fp32 outputs and gradients), with the same
argmax rule (parity.check_argmax: the oracle's lowest index, except at near ties within
the fp32 score-error bound)."""
import numpy as np
import pytest
import torch

import oracle
import parity
import rational_softmax_attention_gb300 as ra
from rational_softmax_attention_gb300.inputs import attention_inputs

pytestmark = pytest.mark.gpu


def _np_pack(mask, words):
    """[G, R, C] bool -> [G, R, words] uint32, bit c % 32 of word c // 32."""
    G, R, C = mask.shape
    out = np.zeros((G, R, words), dtype=np.uint32)
    for c in range(C):
        out[:, :, c // 32] |= mask[:, :, c].astype(np.uint32) << np.uint32(c % 32)
    return out


@pytest.mark.parametrize("G,nq,nk", [(1, 5, 7), (2, 130, 300), (3, 256, 128)])
def test_mask_packing_is_bit_exact(G, nq, nk):
    rng = np.random.default_rng(G * 1000 + nq + nk)
    mask = rng.random((G, nq, nk)) < 0.4
    # a [G, N_Q, N_K] mask broadcasts as one mask per head of a single batch
    mq, mk, MB, MH = ra.pack_attn_mask(torch.from_numpy(mask).cuda(), 1, G, nq, nk)
    torch.cuda.synchronize()
    wq, wk = ra.lib().ra_attention_mask_words(nk), ra.lib().ra_attention_mask_words(nq)
    np.testing.assert_array_equal(mq.cpu().numpy().view(np.uint32), _np_pack(mask, wq))
    np.testing.assert_array_equal(mk.cpu().numpy().view(np.uint32), _np_pack(mask.transpose(0, 2, 1), wk))
    assert (MB, MH) == (1, G)


def _full_mask(mask, B, H):
    m = np.asarray(mask, dtype=bool)
    while m.ndim < 4:
        m = m[None]
    return np.broadcast_to(m, (B, H) + m.shape[2:])


def _check(q, k, v, do, scale, causal, mask, heads=None):
    """Masked GPU forward + backward against the oracle on the given heads."""
    qg, kg, vg, dog = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    B, H, nq, _ = q.shape
    nk = k.shape[2]
    pm = ra.pack_attn_mask(torch.from_numpy(np.ascontiguousarray(mask)).cuda(), B, H, nq, nk)
    o, rm, rs, ra_, _ = ra.ra_attention_forward(qg, kg, vg, scale=scale, causal=causal, out_dtype=torch.float32,
                                                mask=pm)
    dq, dk, dv = ra.ra_attention_backward(qg, kg, vg, o, dog, rm, rs, ra_, scale=scale, causal=causal,
                                          grad_dtype=torch.float32, mask=pm)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    full = _full_mask(mask, B, H)
    for b, h in heads or [(b, h) for b in range(B) for h in range(H)]:
        qd, kd, vd, dod = (t[b, h].double().numpy() for t in (q, k, v, do))
        allowed = full[b, h] & (np.tril(np.ones((nq, nk), dtype=bool)) if causal else True)
        S = np.where(allowed, scale * (qd @ kd.T), -np.inf)
        a_gpu = ra_[b, h].cpu().numpy().astype(np.int64)
        nd = parity.check_argmax(S, a_gpu, parity.score_error_bound(qd, kd, scale),
                                 f"masked [{b},{h}] {tuple(q.shape)} x {nk}", m_gpu=parity.f64(rm[b, h]))
        wo, wm, ws, wa = oracle.ra_attention_head_fwd(qd, kd, vd, scale, causal, mask=full[b, h])
        parity.assert_close_bf16(parity.f64(o[b, h]), wo, f"O[{b},{h}]")
        np.testing.assert_array_equal(rs[b, h].cpu().numpy() == 0, ws == 0)   # empty rows agree
        gq, gk, gv = oracle.ra_attention_head_bwd(qd, kd, vd, dod, scale, causal, argmax=a_gpu if nd else None,
                                                  mask=full[b, h])
        parity.assert_close_bf16(parity.f64(dq[b, h]), gq, f"dq[{b},{h}]")
        parity.assert_close_bf16(parity.f64(dk[b, h]), gk, f"dk[{b},{h}]")
        parity.assert_close_bf16(parity.f64(dv[b, h]), gv, f"dv[{b},{h}]")
    return o, rs, ra_, dq, dk, dv


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("nq,nk", [(128, 128), (200, 300), (300, 129)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("layout", ["shared", "per_batch", "per_head", "full"])
def test_masked_attention_matches_oracle(D, nq, nk, causal, layout):
    B, H = 2, 2
    q, k, v, do = attention_inputs(B, H, nq, nk, D, seed=nq + 3 * nk + D, sigma_qk=1.0, dtype=torch.bfloat16)
    rng = np.random.default_rng(nq * nk + D + int(causal))
    shape = {"shared": (nq, nk), "per_batch": (B, 1, nq, nk), "per_head": (1, H, nq, nk), "full": (B, H, nq, nk)}
    mask = rng.random(shape[layout]) < 0.5
    mask[..., 0] = True   # keep one key per row except where a test removes all
    _check(q, k, v, do, D ** -0.5, causal, mask)


@pytest.mark.parametrize("D,nq,nk,causal", [(128, 257, 300, True), (64, 300, 520, False), (128, 640, 700, False)])
def test_all_true_mask_equals_unmasked(D, nq, nk, causal):
    """An all-true mask (ragged at both ends) gives the unmasked results bit for bit, forward
    and backward: every item runs as an unmasked one over all N_K keys."""
    q, k, v, do = (t.cuda() for t in attention_inputs(1, 2, nq, nk, D, seed=5 + D + nq, dtype=torch.bfloat16))
    pm = ra.pack_attn_mask(torch.ones(nq, nk, dtype=torch.bool, device="cuda"), 1, 2, nq, nk)
    a = ra.ra_attention_forward(q, k, v, causal=causal, out_dtype=torch.float32, mask=pm, tile_counts=True)
    b = ra.ra_attention_forward(q, k, v, causal=causal, out_dtype=torch.float32, tile_counts=True)
    ga = ra.ra_attention_backward(q, k, v, a[0], do, *a[1:4], causal=causal, mask=pm)
    gb = ra.ra_attention_backward(q, k, v, b[0], do, *b[1:4], causal=causal)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    for x, y in zip(list(a) + list(ga), list(b) + list(gb)):
        assert torch.equal(x, y)


def test_fully_masked_rows_give_zeros():
    B, H, nq, nk = 1, 2, 160, 200
    q, k, v, do = attention_inputs(B, H, nq, nk, 64, seed=6, dtype=torch.bfloat16)
    rng = np.random.default_rng(6)
    mask = rng.random((nq, nk)) < 0.5
    mask[:, 0] = True
    empty = [0, 37, 128, 159]
    mask[empty] = False
    o, rs, ra_, dq, dk, dv = _check(q, k, v, do, 0.125, False, mask)
    assert torch.all(o[:, :, empty] == 0) and torch.all(rs[:, :, empty] == 0) and torch.all(ra_[:, :, empty] == -1)
    assert torch.all(dq[:, :, empty] == 0)


def test_key_padding_mask_skips_dead_tiles():
    """Keys past each batch's length are masked out: whole key tiles are dead, so their
    P V products are skipped and counted."""
    B, H, n = 2, 2, 640
    q, k, v, do = attention_inputs(B, H, n, n, 128, seed=7, dtype=torch.bfloat16)
    lengths = [200, 640]
    mask = np.zeros((B, 1, n, n), dtype=bool)
    for b, L in enumerate(lengths):
        mask[b, 0, :, :L] = True
    _check(q, k, v, do, 128 ** -0.5, False, mask, heads=[(0, 0), (1, 1)])
    pm = ra.pack_attn_mask(torch.from_numpy(mask).cuda(), B, H, n, n)
    _, _, _, _, counts = ra.ra_attention_forward(q.cuda(), k.cuda(), v.cuda(), tile_counts=True, mask=pm)
    torch.cuda.synchronize()
    visited, skipped = (int(c) for c in counts.tolist())
    # batch 0 (both heads): key tiles 2..4 of every query tile lie past length 200
    assert visited == B * H * 5 * 5 and skipped == H * 5 * 3


def test_autograd_with_attn_mask():
    q, k, v, do = attention_inputs(1, 2, 96, 96, 64, seed=8, dtype=torch.bfloat16)
    mask = torch.rand(96, 96, generator=torch.Generator().manual_seed(8)) < 0.6
    mask[:, 0] = True
    qg, kg, vg = (t.cuda().requires_grad_(True) for t in (q, k, v))
    out = ra.ra_attention(qg, kg, vg, attn_mask=mask.cuda(), is_causal=True)
    out.float().backward(do.cuda().float())
    torch.cuda.synchronize()
    for b in range(1):
        for h in range(2):
            qd, kd, vd, dod = (t[b, h].double().numpy() for t in (q, k, v, do))
            wo, *_ = oracle.ra_attention_head_fwd(qd, kd, vd, 0.125, True, mask=mask.numpy())
            gq, gk, gv = oracle.ra_attention_head_bwd(qd, kd, vd, dod, 0.125, True, mask=mask.numpy())
            # bf16 outputs and gradients: the fp32 bounds plus half a bf16 ulp of each value
            for name, got, want in (("O", out, wo), ("dq", qg.grad, gq), ("dk", kg.grad, gk), ("dv", vg.grad, gv)):
                g = parity.f64(got[b, h])
                assert np.all(np.abs(g - want) <= 1e-2 + 2.0 ** -8 * np.abs(want)), name


@pytest.mark.parametrize("D,nq,empty", [(64, 300, (0, 128)), (128, 600, (0, 256)), (128, 600, (256, 512))])
def test_query_tiles_with_no_allowed_key_give_zeros(D, nq, empty):
    """A mask that leaves whole query tiles (D = 64: one 128-row tile; D = 128 CTA pairs: the 256
    rows of one product) with no allowed key: every P V product of those rows is skipped, so
    their accumulator is never written, and O must still be exactly 0 there, with the rest of
    the head matching the oracle."""
    B, H, nk = 1, 2, 384
    q, k, v, do = attention_inputs(B, H, nq, nk, D, seed=D + nq, dtype=torch.bfloat16)
    rng = np.random.default_rng(D + nq)
    mask = rng.random((nq, nk)) < 0.5
    mask[:, 0] = True
    mask[empty[0]:empty[1]] = False
    o, rs, ra_, dq, dk, dv = _check(q, k, v, do, D ** -0.5, False, mask)
    lo, hi = empty
    assert torch.all(o[:, :, lo:hi] == 0) and torch.all(rs[:, :, lo:hi] == 0) and torch.all(ra_[:, :, lo:hi] == -1)
    assert torch.all(dq[:, :, lo:hi] == 0)


def _expected_tile_counts(blocks, nq, nk, causal, span):
    """(pairs in range, pairs whose P V product does not run) for a block mask: blocks[qt, kt]
    says whether query tile qt may attend to anything in key tile kt (random fill inside a live
    block, so every live block in causal range holds an allowed pair).  A product covers `span`
    consecutive query tiles and runs on key tile kt when any of them has a live block there in
    range; its pairs (one per query tile with kt in range) all count as run then."""
    nqt, nkt = -(-nq // 128), -(-nk // 128)

    def keys(qt):
        last = min(nk - 1, min(nq - 1, qt * 128 + 127)) if causal else nk - 1
        return last // 128 + 1
    visited = sum(keys(qt) for qt in range(nqt))
    ran = 0
    for p0 in range(0, nqt, span):
        tiles = range(p0, min(p0 + span, nqt))
        for kt in range(nkt):
            if any(kt < keys(qt) and blocks[qt, kt] for qt in tiles):
                ran += sum(kt < keys(qt) for qt in tiles)
    return visited, visited - ran


@pytest.mark.parametrize("D,nq,nk", [(64, 520, 700), (128, 520, 700), (128, 1024, 896)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("layout", ["per_head", "per_batch"])
def test_block_sparse_masks_leave_dead_tiles_out(D, nq, nk, causal, layout):
    """Block-sparse masks (each 128 x 128 block either fully masked or randomly half filled,
    a different block pattern per mask head): fully masked tiles are left out of both passes
    (no copy, no product), the results match the oracle, and the tile counters show exactly
    the pairs no product ran on.  With D = 128 and N_Q > 256 two query tiles share each
    product (CTA pairs), so a key tile is left out only when it is dead for both."""
    B, H = 2, 2
    q, k, v, do = attention_inputs(B, H, nq, nk, D, seed=nq + nk + D, sigma_qk=1.0, dtype=torch.bfloat16)
    rng = np.random.default_rng(nq * 7 + nk + D + int(causal))
    nqt, nkt = -(-nq // 128), -(-nk // 128)
    G = H if layout == "per_head" else B
    blocks = rng.random((G, nqt, nkt)) < 0.45
    blocks[:, :, 0] = True   # every row keeps some key
    fine = rng.random((G, nqt * 128, nkt * 128)) < 0.5
    dense = np.repeat(np.repeat(blocks, 128, axis=1), 128, axis=2) & fine
    dense = dense[:, :nq, :nk]
    dense[:, :, 0] = True
    mask = dense[None] if layout == "per_head" else dense[:, None]
    _check(q, k, v, do, D ** -0.5, causal, mask, heads=[(0, 0), (1, 1)])
    pm = ra.pack_attn_mask(torch.from_numpy(np.ascontiguousarray(mask)).cuda(), B, H, nq, nk)
    _, _, _, _, counts = ra.ra_attention_forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, tile_counts=True,
                                                 mask=pm)
    torch.cuda.synchronize()
    got = tuple(int(c) for c in counts.tolist())
    span = 2 if D == 128 and nq > 256 else 1
    want = [0, 0]
    for b in range(B):
        for h in range(H):
            vis, skip = _expected_tile_counts(blocks[h if layout == "per_head" else b], nq, nk, causal, span)
            want[0] += vis
            want[1] += skip
    assert got == tuple(want)


@pytest.mark.parametrize("D,nq,nk,causal", [(64, 520, 700, False), (128, 640, 700, True), (128, 1024, 896, False)])
def test_block_masks_with_full_dead_and_mixed_tiles(D, nq, nk, causal):
    """Blocks fully allowed (they take the unmasked code), fully masked (left out) and half
    filled (per-row mask words), ragged at both ends: forward and backward against the oracle."""
    B, H = 1, 2
    q, k, v, do = attention_inputs(B, H, nq, nk, D, seed=nq + 2 * nk + D, sigma_qk=1.0, dtype=torch.bfloat16)
    rng = np.random.default_rng(nq + nk + D)
    nqt, nkt = -(-nq // 128), -(-nk // 128)
    kind = rng.integers(0, 3, size=(H, nqt, nkt))   # 0 masked, 1 full, 2 half filled
    kind[:, :, 0] = 1
    fine = rng.random((H, nqt * 128, nkt * 128)) < 0.5
    blocks = np.repeat(np.repeat(kind, 128, axis=1), 128, axis=2)
    dense = ((blocks == 1) | ((blocks == 2) & fine))[:, :nq, :nk]
    _check(q, k, v, do, D ** -0.5, causal, dense[None])


@pytest.mark.parametrize("D,causal", [(64, False), (128, True), (128, False)])
def test_tile_maps_span_several_words(D, causal):
    """More than 32 tiles each way (4264 rows and keys: 34 tiles), so every role's walk over
    the tile maps crosses a 32-tile word, and (causal) the dK/dV kernel's walk starts inside a
    word: a block mask, forward and backward of one whole head against the oracle, and the
    exact count of tiles no product ran on."""
    B, H, n = 1, 1, 34 * 128 - 88
    q, k, v, do = attention_inputs(B, H, n, n, D, seed=4000 + D + int(causal), sigma_qk=1.0, dtype=torch.bfloat16)
    rng = np.random.default_rng(4000 + D)
    nt = -(-n // 128)
    blocks = rng.random((nt, nt)) < 0.35
    blocks[:, 0] = True
    blocks[:, 33] = rng.random(nt) < 0.5    # the second word's tiles
    fine = rng.random((nt * 128, nt * 128)) < 0.6
    dense = (np.repeat(np.repeat(blocks, 128, axis=0), 128, axis=1) & fine)[:n, :n]
    dense[:, 0] = True
    _check(q, k, v, do, D ** -0.5, causal, dense)
    pm = ra.pack_attn_mask(torch.from_numpy(dense).cuda(), B, H, n, n)
    _, _, _, _, counts = ra.ra_attention_forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, tile_counts=True,
                                                 mask=pm)
    torch.cuda.synchronize()
    span = 2 if D == 128 and n > 256 else 1
    assert tuple(int(c) for c in counts.tolist()) == _expected_tile_counts(blocks, n, n, causal, span)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L", [256, 200])
def test_key_padding_equals_truncated_keys(D, causal, L):
    """Keys from L on masked for every query give, bit for bit, the results of the same call
    on the first L keys alone (and zero dK, dV past L): the key tiles wholly below L are
    allowed whole (no mask words read: the unmasked arithmetic), the tiles wholly past L are
    left out, and a tile L falls inside takes the per-row mask words, whose clear bits give
    the exact zeros a ragged N_K gives.  640 query rows: D = 128 runs as CTA pairs."""
    B, H, n = 1, 2, 640
    q, k, v, do = (t.cuda() for t in attention_inputs(B, H, n, n, D, seed=6000 + D + L + int(causal), sigma_qk=1.0,
                                                      dtype=torch.bfloat16))
    pm = ra.pack_attn_mask((torch.arange(n, device="cuda") < L)[None, :].expand(n, n), B, H, n, n)
    kt, vt = k[:, :, :L].contiguous(), v[:, :, :L].contiguous()
    om, rmm, rsm, ram, _ = ra.ra_attention_forward(q, k, v, causal=causal, out_dtype=torch.float32, mask=pm)
    ot, rmt, rst, rat, _ = ra.ra_attention_forward(q, kt, vt, causal=causal, out_dtype=torch.float32)
    gm = ra.ra_attention_backward(q, k, v, om, do, rmm, rsm, ram, causal=causal, mask=pm)
    gt = ra.ra_attention_backward(q, kt, vt, ot, do, rmt, rst, rat, causal=causal)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    for name, a, b in (("o", om, ot), ("row_m", rmm, rmt), ("row_s", rsm, rst), ("row_arg", ram, rat),
                       ("dq", gm[0], gt[0]), ("dk", gm[1][:, :, :L], gt[1]), ("dv", gm[2][:, :, :L], gt[2])):
        assert torch.equal(a, b), name
    assert torch.all(gm[1][:, :, L:] == 0) and torch.all(gm[2][:, :, L:] == 0)
    # the key tiles past L count as pairs no product ran on, as in any masked call
    _, _, _, _, counts = ra.ra_attention_forward(q, k, v, causal=causal, mask=pm, tile_counts=True)
    torch.cuda.synchronize()
    nt = -(-n // 128)
    blocks = np.array([[kt * 128 < L for kt in range(nt)] for _ in range(nt)])
    span = 2 if D == 128 and n > 256 else 1
    vis, skip = _expected_tile_counts(blocks, n, n, causal, span)   # per head
    assert tuple(int(c) for c in counts.tolist()) == (B * H * vis, B * H * skip)


@pytest.mark.parametrize("D,n,causal", [(64, 600, False), (128, 640, False), (128, 600, True)])
def test_staircase_mask_query_tiles_over_their_own_key_prefix(D, n, causal):
    """Query tile qt may see keys 0 .. 128 (qt + 1) - 1 (a prefix per query tile, ragged at
    the end): every query tile's map row is a plain run of its own length, so the dQ kernel
    runs each one as an unmasked one over its own key prefix, while a forward item (two or
    four query tiles of different lengths) and a key tile (dead for the query tiles before
    it) keep the masked code.  Forward and backward against the oracle."""
    B, H = 1, 2
    q, k, v, do = attention_inputs(B, H, n, n, D, seed=7000 + D + n + int(causal), sigma_qk=1.0, dtype=torch.bfloat16)
    rows, cols = np.arange(n)[:, None], np.arange(n)[None, :]
    mask = cols < 128 * (rows // 128 + 1)
    _check(q, k, v, do, D ** -0.5, causal, mask)
