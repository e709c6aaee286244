"""Invariants and special cases that pin the oracle beyond the worked example.

* absorbed == un-absorbed scores and outputs to 1e-12 in fp64 ("Mathematical
  Prerequisites for DeepSeek-V2" sections 6-7; "From Vanilla Transformers to
  Modern LLMs -- Part 3" 3.e.2 and 3.g state the two routes agree),
* softmax rows sum to one,
* textbook single-head attention (H=1, W_UK = W_UV = I) against PyTorch's
  scaled-dot-product attention in fp64, with and without the RoPE part,
* one visible token, identical keys, empty rows,
* block-table permutation invariance, causal query slots, append placement,
* block-range pieces: merged by the log-sum-exp combine they equal the
  whole decode; a range over every block is the decode; one block against
  the brute-force softmax over its keys; the combine's weights on a case
  with known denominators.
"""

import math

import numpy as np
import pytest
import torch

from oracle import mla


def _rand_case(rng, H=3, d_h=5, d_c=7, d_r=4, seqlens=(9, 1, 13), Hq=1, bs=4):
    B = len(seqlens)
    nblk = [-(-s // bs) for s in seqlens]
    total = sum(nblk)
    perm = rng.permutation(total)
    table = np.full((B, max(nblk)), -1)
    off = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[off:off + n]
        off += n
    return dict(
        q_nope=rng.standard_normal((B, Hq, H, d_h)),
        q_rope=rng.standard_normal((B, Hq, H, d_r)),
        cache=rng.standard_normal((total, bs, d_c + d_r)),
        block_table=table,
        seqlens=np.array(seqlens),
        W_UK=rng.standard_normal((H, d_h, d_c)) / math.sqrt(d_c),
        W_UV=rng.standard_normal((H, d_h, d_c)) / math.sqrt(d_c),
        Hq=Hq,
    )


def _decode(case, **kw):
    return mla.mla_decode(case["q_nope"], case["q_rope"], case["cache"], case["block_table"],
                          case["seqlens"], case["W_UK"], case["W_UV"], case["Hq"], **kw)


@pytest.mark.parametrize("seed", range(4))
def test_absorbed_equals_unabsorbed(seed):
    rng = np.random.default_rng(seed)
    case = _rand_case(rng)
    d_c = case["W_UK"].shape[2]
    scale = mla.default_scale(case["W_UK"].shape[1], case["q_rope"].shape[3])
    out, o_lat, lse = _decode(case)
    q_lat = mla.absorb_query(case["q_nope"], case["W_UK"])
    for b in range(len(case["seqlens"])):
        n = int(case["seqlens"][b])
        rows = mla.gather_sequence(case["cache"], case["block_table"][b], n)
        for h in range(case["W_UK"].shape[0]):
            r = mla.attention_row(case["q_nope"][b, 0, h], case["q_rope"][b, 0, h], rows,
                                  case["W_UK"][h], case["W_UV"][h], scale, d_c)
            s_abs = mla.absorbed_scores(q_lat[b, 0, h], case["q_rope"][b, 0, h], rows, d_c, scale)
            assert np.max(np.abs(s_abs - r["s"])) < 1e-12
            p = mla.softmax(s_abs)
            assert abs(p.sum() - 1.0) < 1e-15 * max(n, 1) * 4
            assert np.max(np.abs(p - r["p"])) < 1e-12
            o_abs = p @ rows[:, :d_c]
            assert np.max(np.abs(o_abs - o_lat[b, 0, h])) < 1e-12
    # value absorption: out == W_UV o_lat
    assert np.max(np.abs(mla.out_proj(o_lat, case["W_UV"]) - out)) < 1e-12


@pytest.mark.parametrize("d_r", [0, 6])
def test_textbook_single_head(d_r):
    """H=1, d_c=d_h, W_UK=W_UV=I reduces to textbook attention with k=[c;k_R], v=c."""
    rng = np.random.default_rng(10 + d_r)
    n, d = 11, 8
    rows = rng.standard_normal((n, d + d_r))
    q_nope = rng.standard_normal(d)
    q_rope = rng.standard_normal(d_r)
    scale = 0.37
    eye = np.eye(d)
    r = mla.attention_row(q_nope, q_rope, rows, eye, eye, scale, d)
    q = torch.tensor(np.concatenate([q_nope, q_rope]))[None, None, None, :]
    k = torch.tensor(rows)[None, None]
    v = torch.tensor(rows[:, :d])[None, None]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)
    assert np.max(np.abs(r["out"] - ref[0, 0, 0].numpy())) < 1e-12
    assert np.max(np.abs(r["o_lat"] - ref[0, 0, 0].numpy())) < 1e-12
    logits = (torch.tensor(rows) @ q[0, 0, 0]) * scale
    assert abs(r["lse"] - torch.logsumexp(logits, 0).item()) < 1e-12


def test_single_visible_token():
    rng = np.random.default_rng(3)
    case = _rand_case(rng, seqlens=(1,))
    out, o_lat, lse = _decode(case)
    row = case["cache"][case["block_table"][0, 0], 0]
    d_c = case["W_UK"].shape[2]
    scale = mla.default_scale(case["W_UK"].shape[1], case["q_rope"].shape[3])
    for h in range(case["W_UK"].shape[0]):
        assert np.max(np.abs(o_lat[0, 0, h] - row[:d_c])) < 1e-15
        s0 = (case["W_UK"][h] @ row[:d_c]) @ case["q_nope"][0, 0, h] + row[d_c:] @ case["q_rope"][0, 0, h]
        assert abs(lse[0, 0, h] - s0 * scale) < 1e-12
        assert np.max(np.abs(out[0, 0, h] - case["W_UV"][h] @ row[:d_c])) < 1e-12


def test_identical_keys_average():
    rng = np.random.default_rng(4)
    case = _rand_case(rng, seqlens=(10,))
    row = rng.standard_normal(case["cache"].shape[2])
    case["cache"][:] = row
    out, o_lat, lse = _decode(case)
    d_c = case["W_UK"].shape[2]
    scale = mla.default_scale(case["W_UK"].shape[1], case["q_rope"].shape[3])
    for h in range(case["W_UK"].shape[0]):
        assert np.max(np.abs(o_lat[0, 0, h] - row[:d_c])) < 1e-12
        s = ((case["W_UK"][h] @ row[:d_c]) @ case["q_nope"][0, 0, h]
             + row[d_c:] @ case["q_rope"][0, 0, h]) * scale
        assert abs(lse[0, 0, h] - (s + math.log(10))) < 1e-12


def test_empty_rows():
    """seqlen < Hq leaves the early slots with nothing to attend to."""
    rng = np.random.default_rng(5)
    case = _rand_case(rng, seqlens=(1, 3), Hq=2)
    out, o_lat, lse = _decode(case)
    assert np.all(lse[0, 0] == -np.inf)
    assert np.all(o_lat[0, 0] == 0) and np.all(out[0, 0] == 0)
    assert np.all(np.isfinite(lse[0, 1])) and np.all(np.isfinite(lse[1]))


def test_causal_query_slots():
    """Slot i of Hq=2 sees one token fewer than slot i+1: slot 0 equals an
    Hq=1 step on seqlen - 1 with the same data."""
    rng = np.random.default_rng(6)
    case = _rand_case(rng, seqlens=(9, 13, 5), Hq=2)
    out, o_lat, lse = _decode(case)
    one = dict(case)
    one["Hq"] = 1
    one["q_nope"] = case["q_nope"][:, :1]
    one["q_rope"] = case["q_rope"][:, :1]
    one["seqlens"] = case["seqlens"] - 1
    out1, o_lat1, lse1 = _decode(one)
    assert np.array_equal(o_lat[:, 0], o_lat1[:, 0])
    assert np.array_equal(lse[:, 0], lse1[:, 0])
    assert np.array_equal(out[:, 0], out1[:, 0])
    assert not np.allclose(lse[:, 1], lse[:, 0])


def test_block_table_permutation_invariance():
    rng = np.random.default_rng(7)
    case = _rand_case(rng, seqlens=(17, 6, 12), bs=4)
    ref = _decode(case)
    nb = case["cache"].shape[0]
    perm = rng.permutation(nb)  # physical block p moves to perm[p]
    moved = dict(case)
    moved["cache"] = np.empty_like(case["cache"])
    moved["cache"][perm] = case["cache"]
    bt = case["block_table"].copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    moved["block_table"] = bt
    got = _decode(moved)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)


def test_append_places_rows():
    rng = np.random.default_rng(8)
    bs, D, d_c = 4, 6, 4
    seqlens = np.array([5, 8, 2])
    table = np.array([[3, 0, -1], [1, 4, -1], [2, -1, -1]])
    cache = rng.standard_normal((5, bs, D))
    c_kv = rng.standard_normal((3, 2, d_c))
    k_r = rng.standard_normal((3, 2, D - d_c))
    new = mla.append_to_cache(cache, table, seqlens, c_kv, k_r)
    touched = set()
    for b in range(3):
        for i in range(2):
            pos = seqlens[b] - 2 + i
            blk, slot = table[b][pos // bs], pos % bs
            touched.add((blk, slot))
            assert np.array_equal(new[blk, slot], np.concatenate([c_kv[b, i], k_r[b, i]]))
    for blk in range(5):
        for slot in range(bs):
            if (blk, slot) not in touched:
                assert np.array_equal(new[blk, slot], cache[blk, slot])


# ---- block-range pieces and their merge ------------------------------------


def _blocks(case, first, end):
    return mla.mla_decode_blocks(case["q_nope"], case["q_rope"], case["cache"],
                                 case["block_table"], case["seqlens"], case["W_UK"],
                                 case["W_UV"], case["Hq"], first, end)


@pytest.mark.parametrize("cuts", [(1,), (2,), (1, 3), (0, 1, 2, 3)])
@pytest.mark.parametrize("Hq", [1, 2])
def test_block_pieces_merge_to_the_whole_decode(cuts, Hq):
    # the softmax over a union of disjoint key sets: each piece's normalised
    # output re-weighted by its share of the denominator gives the whole row
    rng = np.random.default_rng(11 + Hq)
    case = _rand_case(rng, seqlens=(9, 1, 13, 16), Hq=Hq)
    bounds = (0,) + cuts + (10**6,)
    pieces = [_blocks(case, a, b) for a, b in zip(bounds, bounds[1:])]
    out, o_lat, lse = _decode(case)
    o_m, lse_m = mla.combine_pieces(np.stack([p[1] for p in pieces]),
                                    np.stack([p[2] for p in pieces]))
    out_m, _ = mla.combine_pieces(np.stack([p[0] for p in pieces]),
                                  np.stack([p[2] for p in pieces]))
    np.testing.assert_allclose(o_m, o_lat, atol=1e-12)
    np.testing.assert_allclose(out_m, out, atol=1e-12)
    np.testing.assert_array_equal(np.isfinite(lse_m), np.isfinite(lse))
    fin = np.isfinite(lse)
    np.testing.assert_allclose(lse_m[fin], lse[fin], atol=1e-12)


def test_block_range_cases():
    rng = np.random.default_rng(5)
    case = _rand_case(rng, seqlens=(9, 1, 13))
    out, o_lat, lse = _decode(case)
    # a range over every block is the decode itself
    _, o_all, lse_all = _blocks(case, 0, 10**6)
    np.testing.assert_array_equal(o_all, o_lat)
    np.testing.assert_array_equal(lse_all, lse)
    # a range past every sequence: nothing visible
    _, o_none, lse_none = _blocks(case, 100, 200)
    assert np.all(o_none == 0) and np.all(lse_none == -math.inf)
    # one block: exactly the softmax over that block's keys (brute force)
    bs = case["cache"].shape[1]
    _, o_1, lse_1 = _blocks(case, 1, 2)
    b, h = 2, 1  # sequence of 13 tokens: block 1 holds positions 4..7
    rows = np.stack([case["cache"][case["block_table"][b, 1], j] for j in range(bs)])
    d_c = case["W_UK"].shape[2]
    K = rows[:, :d_c] @ case["W_UK"][h].T
    s = (K @ case["q_nope"][b, 0, h] + rows[:, d_c:] @ case["q_rope"][b, 0, h]) / math.sqrt(
        case["W_UK"].shape[1] + case["q_rope"].shape[3])
    p = np.exp(s - s.max()) / np.exp(s - s.max()).sum()
    np.testing.assert_allclose(o_1[b, 0, h], p @ rows[:, :d_c], atol=1e-12)
    assert lse_1[b, 0, h] == pytest.approx(s.max() + math.log(np.exp(s - s.max()).sum()),
                                           abs=1e-12)


def test_combine_weights_and_empty_pieces():
    # two pieces with known denominators: weights e^{lse_p} / sum
    o = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])  # [P=2, rows=1, d=2]
    lse = np.array([[math.log(1.0)], [math.log(3.0)]])
    om, lm = mla.combine_pieces(o, lse)
    np.testing.assert_allclose(om[0], [0.25, 0.75], atol=1e-15)
    assert lm[0] == pytest.approx(math.log(4.0), abs=1e-15)
    # an empty piece (lse = -inf) weighs nothing; all empty -> 0 / -inf
    om, lm = mla.combine_pieces(np.array([[[5.0, 7.0]], [[9.0, 9.0]]]),
                                np.array([[0.5], [-math.inf]]))
    np.testing.assert_allclose(om[0], [5.0, 7.0])
    assert lm[0] == pytest.approx(0.5)
    om, lm = mla.combine_pieces(np.ones((3, 1, 2)), np.full((3, 1), -math.inf))
    assert np.all(om == 0) and lm[0] == -math.inf


def _merge_matches_whole(case, cuts=(1, 3)):
    bounds = (0,) + cuts + (10**6,)
    pieces = [_blocks(case, a, b) for a, b in zip(bounds, bounds[1:])]
    _, o_lat, lse = _decode(case)
    o_m, lse_m = mla.combine_pieces(np.stack([p[1] for p in pieces]),
                                    np.stack([p[2] for p in pieces]))
    fin = np.isfinite(lse)
    return (np.allclose(o_m, o_lat, atol=1e-9) and np.array_equal(np.isfinite(lse_m), fin)
            and np.allclose(lse_m[fin], lse[fin], atol=1e-9))


def _combine_unweighted(o_pieces, lse_pieces):  # plain mean of the pieces
    o, lse = _ORIG_COMBINE(o_pieces, lse_pieces)
    fin = np.isfinite(np.asarray(lse_pieces))
    return (np.asarray(o_pieces) * fin[..., None]).sum(0) / np.maximum(fin.sum(0), 1)[..., None], lse


def _combine_lse_max_only(o_pieces, lse_pieces):  # lse = max_p lse_p
    o, _ = _ORIG_COMBINE(o_pieces, lse_pieces)
    return o, np.asarray(lse_pieces).max(axis=0)


def _blocks_off_by_one(q_nope, q_rope, cache, block_table, seqlens, W_UK, W_UV, Hq, first,
                       end, **kw):  # the range ends one block late
    return _ORIG_BLOCKS(q_nope, q_rope, cache, block_table, seqlens, W_UK, W_UV, Hq, first,
                        end + 1, **kw)


_ORIG_COMBINE = mla.combine_pieces
_ORIG_BLOCKS = mla.mla_decode_blocks


@pytest.mark.parametrize("name,attr,fn", [
    ("unweighted mean", "combine_pieces", _combine_unweighted),
    ("lse is the max", "combine_pieces", _combine_lse_max_only),
    ("range one block long", "mla_decode_blocks", _blocks_off_by_one),
])
def test_planted_piece_mistakes_are_caught(name, attr, fn, monkeypatch):
    case = _rand_case(np.random.default_rng(3), seqlens=(9, 1, 13, 16))
    assert _merge_matches_whole(case)
    monkeypatch.setattr(mla, attr, fn)
    assert not _merge_matches_whole(case), f"'{name}' slipped past the merge invariant"
