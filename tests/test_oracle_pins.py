"""Pins of the fp64 oracle to values the pages print.

* "Mathematical Prerequisites for DeepSeek-V2", running example, sections 1-9.
* "From Vanilla Transformers to Modern LLMs -- Part 3", section 3 (one full
  MLA decode step with integer weights), stored in ``tests/golden``.

The ``check_*`` helpers raise ``AssertionError`` on any mismatch; the
mutation tests in ``test_oracle_mutations.py`` reuse them to show that a
planted mistake in the oracle fails at least one pin.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import mla, upstream

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

EXACT = 1e-12  # integer-valued quantities
PRINTED = 1e-3  # 3-decimal values (one unit in the last printed place)


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _close(got, want, tol, what):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    err = float(np.max(np.abs(got - want))) if got.size else 0.0
    assert err <= tol, f"{what}: max|err| {err:.3g} > {tol:g}\n got {got}\nwant {want}"


# ---------------------------------------------------------------------------
# "Mathematical Prerequisites for DeepSeek-V2"
# ---------------------------------------------------------------------------


def check_prereq():
    g = _load("prereq_linear_algebra.json")
    A = np.array(g["A"], float)
    B = np.array(g["B"], float)
    x = np.array(g["x"], float)
    z = np.array(g["z"], float)
    c = g["checks"]
    _close(mla.project(A, x), c["matvec_Ax"]["value"], EXACT, "A x (section 1)")
    _close(mla.project(B, z), c["Bz"]["value"], EXACT, "B z (section 4)")
    # associativity: (A^T B) z == A^T (B z)
    ATB = np.stack([mla.project(A.T, B[:, j]) for j in range(2)], axis=1)
    _close(ATB, c["AT_B"]["value"], EXACT, "A^T B (section 3)")
    _close(mla.project(ATB, z), c["associativity_ATBz"]["value"], EXACT, "(A^T B) z")
    _close(mla.project(A.T, mla.project(B, z)), c["associativity_ATBz"]["value"],
           EXACT, "A^T (B z)")
    bl = c["bilinear"]
    a = np.array(bl["a"], float)
    _close(mla.project(B.T, a), bl["MTa"], EXACT, "M^T a (section 6)")
    _close(mla.bilinear_direct(a, B, z), bl["value"], EXACT, "a^T M b (section 6)")
    _close(mla.bilinear_moved(a, B, z), bl["value"], EXACT, "(M^T a)^T b (section 6)")
    ln = c["linearity"]
    _close(mla.project(A, ln["x2"]), ln["Wx2"], EXACT, "W x2 (section 7)")
    _close(mla.weighted_sum_then_project(A, ln["alpha"], [ln["x1"], ln["x2"]]),
           ln["value"], 1e-12, "W(sum a x) (section 7)")
    _close(mla.project_then_weighted_sum(A, ln["alpha"], [ln["x1"], ln["x2"]]),
           ln["value"], 1e-12, "sum a W x (section 7)")
    lr = c["low_rank"]
    U = np.array(lr["U"], float).reshape(3, 1)
    V = np.array(lr["V"], float).reshape(1, 3)
    _close(mla.project(V, x), [lr["c"]], EXACT, "latent c = V x (section 8)")
    _close(mla.project(U, mla.project(V, x)), lr["value"], EXACT, "U (V x)")
    _close(mla.project(U @ V, x), lr["value"], EXACT, "(U V) x")
    cd = c["concat_dot"]
    _close(mla.concat_dot(cd["a"], cd["b"], cd["c"], cd["d"]), cd["value"], EXACT,
           "[a;b].[c;d] (section 9)")
    _close([mla.dot(cd["a"], cd["c"]), mla.dot(cd["b"], cd["d"])], cd["parts"], EXACT,
           "split dot (section 9)")


def test_prereq_running_example():
    check_prereq()


# ---------------------------------------------------------------------------
# "From Vanilla Transformers to Modern LLMs -- Part 3", section 3
# ---------------------------------------------------------------------------


def p5_library_layout(g):
    """The worked example in the library's layout (W_UK, W_UV transposed into
    [H, d_h, d_c]).

    Returns q_nope [1,1,H,d_h], q_rope [1,1,H,d_r], cache [1,4,d_c+d_r],
    block_table [[0]], seqlens [4], W_UK / W_UV [H,d_h,d_c].
    """
    d_h = g["dims"]["d_h"]
    H = g["dims"]["n_h"]
    pr = g["printed"]
    WUKp = np.array(g["inputs"]["W_UK"]["value"], float)  # [d_c, H*d_h]
    WUVp = np.array(g["inputs"]["W_UV"]["value"], float)
    W_UK = np.stack([WUKp[:, h * d_h:(h + 1) * d_h].T for h in range(H)])
    W_UV = np.stack([WUVp[:, h * d_h:(h + 1) * d_h].T for h in range(H)])
    c = np.array(pr["latents"]["value"], float)
    kr = np.array(pr["k_R_cached"]["value"], float)
    q4 = np.array(pr["q4"]["value"], float)
    q_nope = q4.reshape(1, 1, H, d_h)
    q_rope = np.stack([pr["q_R_head1"]["value"], pr["q_R_head2"]["value"]]).reshape(1, 1, H, 2)
    cache = np.concatenate([c, kr], axis=1)[None]
    return q_nope, q_rope, cache, np.array([[0]]), np.array([4]), W_UK, W_UV


def check_p5_upstream():
    g = _load("towardsai_p3_worked_example.json")
    pr = g["printed"]
    inp = g["inputs"]
    h = np.array(inp["h"]["value"], float)
    # the page's row-vector weights (d x out) are W^T in the column form
    W_DKV = np.array(inp["W_DKV"]["value"], float).T
    _close(upstream.down_project(W_DKV, h), pr["latents"]["value"], EXACT, "c_j = W_DKV h_j (3.b)")
    Wq = np.array(inp["W_q"]["value"], float).T
    _close(mla.project(Wq, h[3]), pr["q4"]["value"], EXACT, "q4 (3.d)")
    W_KR = np.array(inp["W_KR"]["value"], float).T
    k_raw = mla.project(W_KR, h)
    _close(k_raw, pr["k_R_before_rotation"]["value"], EXACT, "k_R before RoPE (3.k)")
    theta = np.array([math.pi / 2])  # the page's toy rotation: 90 degrees per position
    k_rot = np.stack([upstream.rope(k_raw[j], j, theta) for j in range(4)])
    _close(k_rot, pr["k_R_cached"]["value"], 1e-12, "cached rotated k_R (3.k)")
    # the whole cache row of token j, as the fused projection writes it (3.q)
    rows = np.stack([upstream.cache_row(h[j], W_DKV, W_KR, j, theta) for j in range(4)])
    _close(rows, np.concatenate([np.array(pr["latents"]["value"], float),
                                 np.array(pr["k_R_cached"]["value"], float)], axis=1),
           1e-12, "cache rows [c ; k_R] (3.q)")
    W_QR = np.array(inp["W_QR"]["value"], float).T
    qr_raw = mla.project(W_QR, h[3])
    _close(qr_raw, pr["q_R_before_rotation"]["value"], EXACT, "q_R before RoPE (3.l)")
    _close(upstream.rope(qr_raw[0:2], 3, theta), pr["q_R_head1"]["value"], 1e-12, "q_R head 1 (3.l)")
    _close(upstream.rope(qr_raw[2:4], 3, theta), pr["q_R_head2"]["value"], 1e-12, "q_R head 2 (3.l)")
    # relative position (3.n): rotating both by their positions equals rotating
    # only the query by the distance
    both = mla.dot(upstream.rope(qr_raw[0:2], 3, theta), upstream.rope(k_raw[2], 2, theta))
    rel = mla.dot(upstream.rope(qr_raw[0:2], 1, theta), k_raw[2])
    _close([both, rel], [pr["relative_position_score"]["value"]] * 2, 1e-12, "relative position (3.n)")
    # the query of token 4 (position 3) as the query projection builds it
    # (3.d, 3.l): content query and the per-head rotated RoPE queries
    qn, qr = upstream.query_projection(h[3], Wq, W_QR, 2, 2, 2, 3, theta)
    _close(qn.reshape(-1), pr["q4"]["value"], EXACT, "q4 by heads (3.d)")
    _close(qr, [pr["q_R_head1"]["value"], pr["q_R_head2"]["value"]], 1e-12, "q_R heads (3.l)")


def check_p5_content_path():
    g = _load("towardsai_p3_worked_example.json")
    pr = g["printed"]
    q_nope, _, cache, _, _, W_UK, _ = p5_library_layout(g)
    c = cache[0, :, :2]
    for h, name in ((0, "head1"), (1, "head2")):
        K = mla.reconstruct_keys(W_UK[h], c)
        _close(K, pr[f"naive_keys_{name}"]["value"], EXACT, f"naive keys {name} (3.e.1)")
        _close(K @ q_nope[0, 0, h], pr[f"content_scores_{name}"]["value"], EXACT,
               f"content scores {name} (3.e.1)")
    q_lat = mla.absorb_query(q_nope, W_UK)
    _close(q_lat[0, 0, 0], pr["absorbed_query_head1"]["value"], EXACT, "q^A head 1 (3.e.2)")
    _close(q_lat[0, 0, 1], pr["absorbed_query_head2"]["value"], EXACT, "q^A head 2 (3.e.2)")
    _close(c @ q_lat[0, 0, 0], pr["content_scores_head1"]["value"], EXACT, "absorbed scores (3.e.2)")
    # RoPE on the content key breaks absorption but the scores are still
    # defined (3.i): rotate the query by t=3 and each rebuilt key by its j.
    theta = np.array([math.pi / 2])
    K1 = mla.reconstruct_keys(W_UK[0], c)
    qrot = upstream.rope(q_nope[0, 0, 0], 3, theta)
    s = [mla.dot(qrot, upstream.rope(K1[j], j, theta)) for j in range(4)]
    _close(s, pr["rope_on_content_scores_head1"]["value"], 1e-12, "RoPE-on-content scores (3.i)")


def check_p5_norope_decode():
    """The RoPE-free step of 3.f-3.h: d_r = 0 and scale 1/sqrt(d_h)."""
    g = _load("towardsai_p3_worked_example.json")
    pr = g["printed"]
    q_nope, _, cache, bt, sl, W_UK, W_UV = p5_library_layout(g)
    cache0 = cache[:, :, :2]
    q_rope0 = np.zeros((1, 1, 2, 0))
    out, o_lat, _ = mla.mla_decode(q_nope, q_rope0, cache0, bt, sl, W_UK, W_UV, Hq=1,
                                   scale=1 / math.sqrt(2))
    for h, name in ((0, "head1"), (1, "head2")):
        r = mla.attention_row(q_nope[0, 0, h], np.zeros(0), cache0[0], W_UK[h], W_UV[h],
                              1 / math.sqrt(2), 2)
        _close(r["p"], pr[f"norope_softmax_{name}"]["value"], PRINTED, f"softmax {name} (3.f)")
        _close(o_lat[0, 0, h], pr[f"norope_cbar_{name}"]["value"], PRINTED, f"c-bar {name} (3.g)")
        _close(out[0, 0, h], pr[f"norope_o_{name}"]["value"], PRINTED, f"o {name} (3.g)")
    W_O = np.array(g["inputs"]["W_O"]["value"], float)
    _close(mla.output_projection(out[0, 0], W_O), pr["norope_u4"]["value"], PRINTED, "u4 (3.h)")


def check_p5_full_decode():
    """The decoupled-RoPE step of 3.j-3.p with scale 1/sqrt(d_h + d_h^R)."""
    g = _load("towardsai_p3_worked_example.json")
    pr = g["printed"]
    q_nope, q_rope, cache, bt, sl, W_UK, W_UV = p5_library_layout(g)
    scale = mla.default_scale(2, 2)
    _close(scale, 0.5, EXACT, "scale 1/sqrt(d_h + d_hR) (3.o)")
    out, o_lat, lse = mla.mla_decode(q_nope, q_rope, cache, bt, sl, W_UK, W_UV, Hq=1)
    for h, name in ((0, "head1"), (1, "head2")):
        pos = cache[0, :, 2:] @ q_rope[0, 0, h]
        _close(pos, pr[f"positional_scores_{name}"]["value"], EXACT, f"positional {name} (3.m)")
        r = mla.attention_row(q_nope[0, 0, h], q_rope[0, 0, h], cache[0], W_UK[h], W_UV[h],
                              scale, 2)
        _close(r["s"] / scale, pr[f"combined_scores_{name}"]["value"], EXACT,
               f"combined scores {name} (3.o)")
        _close(r["s"], pr[f"scaled_scores_{name}"]["value"], EXACT, f"scaled scores {name} (3.o)")
        _close(r["p"], pr[f"softmax_{name}"]["value"], PRINTED, f"softmax {name} (3.o)")
        _close(o_lat[0, 0, h], pr[f"cbar_{name}"]["value"], PRINTED, f"c-bar {name} (3.p)")
        _close(out[0, 0, h], pr[f"o_{name}"]["value"], PRINTED, f"o {name} (3.p)")
        s = np.array(pr[f"scaled_scores_{name}"]["value"], float)
        want_lse = s.max() + math.log(np.exp(s - s.max()).sum())
        _close(lse[0, 0, h], want_lse, 1e-12, f"lse {name}")
    W_O = np.array(g["inputs"]["W_O"]["value"], float)
    _close(mla.output_projection(out[0, 0], W_O), pr["u4"]["value"], PRINTED, "u4 (3.p)")
    # value absorption: out == W_UV o_lat (3.g / 3.p)
    _close(mla.out_proj(o_lat, W_UV), out, 1e-12, "W_UV o_lat == sum p V")


def check_projection_layouts():
    """Special cases that fix the head and row layouts of the projections
    (the worked example cannot: its query [1, 2, 2, 1] reads the same with
    heads taken contiguously or interleaved).  With identity weights and
    position 0 (no rotation), head h of the query must be coordinates
    h*d_h .. h*d_h+d_h-1 of the hidden state, and the cache row is the hidden
    state itself; at position 1 with theta = pi/2 each RoPE pair (x0, x1)
    becomes (-x1, x0) ("MLA, dim by dim" 3: adjacent pairs)."""
    H, d_h, d_r = 3, 4, 2
    h = np.arange(1.0, 1.0 + H * d_h)
    qn, qr = upstream.query_projection(h, np.eye(H * d_h), np.eye(H * d_r, H * d_h), H, d_h,
                                       d_r, 0, np.array([0.3]))
    _close(qn, h.reshape(H, d_h), EXACT, "query heads are contiguous slices")
    _close(qr, h[:H * d_r].reshape(H, d_r), EXACT, "RoPE query heads are contiguous slices")
    _, qr1 = upstream.query_projection(h, np.eye(H * d_h), np.eye(H * d_r, H * d_h), H, d_h, d_r,
                                       1, np.array([math.pi / 2]))
    want = np.stack([[-h[2 * i + 1], h[2 * i]] for i in range(H)])
    _close(qr1, want, 1e-12, "each head's RoPE pair turns by 90 degrees")
    x = np.arange(1.0, 7.0)
    row = upstream.cache_row(x, np.eye(4, 6), np.eye(2, 6, k=4), 0, np.array([0.3]))
    _close(row, x, EXACT, "cache row [c ; k_R] in order")


def test_projection_layouts():
    check_projection_layouts()


def test_p5_upstream_and_rope():
    check_p5_upstream()


def test_p5_content_path():
    check_p5_content_path()


def test_p5_norope_decode():
    check_p5_norope_decode()


def test_p5_full_decode():
    check_p5_full_decode()


def test_p5_paged_layouts_agree():
    """The same example stored with block size 1, 2 and 3 and permuted blocks."""
    g = _load("towardsai_p3_worked_example.json")
    q_nope, q_rope, cache, bt, sl, W_UK, W_UV = p5_library_layout(g)
    ref = mla.mla_decode(q_nope, q_rope, cache, bt, sl, W_UK, W_UV, Hq=1)
    rows = cache[0]
    for bs in (1, 2, 3):
        nblk = -(-4 // bs)
        perm = np.random.default_rng(bs).permutation(nblk)
        paged = np.zeros((nblk, bs, rows.shape[1]))
        for j in range(4):
            paged[perm[j // bs], j % bs] = rows[j]
        got = mla.mla_decode(q_nope, q_rope, paged, perm[None, :], sl, W_UK, W_UV, Hq=1)
        for a, b in zip(got, ref):
            _close(a, b, 0.0, f"paged block size {bs}")


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
