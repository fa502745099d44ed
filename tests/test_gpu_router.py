"""GPU parity of the MoE router: fp8bs_moe_gate against the oracle's fp64
router and fp8bs_moe_route bit for bit against the oracle's stable counting
sort (DeepSeek-V3 notes, page 2 section 2-2; config block of
"671B 参数如何「激活」37B？").

Gate bound.  The kernel's logits come from bf16 operands with fp32
accumulation: |l - l_exact| <= dim 2^-24 L, L = sum_k |x_k w_k|.  sigmoid
has slope at most 1/4, and its fp32 evaluation (expf, one add, one divide)
adds a few units in the last place, so each affinity (and biased affinity)
is within delta = dim 2^-24 L / 4 + 2^-20 of the exact one.  The selection
is therefore checked in two ways: wherever the exact scores leave margins
wider than 2 delta the chosen experts must be the oracle's exactly, and
everywhere the chosen set must be optimal up to 2 delta.  The gate values
are checked against the oracle's affinities of the chosen experts.
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_18_b300 import synth
from gpu_util import bf16_to_f64, dev, dev_bf16, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp8_block_scaled_18_b300 import fp8bs
    return fp8bs


def _check_gate(ids_g, w_g, x, wg, bias, s_o, ids_o, n_groups, topk_groups, top_k, scale=2.5, min_decided=0.5):
    T, E = s_o.shape
    dim = x.shape[1]
    L = np.abs(bf16_to_f64(x)) @ np.abs(bf16_to_f64(wg)).T                   # [T, E]
    delta = dim * 2.0 ** -24 * L / 4 + 2.0 ** -20
    b_o = s_o + bias.astype(np.float64)[None, :]
    per = E // n_groups
    exact = same = 0
    for t in range(T):
        g_ids = ids_g[t]
        assert len(set(g_ids.tolist())) == top_k and g_ids.min() >= 0 and g_ids.max() < E
        d2 = 2 * delta[t].max()
        gscore = b_o[t].reshape(n_groups, per).max(axis=1)
        kept = sorted(set((g_ids // per).tolist()))
        assert len(kept) <= topk_groups
        # a group holding a chosen expert is among the best topk_groups up to 2 delta
        for g in kept:
            assert (gscore > gscore[g] + d2).sum() < topk_groups, f"token {t}: group {g} not among the best"
        # the chosen experts are the best of the chosen groups' experts up to 2 delta
        cand = np.concatenate([np.arange(g * per, (g + 1) * per) for g in kept])
        worst_chosen = b_o[t, g_ids].min()
        others = np.setdiff1d(cand, g_ids)
        if others.size:
            assert b_o[t, others].max() <= worst_chosen + d2, f"token {t}: a better expert was left out"
        # descending order up to 2 delta
        assert np.all(np.diff(b_o[t, g_ids]) <= d2)
        # unambiguous tokens: exactly the oracle's choice
        srt = np.sort(gscore)[::-1]
        o_ids = ids_o[t]
        o_cand = np.concatenate([np.arange(g * per, (g + 1) * per) for g in sorted(set((o_ids // per).tolist()))])
        bo = np.sort(b_o[t, o_cand])[::-1]
        margins = [srt[topk_groups - 1] - srt[topk_groups] if topk_groups < n_groups else np.inf,
                   bo[top_k - 1] - bo[top_k] if bo.size > top_k else np.inf,
                   np.min(-np.diff(b_o[t, o_ids])) if top_k > 1 else np.inf]
        same += int(np.array_equal(g_ids, o_ids))
        if min(margins) > 2 * d2:
            assert np.array_equal(g_ids, o_ids), f"token {t}: {g_ids} vs oracle {o_ids}"
            exact += 1
        # gate values: the chosen affinities normalised, times the scale
        s_sel = s_o[t, g_ids]
        w_exp = s_sel / s_sel.sum() * scale
        tol = scale * 9 * delta[t].max() / s_sel.sum() + 2.0 ** -21 * np.abs(w_exp)
        assert np.all(np.abs(w_g[t] - w_exp) <= tol), f"token {t}: gate values {w_g[t]} vs {w_exp}"
    # not vacuous: the worst-case bound leaves many near-ties open, but the
    # actual fp32 error is far smaller, so nearly every token matches the
    # oracle outright; at small widths most tokens are also decided by the
    # bound itself (min_decided)
    assert same >= 0.95 * T, f"only {same} of {T} tokens chose the oracle's experts"
    assert exact >= min_decided * T, f"only {exact} of {T} tokens were unambiguous under the bound"
    return exact


@pytest.mark.parametrize("T,dim,E,n_groups,topk_groups,top_k,std", [
    (300, 512, 256, 8, 4, 8, 0.075),     # DeepSeek-V3's routing shape at a reduced width, ragged tokens
    (130, 128, 64, 16, 3, 5, 0.15),      # groups of 4 experts: a 16-column slice spans several groups
    (5, 64, 16, 1, 1, 1, 0.2),           # one group, top-1, one K chunk
    (200, 192, 96, 3, 2, 4, 0.15),       # six 16-column units (E not a multiple of 64), groups of 32
    (77, 128, 80, 5, 3, 7, 0.15),        # five units, groups of 16, K of 2 chunks over 4 CTAs
    (9600, 128, 64, 4, 2, 6, 0.15),      # 75 tiles: more than two waves as clusters, so one CTA per tile
])
def test_gate_vs_oracle(F, orc, T, dim, E, n_groups, topk_groups, top_k, std):
    rng = np.random.default_rng(T + E)
    x = synth.normal_bf16(rng, (T, dim), 1.0)
    wg = synth.normal_bf16(rng, (E, dim), std)
    bias = rng.uniform(-0.1, 0.1, size=E).astype(np.float32)
    ids, w = F.fp8bs_moe_gate(dev_bf16(x), dev_bf16(wg), dev(bias), n_groups=n_groups, topk_groups=topk_groups,
                              top_k=top_k)
    assert F.fp8bs_sync_status() == 0
    ids_o, _, s_o = orc.moe_gate(x, wg, bias, n_groups=n_groups, topk_groups=topk_groups, top_k=top_k,
                                 want_scores=True)
    _check_gate(host(ids), host(w).astype(np.float64), x, wg, bias, s_o, ids_o, n_groups, topk_groups, top_k)


def test_gate_full_width(F, orc):
    """The gate at the configuration's width: 256 experts, dim 7168, gate
    weight ~N(0, 0.02), bias ~U(-0.1, 0.1), 384 tokens.  At this width the
    worst-case logit bound (dim 2^-24 L, about 0.01 on the affinities) is
    wider than the typical gap between the 8th and 9th expert, so no token is
    decided by the bound alone; the selections are checked for optimality
    within it and must equal the oracle's on at least 95 % of the tokens."""
    rng = np.random.default_rng(4)
    x = synth.activations(rng, 384, synth.DIM)
    gw = synth.normal_bf16(rng, (synth.N_EXPERTS, synth.DIM), 0.02)
    bias = rng.uniform(-0.1, 0.1, size=synth.N_EXPERTS).astype(np.float32)
    ids, w = F.fp8bs_moe_gate(dev_bf16(x), dev_bf16(gw), dev(bias))
    assert F.fp8bs_sync_status() == 0
    ids_o, _, s_o = orc.moe_gate(x, gw, bias, want_scores=True)
    _check_gate(host(ids), host(w).astype(np.float64), x, gw, bias, s_o, ids_o, 8, 4, 8, min_decided=0.0)


@pytest.mark.parametrize("E,n_groups", [(256, 8), (96, 3)])
def test_gate_exact_ties_go_to_lower_index(F, orc, E, n_groups):
    """Group 1 is an exact copy of group 0 (weight rows and bias), so those
    experts' logits, and the two groups' scores, tie exactly; the selection
    must then prefer the lower group and the lower expert: wherever expert
    e + per is chosen, e is chosen too and ranks before it."""
    rng = np.random.default_rng(E)
    T, dim, per = 256, 256, E // n_groups
    x = synth.normal_bf16(rng, (T, dim), 1.0)
    wg = synth.normal_bf16(rng, (E, dim), 0.1)
    wg[per:2 * per] = wg[:per]
    bias = rng.uniform(-0.1, 0.1, size=E).astype(np.float32)
    bias[per:2 * per] = bias[:per]
    ids, w = F.fp8bs_moe_gate(dev_bf16(x), dev_bf16(wg), dev(bias), n_groups=n_groups, topk_groups=2, top_k=6)
    assert F.fp8bs_sync_status() == 0
    ids, w = host(ids), host(w)
    ids_o, _ = orc.moe_gate(x, wg, bias, n_groups=n_groups, topk_groups=2, top_k=6)
    twins = 0
    for t in range(T):
        pos = {int(e): i for i, e in enumerate(ids[t])}
        for e, i in pos.items():
            if per <= e < 2 * per:
                twins += 1
                assert e - per in pos and pos[e - per] < i, f"token {t}: {ids[t]}"
                assert w[t, i] == w[t, pos[e - per]]
    assert twins > 0.2 * T
    assert (ids == ids_o).all(axis=1).mean() >= 0.95


def test_gate_without_bias_and_strided_x(F, orc):
    """bias NULL (zeros) and an x whose rows are strided."""
    rng = np.random.default_rng(9)
    T, dim, E = 200, 256, 128
    xs = synth.normal_bf16(rng, (T, dim + 64), 1.0)
    wg = synth.normal_bf16(rng, (E, dim), 0.1)
    xt = dev_bf16(xs)[:, :dim]
    ids, w = F.fp8bs_moe_gate(xt, dev_bf16(wg), None, n_groups=8, topk_groups=2, top_k=6)
    assert F.fp8bs_sync_status() == 0
    x = np.ascontiguousarray(xs[:, :dim])
    zero = np.zeros(E, dtype=np.float32)
    ids_o, _, s_o = orc.moe_gate(x, wg, zero, n_groups=8, topk_groups=2, top_k=6, want_scores=True)
    _check_gate(host(ids), host(w).astype(np.float64), x, wg, zero, s_o, ids_o, 8, 2, 6)


# ------------------------------------------------------------------ routing tables


@pytest.mark.parametrize("T,k,E", [(1500, 8, 256), (4096, 8, 256), (3, 2, 16), (1025, 1, 64), (20000, 6, 128)])
def test_route_bit_exact(F, orc, T, k, E):
    rng = np.random.default_rng(T + k)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    ids[: T // 3, 0] = 5                                           # one busy expert
    for t in range(T // 3):                                        # keep a token's experts distinct
        if len(set(ids[t].tolist())) < k:
            rest = [e for e in range(E) if e != 5]
            ids[t, 1:] = rng.choice(rest, size=k - 1, replace=False)
    w = rng.uniform(0.05, 1.0, size=(T, k)).astype(np.float32)
    off, tor, rot, wor = F.fp8bs_moe_route(dev(ids), dev(w), E)
    assert F.fp8bs_sync_status() == 0
    off_o, tor_o, rot_o, wor_o = orc.moe_route(ids, w, E)
    assert np.array_equal(host(off), off_o)
    assert np.array_equal(host(tor), tor_o)
    assert np.array_equal(host(rot), rot_o)
    assert np.array_equal(host(wor).view(np.uint32), wor_o.view(np.uint32))


def test_route_of_the_generator(F):
    """The configuration's own selections (4096 tokens, top-8 of 256): the
    device tables equal the generator's grouping (numpy's stable sort)."""
    case = synth.moe()
    T, k = case.rows_of_token.shape
    expert_of_row = np.searchsorted(case.offsets, np.arange(T * k), side="right") - 1
    ids = expert_of_row[case.rows_of_token].astype(np.int32)
    w = case.weight_of_row[case.rows_of_token].astype(np.float32)
    off, tor, rot, wor = F.fp8bs_moe_route(dev(ids), dev(w), case.n_experts)
    assert F.fp8bs_sync_status() == 0
    assert np.array_equal(host(off), case.offsets)
    assert np.array_equal(host(tor), case.token_of_row.astype(np.int32))
    assert np.array_equal(host(rot), case.rows_of_token)
    assert np.array_equal(host(wor).view(np.uint32), case.weight_of_row.view(np.uint32))


def test_route_bad_ids(F):
    """Out-of-range ids get no row; a repeated expert leaves a row with token
    -1; both report FP8BS_ERR_INDEX; the rest stays consistent."""
    ids = np.array([[0, 1], [2, 9], [3, -1], [4, 4]], dtype=np.int32)
    w = np.full((4, 2), 0.5, dtype=np.float32)
    off, tor, rot, wor = F.fp8bs_moe_route(dev(ids), dev(w), 8)
    assert F.fp8bs_sync_status() == F.FP8BS_ERR_INDEX
    rot_h, tor_h = host(rot), host(tor)
    assert rot_h[1, 1] == -1 and rot_h[2, 1] == -1
    for t, kk in [(0, 0), (0, 1), (1, 0), (2, 0)]:
        assert tor_h[rot_h[t, kk]] == t
    n_rows = int(host(off)[-1])                      # 6 selections name an expert in range
    assert n_rows == 6
    assert (tor_h[:n_rows] == -1).sum() == 1         # expert 4's second row: token 3 named it twice
