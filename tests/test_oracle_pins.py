"""Pins of the oracle to facts outside itself: numbers the pages print, closed forms worked
by hand, special cases, invariants the pages' equations imply, and brute force on tiny
inputs. Each test is chosen so that a plausible slip in the oracle (a dropped term, a wrong
sign or index, a transposed operand, a wrong tie rule) fails it. CPU only."""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_moe_ffn_router_gb300 import synth
from sparse_moe_ffn_router_gb300.workloads import WORKLOADS
from tests.inputs import bf16, top_gaps

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def sig(z):
    return 1.0 / (1.0 + math.exp(-z))


def _closed(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"sig": sig, "exp": math.exp}))  # noqa: S307


def _zero_layer(H, E, I, Is):
    z = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)  # noqa: E731
    return dict(router_w=z(E, H), router_b=None, gate_up=z(E, 2 * I, H), down=z(E, H, I),
                shared_gate_up=z(2 * Is, H), shared_down=z(H, Is), shared_gate=z(1, H))


def _rand_layer(H, E, I, Is, seed, router_std=0.02):
    return synth.make_weights(H, E, I, Is, seed, router_std=router_std)


# ---------------------------------------------------------------------------------------
# Numbers printed on the pages


def test_page_parameter_counts_pin_shapes():
    facts = json.load(open(os.path.join(GOLDEN, "page_facts.json")))
    g = facts["generics"]["value"]
    H, E, K, I = g["H"], g["Experts"], g["TopK"], g["ExpertInner"]
    per_expert = 3 * I * H  # gate + up + down, each I*H
    assert round(per_expert / 1e6, 2) == facts["params_per_expert_millions"]["value"]
    assert round(per_expert / 1e6, 1) == facts["params_per_expert_rough_millions"]["value"]
    assert round(K * per_expert / 1e6, 1) == facts["active_expert_params_millions"]["value"]
    # The page's 806M is E times its rounded 3.15M per expert (256 * 3.15 = 806.4); the exact
    # count 805.3M lies within E times the rounding half-unit of 3.15M.
    assert round(E * round(per_expert / 1e6, 2)) == facts["total_expert_params_millions"]["value"]
    assert abs(E * per_expert / 1e6 - facts["total_expert_params_millions"]["value"]) <= E * 0.005
    assert [E, 2 * I, H] == facts["gate_up_shape"]["value"]
    assert facts["router"]["value"] == [H, E]
    for name in ("decode_T1", "decode_T64", "prefill_T4096_zipf", "stack40_decode_T32"):
        wl = WORKLOADS[name]
        assert (wl.H, wl.E, wl.K, wl.I, wl.Is) == (H, E, K, I, g["SharedInner"])


# ---------------------------------------------------------------------------------------
# Hand-worked layers (closed forms)


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "hand_cases.json")))["cases"],
                         ids=lambda c: c["name"])
def test_hand_cases(case):
    dims = tuple(case["dims"])
    w = {k: bf16(case[k]) for k in ("router_w", "gate_up", "down", "shared_gate_up", "shared_down", "shared_gate")}
    w["router_b"] = None
    r = oracle.forward(dims, bf16(case["x"]), w, taps=True)
    ex = case["expect"]
    np.testing.assert_allclose(r["out"][0], [_closed(e) for e in ex["out"]], rtol=1e-14, atol=1e-15)
    if "sg" in ex:
        assert r["sg"][0] == pytest.approx(_closed(ex["sg"]), rel=1e-15)
    if "h" in ex:
        np.testing.assert_allclose(r["h"][0, :, 0], [_closed(e) for e in ex["h"]], rtol=1e-14)
    if "ids" in ex:
        assert r["ids"].tolist() == ex["ids"]
    if "w" in ex:
        np.testing.assert_allclose(r["w"], ex["w"], rtol=1e-15)
    if "w_expr" in ex:
        np.testing.assert_allclose(r["w"][0], [_closed(e) for e in ex["w_expr"]], rtol=1e-14)


def test_residual_is_added_exactly():
    H, E, K, I, Is, T = 64, 8, 2, 16, 16, 5
    w = _rand_layer(H, E, I, Is, seed=11)
    x = synth.make_x(T, H, 11)
    res = synth.make_x(T, H, 12)
    a = oracle.forward((T, H, E, K, I, Is), x, w)["out"]
    b = oracle.forward((T, H, E, K, I, Is), x, w, residual=res)["out"]
    np.testing.assert_allclose(b - a, oracle.bf16_bits_to_f64(res), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------------------
# Router orientation, bias, selection, tie rule and renormalisation, on one-hot tokens.
# With x = e_h the logits are exactly column h of the router weight plus the bias, so the
# expected routing follows from the bf16 values alone.


@pytest.mark.parametrize("E,K,with_bias", [(256, 8, False), (256, 8, True), (32, 4, True), (8, 8, False)])
def test_one_hot_routing_closed_form(E, K, with_bias):
    H, T = 16, 16
    wr = synth.normal_bf16((E, H), 0.02, synth.stream_key(5, 0, "router_w"))
    br = synth.zipf_bias(E, 1.1, 5) if with_bias else None
    x = torch.zeros(T, H, dtype=torch.bfloat16)
    for t in range(T):
        x[t, t % H] = 1.0
    r = oracle.route((T, H, E, K, 4, 4), x, wr, br)
    col = oracle.bf16_bits_to_f64(wr)
    b = oracle.bf16_bits_to_f64(br) if with_bias else np.zeros(E)
    for t in range(T):
        l = col[:, t % H] + b
        order = np.lexsort((np.arange(E), -l))  # score descending, then the lower index
        assert r["ids"][t].tolist() == order[:K].tolist()
        sel = l[order[:K]]
        ew = np.exp(sel - sel.max())
        np.testing.assert_allclose(r["w"][t], ew / ew.sum(), rtol=1e-13)


def test_all_equal_scores_pick_lowest_indices():
    H, E, K, T = 8, 32, 4, 3
    w = _zero_layer(H, E, 4, 4)
    r = oracle.route((T, H, E, K, 4, 4), synth.make_x(T, H, 1), w["router_w"])
    assert r["ids"].tolist() == [list(range(K))] * T
    np.testing.assert_array_equal(r["w"], np.full((T, K), 1.0 / K))


@pytest.mark.parametrize("E,K", [(256, 8), (32, 4), (16, 1), (8, 8)])
def test_selection_equals_brute_force_full_sort(E, K):
    """The oracle selects by per-expert ranks; compare with a full sort of the probabilities."""
    H, T = 64, 48
    wr = synth.normal_bf16((E, H), 0.3, synth.stream_key(7, 0, "router_w"))
    x = synth.make_x(T, H, 7)
    r = oracle.route((T, H, E, K, 4, 4), x, wr, want_probs=True)
    p = r["probs"]
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-p[t, e], e))
        assert r["ids"][t].tolist() == order[:K]


def test_renorm_invariants_and_slot_order():
    wl = WORKLOADS["decode_T64"]
    H = 256
    E, K = wl.E, wl.K
    wr = synth.normal_bf16((E, H), 0.05, synth.stream_key(9, 0, "router_w"))
    x = synth.make_x(64, H, 9)
    r = oracle.route((64, H, E, K, 4, 4), x, wr, want_probs=True)
    np.testing.assert_allclose(r["w"].sum(1), 1.0, rtol=0, atol=1e-12)
    assert (r["w"] > 0).all() and (r["w"] <= 1).all()
    assert (np.diff(r["w"], axis=1) <= 0).all()  # slots run from the largest weight down
    for t in range(64):
        assert len(set(r["ids"][t].tolist())) == K
    assert r["ids"].min() >= 0 and r["ids"].max() < E
    np.testing.assert_allclose(r["probs"].sum(1), 1.0, atol=1e-12)


def test_top1_weight_is_one():
    H, E, T = 32, 16, 10
    wr = synth.normal_bf16((E, H), 0.5, synth.stream_key(3, 0, "router_w"))
    r = oracle.route((T, H, E, 1, 4, 4), synth.make_x(T, H, 3), wr)
    np.testing.assert_array_equal(r["w"], 1.0)


# ---------------------------------------------------------------------------------------
# Expert math: halves of the merged gate_up tensor and orientation of each projection.


def test_expert_projection_orientation_closed_form():
    """One-hot x at column c and a down matrix with one non-zero per inner index give
    y[o] = SiLU(Wg[j, c]) * Wu[j, c] * d_j at o = (j + 1) mod H, zero elsewhere. A gate/up
    swap, a transposed projection or a wrong row offset changes the result."""
    H, E, I, Is = 12, 4, 5, 5
    c = 7
    w = _zero_layer(H, E, I, Is)
    w["router_b"] = torch.tensor([0, 0, 4.0, 0], dtype=torch.bfloat16)  # expert 2 always wins
    gu = synth.normal_bf16((E, 2 * I, H), 1.0, synth.stream_key(1, 0, "gate_up"))
    w["gate_up"] = gu
    dvals = [1.5, -2.0, 0.75, 3.0, -0.5]
    down = torch.zeros(E, H, I)
    for j in range(I):
        down[2, (j + 1) % H, j] = dvals[j]
        down[0, j, j] = 100.0  # a different expert that must not be used
    w["down"] = down.to(torch.bfloat16)
    x = torch.zeros(1, H, dtype=torch.bfloat16)
    x[0, c] = 1.0
    r = oracle.forward((1, H, E, 1, I, Is), x, w, taps=True)
    assert r["ids"].tolist() == [[2]]
    g = oracle.bf16_bits_to_f64(gu)[2]
    expect = np.zeros(H)
    for j in range(I):
        gj, uj = g[j, c], g[I + j, c]
        expect[(j + 1) % H] = gj * sig(gj) * uj * dvals[j]
    np.testing.assert_allclose(r["out"][0], expect, rtol=1e-13, atol=1e-15)
    # the shared expert is zero, its gate is sigmoid(0)
    assert r["sg"][0] == 0.5


def test_identical_experts_make_routing_irrelevant():
    """With every routed expert equal, the renormalised weights sum to one, so the routed
    part equals that one expert for any routing: compare with a 1-expert layer."""
    H, E, K, I, Is, T = 48, 16, 4, 12, 8, 6
    w1 = _rand_layer(H, 1, I, Is, seed=21)
    wE = dict(w1)
    wE["router_w"] = synth.normal_bf16((E, H), 0.5, synth.stream_key(21, 0, "router_w"))
    wE["gate_up"] = w1["gate_up"].expand(E, -1, -1).contiguous()
    wE["down"] = w1["down"].expand(E, -1, -1).contiguous()
    x = synth.make_x(T, H, 21)
    a = oracle.forward((T, H, E, K, I, Is), x, wE)["out"]
    b = oracle.forward((T, H, 1, 1, I, Is), x, w1)["out"]
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_dense_mixture_when_k_equals_e():
    """K = E: the renormalised weights are the full softmax, and the routed part is
    sum_e softmax(l)_e * expert_e(x); each expert_e(x) is taken from a 1-expert layer."""
    H, E, I, Is, T = 10, 4, 6, 6, 3
    w = _rand_layer(H, E, I, Is, seed=31, router_std=1.0)
    x = torch.zeros(T, H, dtype=torch.bfloat16)
    for t in range(T):
        x[t, 2 * t + 1] = 1.0
    out = oracle.forward((T, H, E, E, I, Is), x, w)["out"]
    zero_shared = dict(shared_gate_up=torch.zeros(2 * Is, H, dtype=torch.bfloat16),
                       shared_down=torch.zeros(H, Is, dtype=torch.bfloat16))
    shared_only = oracle.forward((T, H, E, E, I, Is), x, {**w, "gate_up": torch.zeros_like(w["gate_up"])})["out"]
    col = oracle.bf16_bits_to_f64(w["router_w"])
    expect = shared_only.copy()
    for t in range(T):
        l = col[:, 2 * t + 1]
        p = np.exp(l - l.max())
        p /= p.sum()
        for e in range(E):
            we = {**w, **zero_shared, "router_w": w["router_w"][e:e + 1], "gate_up": w["gate_up"][e:e + 1],
                  "down": w["down"][e:e + 1]}
            ye = oracle.forward((1, H, 1, 1, I, Is), x[t:t + 1], we)["out"][0]
            expect[t] += p[e] * ye
    np.testing.assert_allclose(out, expect, rtol=1e-12, atol=1e-13)


def test_down_scaling_is_linear():
    H, E, K, I, Is, T = 32, 8, 3, 8, 8, 4
    w = _rand_layer(H, E, I, Is, seed=41)
    w["shared_down"] = torch.zeros_like(w["shared_down"])
    x = synth.make_x(T, H, 41)
    a = oracle.forward((T, H, E, K, I, Is), x, w)["out"]
    b = oracle.forward((T, H, E, K, I, Is), x, {**w, "down": (w["down"].float() * 2).to(torch.bfloat16)})["out"]
    np.testing.assert_array_equal(b, 2 * a)


def test_tokens_are_independent():
    H, E, K, I, Is, T = 64, 16, 4, 16, 16, 9
    w = _rand_layer(H, E, I, Is, seed=51)
    x = synth.make_x(T, H, 51)
    x[5] = x[2]
    a = oracle.forward((T, H, E, K, I, Is), x, w)["out"]
    np.testing.assert_array_equal(a[5], a[2])
    pi = np.random.default_rng(0).permutation(T)
    b = oracle.forward((T, H, E, K, I, Is), x[torch.as_tensor(pi)], w)["out"]
    np.testing.assert_array_equal(b, a[pi])


# ---------------------------------------------------------------------------------------
# Dispatch (counting sort) against a comparison sort.


@pytest.mark.parametrize("T,E,K", [(0, 8, 2), (1, 256, 8), (37, 32, 4), (300, 256, 8)])
def test_permutation_structure(T, E, K):
    rng = np.random.default_rng(T)
    ids = np.array([rng.choice(E, K, replace=False) for _ in range(T)], dtype=np.int32).reshape(T, K)
    r = oracle.permute((T, 8, E, K, 4, 4), ids)
    flat = ids.ravel()
    expect_perm = sorted(range(T * K), key=lambda j: (flat[j], j // K))
    assert r["perm"].tolist() == expect_perm
    assert r["counts"].tolist() == [int((flat == e).sum()) for e in range(E)]
    assert r["offsets"][0] == 0 and r["offsets"][-1] == T * K
    np.testing.assert_array_equal(np.diff(r["offsets"]), r["counts"])
    if T:
        np.testing.assert_array_equal(r["perm"][r["inv"]], np.arange(T * K))


# ---------------------------------------------------------------------------------------
# RMSNorm and bf16 rounding.


def test_rmsnorm_closed_form():
    x = bf16([[3.0, 4.0], [-2.0, -2.0]])
    out = oracle.rmsnorm(x, eps=1e-6)
    np.testing.assert_allclose(out[0], np.array([3.0, 4.0]) / math.sqrt(12.5 + 1e-6), rtol=1e-15)
    np.testing.assert_allclose(out[1], [-2.0 / math.sqrt(4.0 + 1e-6)] * 2, rtol=1e-15)
    g = bf16([2.0, 0.5])
    np.testing.assert_allclose(oracle.rmsnorm(x, g)[0], np.array([6.0, 2.0]) / math.sqrt(12.5 + 1e-6), rtol=1e-15)


def test_round_bf16_nearest_even_without_double_rounding():
    assert oracle.round_bf16(1.0) == 0x3F80
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 0x3F80  # tie -> even
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82  # tie -> even (up)
    assert oracle.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81  # just above the tie
    assert oracle.round_bf16(-(1.0 + 2.0 ** -8 + 2.0 ** -40)) == 0xBF81
    assert oracle.round_bf16(-2.5) == 0xC020


# ---------------------------------------------------------------------------------------
# The input generator (no layer arithmetic) and the routing skew of the prefill workload.


def test_generator_matches_reference_splitmix64():
    key = synth.stream_key(3, 1, "gate_up")
    z = synth.uniform_u64(512, key)
    assert z.tolist() == [synth._signed(synth.splitmix64_py(key, i)) for i in range(512)]
    # published test vector of SplitMix64 with seed 1234567 (first output of the sequential form)
    assert synth.splitmix64_py(1234567, 0) == 6457827717110365317


def test_generator_statistics_and_row_redraw():
    x = synth.normal_bf16((1 << 18,), 1.0, synth.stream_key(0, 0, "x")).double()
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1) < 0.01
    a = synth.make_x(6, 32, 2)
    b = synth.make_x(6, 32, 2, attempts=[0, 0, 1, 0, 0, 0])
    assert torch.equal(a[[0, 1, 3, 4, 5]], b[[0, 1, 3, 4, 5]]) and not torch.equal(a[2], b[2])


def test_prefill_router_bias_gives_zipf_like_load():
    wl = WORKLOADS["prefill_T4096_zipf"]
    wr = synth.normal_bf16((wl.E, wl.H), 0.02, synth.stream_key(wl.seed, 0, "router_w"))
    br = synth.zipf_bias(wl.E, wl.zipf_s, wl.seed)
    x = synth.make_x(wl.T, wl.H, wl.seed)
    r = oracle.route(wl.dims, x, wr, br)
    loads = np.sort(r["counts"])[::-1].astype(float)
    nz = loads > 0
    slope = np.polyfit(np.log(np.arange(1, wl.E + 1)[nz]), np.log(loads[nz]), 1)[0]
    print(f"prefill load: fitted log-log slope {slope:.3f}, max {loads[0]:.0f}, min {loads[nz][-1]:.0f}")
    assert -1.15 <= slope <= -1.05
    assert r["counts"].sum() == wl.T * wl.K


def test_gap_control_separates_scores():
    from tests.inputs import gap_controlled_x
    wl = WORKLOADS["decode_T64"]
    wr = synth.normal_bf16((wl.E, wl.H), 0.02, synth.stream_key(wl.seed, 0, "router_w"))
    x, attempts = gap_controlled_x(wl.dims, wr, None, wl.seed)
    g = top_gaps(oracle.router_logits(wl.dims, x, wr), wl.K)
    assert (g >= 1e-3).all()
    print(f"rows redrawn: {(attempts > 0).sum()} of {wl.T}")


# ---------------------------------------------------------------------------------------
# Load-balancing statistics (inputs of the auxiliary loss): closed forms and invariants


def test_stats_uniform_scores_closed_form():
    """All scores equal: every expert has probability 1/E and every token picks experts
    0..K-1, so P = 1/E, f = 1/K on the first K experts and 0 elsewhere, and the loss is the
    coefficient itself."""
    H, E, K, T = 8, 32, 4, 5
    w = _zero_layer(H, E, 4, 4)
    s = oracle.router_stats((T, H, E, K, 4, 4), synth.make_x(T, H, 1), w["router_w"])
    np.testing.assert_array_equal(s["P"], np.full(E, 1.0 / E))
    np.testing.assert_array_equal(s["f"], np.r_[np.full(K, 1.0 / K), np.zeros(E - K)])
    assert s["loss"] == pytest.approx(0.001, rel=1e-15)


def test_stats_two_experts_reduce_to_the_logistic_function():
    """E = 2, K = 1, one-hot tokens: the softmax of two scores is the logistic function of
    their difference, so P_0 is the mean of sig(l_t0 - l_t1) over the tokens."""
    H, E, K = 16, 2, 1
    wr = torch.zeros(E, H, dtype=torch.bfloat16)
    wr[0, 0] = 1.0  # expert 0 scores x[0]
    wr[1, 1] = 1.0  # expert 1 scores x[1]
    x = torch.zeros(3, H, dtype=torch.bfloat16)
    x[0, 0] = 2.0  # scores (2, 0): expert 0
    x[1, 0] = 4.0  # scores (4, 0): expert 0
    x[2, 0], x[2, 1] = 0.5, 1.0  # scores (0.5, 1): expert 1
    s = oracle.router_stats((3, H, E, K, 4, 4), x, wr)
    p0 = (sig(2.0) + sig(4.0) + sig(-0.5)) / 3
    np.testing.assert_allclose(s["P"], [p0, 1.0 - p0], rtol=1e-14)
    np.testing.assert_array_equal(s["f"], [2 / 3, 1 / 3])
    assert s["loss"] == pytest.approx(0.002 * (2 / 3 * p0 + 1 / 3 * (1 - p0)), rel=1e-14)


def test_stats_invariants_and_expert_relabelling():
    """Random layers: P and f are distributions over the experts, f * T * K are the routing
    counts, and relabelling the experts (permuting the router rows and the bias) permutes P
    and f and leaves the loss unchanged."""
    T, H, E, K = 24, 128, 32, 4
    dims = (T, H, E, K, 64, 64)
    w = _rand_layer(H, E, 64, 64, 9, router_std=0.5)
    br = synth.zipf_bias(E, 1.1, 9)
    x = synth.make_x(T, H, 9)
    s = oracle.router_stats(dims, x, w["router_w"], br)
    assert s["P"].sum() == pytest.approx(1.0, abs=1e-13) and s["f"].sum() == pytest.approx(1.0, abs=1e-13)
    assert (s["P"] > 0).all() and (s["f"] >= 0).all()
    counts = oracle.route(dims, x, w["router_w"], br)["counts"]
    np.testing.assert_array_equal(np.rint(s["f"] * T * K).astype(np.int64), counts)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(E))
    s2 = oracle.router_stats(dims, x, w["router_w"][perm], br[perm])
    np.testing.assert_allclose(s2["P"], s["P"][perm.numpy()], rtol=1e-12, atol=1e-18)
    np.testing.assert_array_equal(s2["f"], s["f"][perm.numpy()])
    assert s2["loss"] == pytest.approx(s["loss"], rel=1e-12)


# ---------------------------------------------------------------------------------------
# bf16-typed router outputs: the pages' interface types the router and the shared gate as
# Linear<..., T> with T = bf16 and ranks bf16 logits ("Qwen3.6 35B-A3B", Blocks: SparseMoe).
# Under this reading each score, bias included, is rounded to the nearest bf16 before the
# softmax, the ranking and the sigmoid. The cases below are worked by hand; H = 2 tokens with
# x = (1, 1) make every score the sum of a row's two entries (plus the bias).

BF16 = oracle.BF16_SCORES


def _two_column_router(rows):
    """Router weight [E, 2] with the given (w0, w1) rows and x = (1, 1): score_e = w0 + w1."""
    return bf16(np.array(rows, np.float64)), bf16(np.ones((1, 2)))


def test_bf16_scores_rounding_makes_a_tie_broken_by_the_lower_index():
    # exact scores 1, 1 + 2^-10, 1/2, 1 + 2^-9: bf16 has 8 significant bits, so the three
    # near 1 all round to 1.0 and tie; the tie goes to the lower indices 0 and 1
    wr, x = _two_column_router([[1.0, 0.0], [1.0, 2.0 ** -10], [0.5, 0.0], [1.0, 2.0 ** -9]])
    exact = oracle.route((1, 2, 4, 2, 4, 4), x, wr)
    typed = oracle.route((1, 2, 4, 2, 4, 4, BF16), x, wr)
    assert exact["ids"].tolist() == [[3, 1]]
    assert typed["ids"].tolist() == [[0, 1]]
    np.testing.assert_array_equal(typed["w"], [[0.5, 0.5]])  # equal scores, equal weights
    # K = 3 takes all three tied experts in index order; their weights stay equal
    typed3 = oracle.route((1, 2, 4, 3, 4, 4, BF16), x, wr)
    assert typed3["ids"].tolist() == [[0, 1, 3]]
    np.testing.assert_allclose(typed3["w"], [[1 / 3, 1 / 3, 1 / 3]], rtol=1e-15)


def test_bf16_scores_round_after_the_bias_to_even():
    # expert 1 scores 1 + 2^-8 only through its bias: the exact midpoint between 1 and the next
    # bf16 (1 + 2^-7), which rounds to the even neighbour 1.0 and ties with expert 0. Rounding
    # before adding the bias would leave 1 + 2^-8 and pick expert 1.
    wr, x = _two_column_router([[1.0, 0.0], [1.0, 0.0], [0.25, 0.0]])
    br = bf16([0.0, 2.0 ** -8, 0.0])
    assert oracle.route((1, 2, 3, 1, 4, 4), x, wr, br)["ids"].tolist() == [[1]]
    assert oracle.route((1, 2, 3, 1, 4, 4, BF16), x, wr, br)["ids"].tolist() == [[0]]
    # above the midpoint (1 + 3 * 2^-9) it rounds up to 1 + 2^-7 and wins again
    br_up = bf16([0.0, 3 * 2.0 ** -9, 0.0])
    assert oracle.route((1, 2, 3, 1, 4, 4, BF16), x, wr, br_up)["ids"].tolist() == [[1]]


def test_bf16_scores_shared_gate_is_rounded_before_the_sigmoid():
    H, E, I, Is = 2, 4, 4, 4
    w = _zero_layer(H, E, I, Is)
    w["shared_gate"] = bf16([[1.0, 2.0 ** -10]])  # z = 1 + 2^-10 exactly, 1.0 in bf16
    x = bf16(np.ones((1, H)))
    exact = oracle.forward((1, H, E, 2, I, Is), x, w, taps=True)
    typed = oracle.forward((1, H, E, 2, I, Is, BF16), x, w, taps=True)
    assert exact["sg"][0] == pytest.approx(sig(1.0 + 2.0 ** -10), rel=1e-15)
    assert typed["sg"][0] == pytest.approx(sig(1.0), rel=1e-15)


def test_bf16_scores_change_nothing_when_every_score_is_a_bf16_value():
    # one-hot tokens: every score is one bf16 weight, already representable, so both readings
    # route identically (ids, weights and dispatch)
    H, E, K, T = 16, 64, 6, 16
    wr = synth.normal_bf16((E, H), 0.02, synth.stream_key(9, 0, "router_w"))
    x = torch.zeros(T, H, dtype=torch.bfloat16)
    for t in range(T):
        x[t, (3 * t) % H] = 1.0
    a = oracle.route((T, H, E, K, 4, 4), x, wr)
    b = oracle.route((T, H, E, K, 4, 4, BF16), x, wr)
    for k in ("ids", "counts", "offsets", "perm", "inv"):
        np.testing.assert_array_equal(a[k], b[k])
    np.testing.assert_array_equal(a["w"], b["w"])
