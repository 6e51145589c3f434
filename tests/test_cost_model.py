"""The alpha-beta cost-model helper (host only) against the values the
lecture notes print for their worked examples and exercise answers
(tests/golden/lecture14_cost_model_answers.txt), rounded as printed."""
import math
import os
import re

import pytest

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "lecture14_cost_model_answers.txt")


@pytest.fixture(scope="module")
def dpr():
    from gradient_reduction_gb300 import build
    build.build()
    import gradient_reduction_gb300 as g
    return g


def _golden():
    out = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        lhs, rhs = line.split("=", 1) if line.count("=") == 1 else line.rsplit("=", 1)
        name = lhs.split()[0]
        params = dict(re.findall(r"(\w+)=([0-9.e+-]+)", lhs))
        val, unit = rhs.split()
        out[name] = ({k: float(v) for k, v in params.items()}, float(val), unit)
    return out


G = _golden()


def _printed(name, got, unit_scale=1.0):
    """got (in the golden's unit) rounds to the printed value at its precision."""
    _, want, _ = G[name]
    text = [l for l in open(GOLDEN) if l.startswith(name + " ")][0].split("=")[-1].split()[0]
    decimals = len(text.split(".")[1]) if "." in text and "e" not in text else 0
    if "e" in text:                       # magnitudes printed as e.g. 235e3: within 1 unit
        step = 10 ** int(text.split("e")[1])
        assert abs(got - want) < step, (name, got, want)
    else:                                 # within half a unit of the last printed digit
        assert abs(got - want) <= 0.5 * 10 ** -decimals + 1e-9, (name, got, want)


def test_section_3_1_segmented_broadcast(dpr):
    p = G["sec3.1_unsegmented"][0]
    t1 = dpr.dpr_cost_ring_broadcast(8, p["N"], p["alpha"], p["B"], 1)
    _printed("sec3.1_unsegmented", t1 * 1e3)
    t64 = dpr.dpr_cost_ring_broadcast(8, p["N"], p["alpha"], p["B"], 64)
    _printed("sec3.1_segmented", t64 * 1e3)
    s, t = dpr.dpr_cost_best_segments(8, p["N"], p["alpha"], p["B"])
    assert s == 64 and t == t64
    # the segment count is an interior optimum: the continuous minimum of
    # (K-2+S)(alpha + N/(S B)) is at S* = sqrt((K-2) N / (alpha B)) ~ 55
    s_star = math.sqrt(6 * p["N"] / (p["alpha"] * p["B"]))
    assert 32 < s_star < 64


def test_section_3_4_crossover_and_regimes(dpr):
    p = G["sec3.4_ring_tree_cross"][0]
    n = dpr.dpr_cost_crossover("ring", "tree", 8, p["alpha"], p["beta"])
    _printed("sec3.4_ring_tree_cross", n)
    # the section's regimes: 1-10 KB naive fastest, 100 KB tree, >= 1 MB ring
    for size, best in ((1e3, "naive"), (1e4, "naive"), (1e5, "tree"), (1e6, "ring"), (1e8, "ring")):
        t = {a: dpr.dpr_cost_allreduce(a, 8, size, p["alpha"], p["beta"]) for a in ("ring", "tree", "naive")}
        assert min(t, key=t.get) == best, (size, t)


def test_exercise_5(dpr):
    p = G["ex5_ring"][0]
    t = dpr.dpr_cost_allreduce("ring", 16, p["N"], p["alpha"], p["beta"])
    _printed("ex5_ring", t * 1e3)
    latency = 2 * 15 * p["alpha"]
    _printed("ex5_latency_part", latency * 1e3)
    assert dpr.dpr_cost_allreduce("ring", 16, p["N"], 0.0, p["beta"]) == pytest.approx(t - latency)


def test_exercise_6(dpr):
    p = G["ex6_unsegmented"][0]
    _printed("ex6_unsegmented", dpr.dpr_cost_ring_broadcast(4, p["N"], 0.0, p["B"], 1) * 1e3)
    _printed("ex6_100_segments", dpr.dpr_cost_ring_broadcast(4, p["N"], 0.0, p["B"], 100) * 1e3)
    _printed("ex6_100_segments_alpha",
             dpr.dpr_cost_ring_broadcast(4, p["N"], 20e-6, p["B"], 100) * 1e3)


def test_exercise_7(dpr):
    p = G["ex7_ring_naive_cross"][0]
    n = dpr.dpr_cost_crossover("ring", "naive", 8, p["alpha"], p["beta"])
    _printed("ex7_ring_naive_cross", n)
    assert n == pytest.approx(12 * p["alpha"] * p["beta"] / 12.25)


def test_exercise_8(dpr):
    p = G["ex8_ring"][0]
    _printed("ex8_ring", dpr.dpr_cost_allreduce("ring", 16, p["N"], 0.0, p["beta"]))


@pytest.mark.parametrize("K", [2, 4, 8])
def test_exercise_11(dpr, K):
    p = G[f"ex11_speedup_k{K}"][0]
    _printed(f"ex11_speedup_k{K}", dpr.dpr_cost_dp_speedup(p["T1"], K, p["N"], 0.0, p["beta"]))


@pytest.mark.parametrize("name,K", [("sec4.4_speedup_10MB_k8", 8), ("sec4.4_speedup_100MB_k8", 8),
                                    ("sec4.4_speedup_400MB_k2", 2)])
def test_section_4_4_speedups(dpr, name, K):
    p = G[name][0]
    _printed(name, dpr.dpr_cost_dp_speedup(p["T1"], K, p["N"], p["alpha"], p["beta"]))


def test_invalid_arguments(dpr):
    with pytest.raises(dpr.DprError):
        dpr.dpr_cost_allreduce("ring", 8, 1e6, 5e-6, 0.0)
    with pytest.raises(dpr.DprError):
        dpr.dpr_cost_ring_broadcast(8, 1e6, 5e-6, 25e9, 0)
    with pytest.raises(dpr.DprError):
        dpr.dpr_cost_crossover("ring", "ring", 8, 5e-6, 25e9)
