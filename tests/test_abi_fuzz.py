"""Host-side validation of topo_cfg against the rules include/topo.h states:
random configurations, most of them one field away from a valid one.  A cfg
that breaks a stated rule must be rejected (workspace size 0); one that keeps
every rule and is well inside the shared-memory budget must be accepted.  No
GPU is needed: topo_workspace_bytes only validates and sizes."""
import pytest

import moe_expert_routing_ids_gb300 as topo

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

FIELDS = ("T", "E", "k", "R", "ranks_per_node", "n_slot", "tok_bytes", "expert_bytes",
          "c_intra", "c_inter", "max_refine_iters")


def stated_rules_hold(c):
    T, E, k, R, rpn, ns = c["T"], c["E"], c["k"], c["R"], c["ranks_per_node"], c["n_slot"]
    tb, eb, ci, ce, mi = c["tok_bytes"], c["expert_bytes"], c["c_intra"], c["c_inter"], c["max_refine_iters"]
    if not (T >= 0 and E >= 1 and 1 <= k <= 64 and R >= 1 and 1 <= rpn <= 32 and ns >= 0):
        return False
    if R % rpn or E % R or T % R or T * k > 2**31 - 1 or E >= 2**26:
        return False
    if not (tb >= 0 and eb >= 0 and ci >= 1 and ce >= ci and mi >= 0):
        return False
    if tb * ce >= 2**31 or eb * ce >= 2**40:
        return False
    return R * ns <= 2**20 and E // R + ns <= 32767


def well_inside_the_budget(c):
    return (c["E"] <= 512 and c["R"] <= 128 and c["ranks_per_node"] <= 16 and
            c["E"] // c["R"] + c["n_slot"] <= 100 and c["T"] <= 1 << 24)


@st.composite
def configs(draw):
    rpn = draw(st.sampled_from([1, 2, 4, 8, 16]))
    R = rpn * draw(st.integers(1, 8))
    E = R * draw(st.integers(1, 8))
    T = R * draw(st.integers(0, 4096))
    c = dict(T=T, E=E, k=draw(st.integers(1, min(E, 16))), R=R, ranks_per_node=rpn,
             n_slot=draw(st.integers(0, 40)), tok_bytes=draw(st.integers(0, 1 << 16)),
             expert_bytes=draw(st.integers(0, 1 << 30)), c_intra=draw(st.integers(1, 3)),
             c_inter=0, max_refine_iters=draw(st.integers(0, 50)))
    c["c_inter"] = c["c_intra"] + draw(st.integers(0, 5))
    if draw(st.booleans()):                              # one field off its valid range
        f = draw(st.sampled_from(FIELDS))
        c[f] = draw(st.one_of(st.integers(-3, 0), st.integers(-(2**31), 2**31 - 1),
                              st.sampled_from([33, 65, 1 << 20, 2**26, 2**31 - 1])))
        if f in ("tok_bytes", "expert_bytes"):
            c[f] = draw(st.one_of(st.integers(-(2**40), -1), st.integers(2**28, 2**45)))
    return c


def _workspace(c, L):
    cfg = dict(c, main_rank=None)
    return topo.topo_workspace_bytes(topo.make_cfg(**cfg), L, topo.TOPO_CALL_CHAIN)


@settings(max_examples=400, deadline=None)
@given(configs(), st.integers(1, 4))
def test_cfg_validation_follows_the_stated_rules(c, L):
    try:
        topo.lib()
    except RuntimeError:
        pytest.skip("library not built")
    n = _workspace(c, L)
    if not stated_rules_hold(c):
        assert n == 0, c
    elif well_inside_the_budget(c):
        assert n > 0, c
