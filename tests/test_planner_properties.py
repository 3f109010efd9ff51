"""Property checks of the C planner (muon_plan_describe, host only) on random
shape lists: its groups and member order equal the oracle's bucketing
(«MindSpore HyperParallel X 盘古,Muon优化器实现6倍性能跃升», 矩阵融合优化
Fig. 6: same trailing shape, one batch; Muon亲和的专家切分 Fig. 4: [E, M, N]
is E matrices), with and without orientation merging, and every group's
orientation flag and path follow from its members' shapes alone."""
import pytest

import newton_schulz_bucket_gb300 as pkg
from oracle import muon_ref

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies

DIMS = [1, 2, 3, 5, 8, 24, 63, 64, 65, 128, 1000]
dim = st.sampled_from(DIMS)
shape2 = st.lists(dim, min_size=2, max_size=2)
shape3 = st.tuples(st.integers(1, 4), dim, dim).map(list)
shape_lists = st.lists(st.one_of(shape2, shape3), min_size=1, max_size=24)


@hypothesis.settings(max_examples=150, deadline=None, derandomize=True)
@hypothesis.given(shapes=shape_lists, merge=st.booleans())
def test_planner_equals_oracle_bucketing(shapes, merge):
    d = pkg.describe(shapes, merge_transposed=merge)
    ref = muon_ref.bucket_shapes(shapes, merge_transposed=merge)
    assert [(g["rows"], g["cols"], g["batch"]) for g in d["groups"]] == \
        [(g["rows"], g["cols"], len(g["members"])) for g in ref]
    assert d["members"] == [m for g in ref for m in g["members"]]
    first = 0
    for g, rg in zip(d["groups"], ref):
        assert g["first_member"] == first
        first += g["batch"]
        orient = {shapes[p][-2] > shapes[p][-1] for p, _ in rg["members"]}
        assert g["transposed"] == ("mixed" if len(orient) == 2 else orient.pop())
        m = min(g["rows"], g["cols"])
        assert g["path"] == ("skinny" if m <= 64 else "tensor")
        assert g["workspace_bytes"] > 0
    assert first == sum(s[0] if len(s) == 3 else 1 for s in shapes)
    # one workspace holds every group's scratch plus the per-member pointer
    # table (three pointers, the orientation and the scale: 32 bytes each)
    assert d["workspace_bytes"] >= sum(g["workspace_bytes"] for g in d["groups"]) + \
        32 * len(d["members"])


def test_options_add_their_buffers():
    """Nesterov on the skinny path keeps U = G + beta M' (fp32) for the
    direct kernel, and keep_update keeps O (fp32): each adds one fp32 copy of
    the group's data."""
    shapes = [[24, 10240]] * 3 + [[2, 40, 1000]]
    base = pkg.describe(shapes)["groups"]
    for opt in ("nesterov", "keep_update"):
        more = pkg.describe(shapes, **{opt: True})["groups"]
        for g0, g1 in zip(base, more):
            assert g1["workspace_bytes"] - g0["workspace_bytes"] >= \
                4 * g0["batch"] * g0["rows"] * g0["cols"], (opt, g0)


@hypothesis.settings(max_examples=60, deadline=None, derandomize=True)
@hypothesis.given(shapes=shape_lists)
def test_fp32_mode_and_thresholds(shapes):
    """fp32 mode sends every group to the SIMT path; a lower skinny threshold
    moves exactly the groups above it to the tensor path."""
    assert {g["path"] for g in pkg.describe(shapes, mode="fp32")["groups"]} == {"simt"}
    d = pkg.describe(shapes, skinny_threshold=8)
    for g in d["groups"]:
        assert g["path"] == ("skinny" if min(g["rows"], g["cols"]) <= 8 else "tensor")
