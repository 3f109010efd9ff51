"""Host-side tests of the C ABI: the library loads, exports every declared
symbol, and its planner (no device involved) buckets like the oracle's
reference bucketing and the pages' examples; argument errors are statuses."""
import ctypes as C
import json
import os
import re

import pytest

import newton_schulz_bucket_gb300 as pkg
from newton_schulz_bucket_gb300 import _capi
from oracle import muon_ref

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_capi.lib_path()):
        from newton_schulz_bucket_gb300 import build
        build.build()
    return _capi.load()


@pytest.mark.parametrize("header,expected", [("muon.h", "EXPORTED"),
                                             ("muon_testing.h", "EXPORTED_TESTING")])
def test_exports_every_declared_symbol(lib, header, expected):
    hdr = open(os.path.join(ROOT, "include", header), encoding="utf-8").read()
    declared = set(re.findall(r"^\s*(?:[A-Za-z_0-9]+\s*\*?\s+)+\*?(muon_[a-z_0-9]+)\s*\(", hdr, re.M))
    assert declared, "no declarations parsed"
    assert declared == set(getattr(_capi, expected))
    for name in declared:
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.muon_version().decode().count(".") == 2
    for s, name in [(0, "MUON_OK"), (1, "MUON_ERR_INVALID_ARG"), (5, "MUON_ERR_TIMEOUT")]:
        assert lib.muon_status_string(s).decode() == name


def _golden_cases():
    cases = json.load(open(os.path.join(HERE, "golden", "pages_shapes.json"), encoding="utf-8"))
    for case in cases["cases"]:
        s = case["shapes"]
        shapes = [s["shape"]] * s["repeat"] if "repeat" in s else s["list"]
        yield case, shapes


def test_planner_matches_pages_examples(lib):
    for case, shapes in _golden_cases():
        d = pkg.describe(shapes)
        got = [{"rows": g["rows"], "cols": g["cols"], "batch": g["batch"]} for g in d["groups"]]
        assert got == case["groups"], case["cite"]


@pytest.mark.parametrize("shapes", [
    [[4, 8], [3, 8, 4], [4, 8], [2, 3, 8], [8, 4]],
    [[24, 10240]] * 5 + [[32, 24, 10240]] + [[4096, 4096], [16384, 4096]],
    [[7, 5, 3], [5, 3], [3, 5], [1, 1], [1, 9], [9, 1]],
])
def test_planner_matches_oracle_bucketing(lib, shapes):
    d = pkg.describe(shapes)
    ref = muon_ref.bucket_shapes(shapes)
    assert [(g["rows"], g["cols"], g["batch"]) for g in d["groups"]] == \
        [(g["rows"], g["cols"], len(g["members"])) for g in ref]
    flat = [m for g in ref for m in g["members"]]
    assert d["members"] == flat
    first = 0
    for g in d["groups"]:
        assert g["first_member"] == first
        assert g["transposed"] == (g["rows"] > g["cols"])
        first += g["batch"]


@pytest.mark.parametrize("shapes", [
    [[4, 8], [3, 8, 4], [4, 8], [2, 3, 8], [8, 4]],
    [[4096, 16384], [16384, 4096]] * 3 + [[4096, 4096]],
    [[24, 10240], [10240, 24], [2, 24, 10240], [5, 3], [3, 5], [1, 9], [9, 1]],
])
def test_merged_orientation_buckets(lib, shapes):
    """[r, c] and [c, r] share a group keyed by (min, max) with the merge flag;
    the member order and group order match the oracle's merged bucketing."""
    d = pkg.describe(shapes, merge_transposed=True)
    ref = muon_ref.bucket_shapes(shapes, merge_transposed=True)
    assert [(g["rows"], g["cols"], g["batch"]) for g in d["groups"]] == \
        [(g["rows"], g["cols"], len(g["members"])) for g in ref]
    assert d["members"] == [m for g in ref for m in g["members"]]
    for g, rg in zip(d["groups"], ref):
        orient = {shapes[p][-2] > shapes[p][-1] for p, _ in rg["members"]}
        want = "mixed" if len(orient) == 2 else orient.pop()
        assert g["transposed"] == want
    assert len(d["groups"]) == len({(min(s[-2:]), max(s[-2:])) for s in shapes})


def test_planner_paths(lib):
    d = pkg.describe([[24, 10240], [64, 7168], [4096, 4096], [10240, 24]])
    paths = [g["path"] for g in d["groups"]]
    assert paths[0] == "skinny" and paths[1] == "skinny" and paths[3] == "skinny"
    assert paths[2] == "tensor"
    d = pkg.describe([[24, 10240]], mode="fp32")
    assert d["groups"][0]["path"] == "simt"
    d = pkg.describe([[24, 10240]], skinny_threshold=-1)
    assert d["groups"][0]["path"] == "tensor"
    # scratch grows with the batch: the skinny path keeps the 16-bit iterate
    s1 = pkg.describe([[24, 10240]] * 1)["groups"][0]["workspace_bytes"]
    s3 = pkg.describe([[24, 10240]] * 3)["groups"][0]["workspace_bytes"]
    assert s1 >= 24 * 10240 * 2 and s3 >= 3 * 24 * 10240 * 2 and s3 > s1
    w1 = pkg.describe([[512, 512]] * 1)["groups"][0]["workspace_bytes"]
    w4 = pkg.describe([[512, 512]] * 4)["groups"][0]["workspace_bytes"]
    assert w4 >= 4 * (2 * 512 * 512 * 2) and w4 > w1


@pytest.mark.parametrize("bad", [[[0, 4]], [[4]], [[1, 2, 3, 4]], [[2, 0, 3]], []])
def test_planner_rejects_bad_shapes(lib, bad):
    with pytest.raises(pkg.MuonError) as ei:
        pkg.describe(bad)
    assert ei.value.status == _capi.MUON_ERR_INVALID_ARG


def test_bad_options_are_statuses(lib):
    for kw in [dict(eps=-1.0), dict(eps=float("nan")), dict(skinny_threshold=65),
               dict(max_streams=17), dict(column_shards=3), dict(column_shards=16),
               dict(column_shards=-1)]:
        with pytest.raises(pkg.MuonError) as ei:
            pkg.describe([[4, 4]], **kw)
        assert ei.value.status == _capi.MUON_ERR_INVALID_ARG
    with pytest.raises(pkg.MuonError):
        pkg.describe([[4, 4]], mode="fp32", path="skinny")
    o = _capi.muon_plan_options()
    lib.muon_default_options(C.byref(o))
    o.reserved[3] = 1
    sh = (_capi.muon_shape_t * 1)()
    sh[0].ndim = 2; sh[0].dims[0] = 4; sh[0].dims[1] = 4
    ng = C.c_int32()
    st = lib.muon_plan_describe(sh, 1, C.byref(o), None, 0, C.byref(ng), None, None, 0, None, None)
    assert st == _capi.MUON_ERR_INVALID_ARG


def test_null_arguments_are_statuses(lib):
    assert lib.muon_step(None, None, None, None, 0.9, 0.1, 0.0, 5, 1.0, 1.0, 1.0, None) == \
        _capi.MUON_ERR_INVALID_ARG
    assert lib.muon_step_host(None, None, None, None, 0.9, 0.1, 0.0, 5, 1.0, 1.0, 1.0, None) == \
        _capi.MUON_ERR_INVALID_ARG
    assert lib.muon_plan_destroy(None) == _capi.MUON_OK
    assert lib.muon_plan_num_groups(None) == 0
    assert lib.muon_plan_workspace_bytes(None) == 0
    assert lib.muon_plan_create(None, 0, None, 0, None) == _capi.MUON_ERR_INVALID_ARG
    assert lib.muon_debug_copy_update(None, 0, 0, None) == _capi.MUON_ERR_INVALID_ARG
    assert lib.muon_plan_check_error(None) == _capi.MUON_ERR_INVALID_ARG
    assert lib.muon_plan_group_elapsed_ms(None, 0, None) == _capi.MUON_ERR_INVALID_ARG
    assert lib.muon_last_error().decode() != ""
    assert lib.muon_testing_tc_gemm(7, 0, 1, 8, 8, None, None, None, None, 1.0, 0.0, 0.0, 0.0,
                                    None) == _capi.MUON_ERR_INVALID_ARG


def test_describe_large_config_without_device(lib):
    from newton_schulz_bucket_gb300 import workloads as W
    w = W.get("c5_mixed_1000")
    d = pkg.describe(w.shapes)
    assert len(d["groups"]) == 12 and sum(g["batch"] for g in d["groups"]) == 1000
    w = W.get("c4_dense_h4096")
    d = pkg.describe(w.shapes)
    assert [(g["rows"], g["cols"], g["batch"]) for g in d["groups"]] == [
        (4096, 12288, 32), (4096, 4096, 32), (4096, 16384, 32), (16384, 4096, 32)]
    assert d["groups"][3]["transposed"]


def test_resident_path_on_request(lib):
    """The resident path runs only when asked for, on groups with min dim <=
    128 and max dim <= 4096 (either orientation, any width); it keeps no
    scratch of its own (only the optional copy of O)."""
    shapes = [[128, 4096], [4096, 128], [100, 700], [65, 65]]
    assert {g["path"] for g in pkg.describe(shapes)["groups"]} == {"tensor"}
    d = pkg.describe(shapes, path="resident")
    assert [g["path"] for g in d["groups"]] == ["resident"] * 4
    assert all(g["workspace_bytes"] == 0 for g in d["groups"])
    assert pkg.describe(shapes, path="resident", keep_update=True)["groups"][0]["workspace_bytes"] >= \
        4 * 128 * 4096
    for bad in ([129, 4096], [128, 4104], [4104, 128]):
        with pytest.raises(pkg.MuonError) as ei:
            pkg.describe([bad], path="resident")
        assert ei.value.status == 2  # MUON_ERR_UNSUPPORTED
