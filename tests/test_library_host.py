"""Host-side checks of libeagle that need no GPU: the library builds, loads
and exports every function include/eagle.h declares; plans and shape
validation behave as documented."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from eagle_feature_level_gb300.build import build
    build()
    import eagle_feature_level_gb300 as E
    return E


def declared_functions():
    text = open(os.path.join(ROOT, "include", "eagle.h")).read()
    return sorted(set(re.findall(r"^\s*(?:eagle_status|const char\*|long long)\s+(eagle_\w+)\(", text, re.M)))


def test_exports_match_header(lib):
    so = lib._binding.LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", so], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (eagle_\w+)", out))
    decl = declared_functions()
    assert decl, "no declarations parsed"
    missing = [f for f in decl if f not in exported]
    assert not missing, missing
    assert set(decl) == set(lib._binding.EXPORTED)


def test_status_strings(lib):
    assert lib.eagle_status_string(0) == "ok"
    assert "capacity" in lib.eagle_status_string(4)


def test_plan_eagle2_layout(lib):
    p = lib.eagle_plan_eagle2(10, 6, 60)
    assert (p.kind, p.top_k, p.depth, p.top_m, p.n_expanded, p.n_layers) == (0, 10, 6, 60, 51, 6)
    assert list(p.layer_e0[:6]) == [0, 1, 11, 21, 31, 41]
    assert list(p.layer_rows[:6]) == [1, 10, 10, 10, 10, 10]
    big = lib.eagle_plan_eagle2(10, 8, 255)      # 71 expanded slots, 256 tree slots
    assert (big.n_expanded, big.top_m, big.layer_e0[7]) == (71, 255, 61)
    for args in ((16, 18, 60),                    # 273 expanded slots > 256
                 (10, 8, 256)):                   # 257 tree slots > 256
        with pytest.raises(lib.EagleError) as e:
            lib.eagle_plan_eagle2(*args)
        assert e.value.name == "EAGLE_ERR_CAPACITY"


def test_plan_static_matches_template_shape(lib):
    from eagle_feature_level_gb300.runtime import plan_for
    p = plan_for("static26")
    assert (p.top_k, p.depth, p.top_m, p.n_expanded) == (4, 5, 26, 14)
    assert list(p.layer_rows[:5]) == [1, 4, 4, 4, 1]
    assert list(p.layer_e0[:5]) == [0, 1, 5, 9, 13]
    p8 = plan_for("static8")
    assert (p8.top_k, p8.n_expanded, list(p8.layer_rows[:3])) == (3, 4, [1, 2, 1])
    t4 = plan_for("ternary4")                    # 120 nodes: template indices past int8
    assert (t4.top_k, t4.depth, t4.top_m, t4.n_expanded) == (3, 4, 120, 40)
    assert list(t4.layer_rows[:4]) == [1, 3, 9, 27] and list(t4.layer_e0[:4]) == [0, 1, 4, 13]
    assert t4.node_parent[119] == 38 and t4.node_exp[38] == 39


def test_plan_static_rejects_bad_templates(lib):
    for parents, ranks in (([0], [0]),           # parent after itself
                           ([-1, -1], [0, 0]),   # duplicate (parent, rank)
                           ([-1, 0, -1], [0, 0, 1])):   # not listed by depth
        with pytest.raises(lib.EagleError) as e:
            lib.eagle_plan_static(parents, ranks)
        assert e.value.name == "EAGLE_ERR_INVALID_TREE"


def test_create_validates_shapes_before_the_device(lib):
    B = lib._binding
    good = dict(d=64, n_q_heads=4, n_kv_heads=4, head_dim=16, d_ff=172, vocab=512, rms_eps=1e-5,
                rope_theta=1e4)
    lim = B.eagle_limits(1, 4, 4, 3, 9, 64)
    for bad in (dict(d=96), dict(head_dim=24), dict(n_kv_heads=3), dict(vocab=40000)):
        dd = dict(good, **bad)
        dims = B.eagle_dims(dd["d"], dd["n_q_heads"], dd["n_kv_heads"], dd["head_dim"], dd["d_ff"],
                            dd["vocab"], dd["rms_eps"], dd["rope_theta"])
        with pytest.raises(B.EagleError) as e:
            B.eagle_create(dims, lim)
        assert e.value.name == "EAGLE_ERR_SHAPE"
    dims = B.eagle_dims(*[good[k] for k in ("d", "n_q_heads", "n_kv_heads", "head_dim", "d_ff", "vocab",
                                            "rms_eps", "rope_theta")])
    with pytest.raises(B.EagleError) as e:
        B.eagle_create(dims, B.eagle_limits(1, 300, 4, 3, 9, 64))
    assert e.value.name == "EAGLE_ERR_CAPACITY"
