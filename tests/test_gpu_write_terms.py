"""GPU parity of the scaled, weight-decayed write P' = P (1 - lr wd) - lr s O
in bf16 mode, on inputs where every term of it is many bf16 ulps of P'.

With the configs' scalars (lr = 0.02, P of std 0.02) the update lr s O and
the decay lr wd P are each about one bf16 ulp of P', so a wrong scale s, a
dropped or doubled decay, or a decay applied after the update would stay
inside the bf16 P' bound.  Here lr = wd = 0.5 and P has std 1e-2: lr s O is
then tens to hundreds of ulps of P' and lr wd P at least several, so each
of those mistakes moves P' outside the bound (one bf16 ulp of P' plus
lr s |dO|).
Each kernel that writes P is covered: the Gram-space skinny kernel (both
orientations, m = 24 and m = 64), the direct skinny iteration (k = 70), the
resident kernel (both orientations, vector and element-wise forms), the
tensor path (both orientations), merged [r, c] + [c, r] buckets, and both
non-trivial scale modes."""
import numpy as np
import pytest

from newton_schulz_bucket_gb300 import workloads as W
from oracle import muon_ref
from oracle_pins import SCHEDULE

from parity import GpuRun, check_all

pytestmark = pytest.mark.gpu

BIG = dict(lr=0.5, wd=0.5, p_std=1e-2)


def _terms_visible(run, scale_mode):
    """The update and decay terms are each far above one bf16 ulp of P'."""
    w = run.w
    for (i, e) in run.members:
        shp = w.shapes[i]
        s = muon_ref.scale_factor(shp[-2], shp[-1], scale_mode)
        O = run.O(i, e)
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(run.p1(i, e)), 2.0 ** -126))) - 7)
        upd = w.lr * s * np.sqrt(np.mean(O ** 2))
        dec = w.lr * w.wd * np.sqrt(np.mean(run.p0(i, e) ** 2))
        med = np.median(ulp)
        assert upd > 20 * med and dec > 3 * med, (shp, upd, dec, med)


@pytest.mark.parametrize("scale_mode", ["sqrt_aspect", "rms_0_2"])
def test_write_terms_gram_space_skinny(scale_mode):
    w = W.custom([[24, 4096], [4096, 24], [2, 64, 1504], [1504, 64]], seed=41, **BIG)
    run = GpuRun(w, scale=scale_mode)
    assert {g["path"] for g in run.plan.groups()} == {"skinny"}
    _terms_visible(run, scale_mode)
    check_all(run, scale_mode=scale_mode)
    run.close()


@pytest.mark.parametrize("scale_mode", ["sqrt_aspect", "rms_0_2"])
def test_write_terms_resident_path(scale_mode):
    w = W.custom([[128, 768], [768, 128], [100, 700]], seed=45, **BIG)
    run = GpuRun(w, scale=scale_mode, path="resident")
    assert {g["path"] for g in run.plan.groups()} == {"resident"}
    _terms_visible(run, scale_mode)
    check_all(run, scale_mode=scale_mode)
    run.close()


def test_write_terms_direct_skinny_iteration():
    w = W.custom([[24, 2048], [1024, 40]], seed=42, ns_steps=70, **BIG)
    w.coeffs = SCHEDULE
    run = GpuRun(w)
    _terms_visible(run, "sqrt_aspect")
    check_all(run)
    run.close()


@pytest.mark.parametrize("scale_mode", ["sqrt_aspect", "rms_0_2"])
def test_write_terms_tensor_path(scale_mode):
    w = W.custom([[256, 768], [768, 256]], seed=43, **BIG)
    run = GpuRun(w, scale=scale_mode)
    assert {g["path"] for g in run.plan.groups()} == {"tensor"}
    _terms_visible(run, scale_mode)
    check_all(run, scale_mode=scale_mode)
    run.close()


@pytest.mark.parametrize("shapes", [[[24, 3000], [3000, 24]], [[256, 640], [640, 256]]],
                         ids=["skinny", "tensor"])
def test_write_terms_merged_buckets(shapes):
    w = W.custom(shapes, seed=44, **BIG)
    run = GpuRun(w, merge_transposed=True, scale="rms_0_2")
    assert len(run.plan.groups()) == 1 and run.plan.groups()[0]["transposed"] == "mixed"
    _terms_visible(run, "rms_0_2")
    check_all(run, scale_mode="rms_0_2")
    run.close()
