"""The oracle pins must catch plausible mistakes.

Each case plants one mistake in a COPY of the oracle's C source (a dropped term, a wrong sign,
a wrong operand, a wrong index order, an off-by-one), compiles it on the CPU, and runs the pin
tests of test_oracle_pins.py against it: at least one pin must fail.  The real oracle is not
touched.
"""
import os

import pytest

from oracle import oracle as oracle_mod
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle_mod.__file__), "vsa_oracle.c")

MUTATIONS = {
    "dk_drops_sm_scale": ("dk[trow * D + x] += ds * qr[x] * sm_scale;",
                          "dk[trow * D + x] += ds * qr[x];"),
    "ds_wrong_sign_in_dq": ("double ds = p * (dp - delta);\n          for (int x = 0; x < D; ++x) dqr",
                            "double ds = p * (dp + delta);\n          for (int x = 0; x < D; ++x) dqr"),
    "dp_uses_q_not_do": ("double dp = dot(dor, v + trow * D, D);",
                         "double dp = dot(qr, v + trow * D, D);"),
    "dv_uses_q_not_do": ("dv[trow * D + x] += p * dor[x];", "dv[trow * D + x] += p * qr[x];"),
    "lse_natural_log": ("lse[row] = mz + log2(l);", "lse[row] = mz + log(l);"),
    "delta_uses_q": ("double delta = dot(o + row * D, dor, D);\n      double *dqr",
                     "double delta = dot(o + row * D, qr, D);\n      double *dqr"),
    "invert_descending": ("for (int i = 0; i < nq; ++i) {\n        long r = bh * nq + i;",
                          "for (int i = nq - 1; i >= 0; --i) {\n        long r = bh * nq + i;"),
    "vbs_off_by_one": ("return n < 0 ? 0 : (n > blk ? blk : n);",
                       "return n < 0 ? 0 : (n > blk ? blk : n - (n > 1));"),
    "active_prefix_short": ("for (int s = 0; s < cnt; ++s)\n    if (row[s] == j)",
                            "for (int s = 0; s + 1 < cnt; ++s)\n    if (row[s] == j)"),
    # Right at 64-token blocks only: caught by the 128-token pins.
    "fwd_key_row_assumes_64": ("long t = (long)j * blk + u;\n          double w = exp2(",
                               "long t = (long)j * 64 + u;\n          double w = exp2("),
}


class _Bound:
    """The oracle module's interface, bound to another compiled library."""

    def __init__(self, lib):
        self.lib = lib

    def invert(self, *a, **kw):
        return oracle_mod.invert(*a, lib=self.lib, **kw)

    def fwd(self, *a, **kw):
        return oracle_mod.fwd(*a, lib=self.lib, **kw)

    def bwd(self, *a, **kw):
        return oracle_mod.bwd(*a, lib=self.lib, **kw)


PIN_TESTS = [
    lambda o: pins.test_invert_golden_fixture(o),
    lambda o: pins.test_invert_brute_force(o, 0),
    lambda o: pins.test_forward_matches_dense_masked(o, True, 64),
    lambda o: pins.test_forward_matches_dense_masked(o, True, 128),
    lambda o: pins.test_forward_closed_forms(o),
    lambda o: pins.test_backward_matches_autograd(o, True, None, 64),
    lambda o: pins.test_backward_matches_autograd(o, True, (2,), 128),
    lambda o: pins.test_backward_finite_differences(o),
    lambda o: pins.test_backward_invariants_and_zero_rows(o),
    lambda o: pins.test_backward_closed_forms(o),
]


def test_unmutated_copy_passes_all_pins():
    with open(SRC) as f:
        src = f.read()
    bound = _Bound(oracle_mod.build_variant(src, "identity"))
    for t in PIN_TESTS:
        t(bound)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    old, new = MUTATIONS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, "mutation anchor not unique: " + name
    bound = _Bound(oracle_mod.build_variant(src.replace(old, new), name))
    failures = 0
    for t in PIN_TESTS:
        try:
            t(bound)
        except AssertionError:
            failures += 1
    assert failures > 0, "no pin caught the planted mistake " + name


# The work order is plain Python in oracle.py: its mistakes are planted in a copy of that
# function's source, executed on its own, and the work-order pins must catch each.
WORK_ORDER_MUTATIONS = {
    "order_ascending": ("key=lambda x: -counts[x]", "key=lambda x: counts[x]"),
    "order_ties_descending": ("key=lambda x: -counts[x]", "key=lambda x: (-counts[x], -x)"),
    "order_no_clamp": ("min(max(int(c), 0), int(max_q))", "int(c)"),
    "order_local_ids": ("out.append(bh * nb + j)", "out.append(j)"),
}


class _OrderBound:
    def __init__(self, fn):
        self.work_order = fn


def _work_order_variant(old, new):
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(oracle_mod.work_order))
    assert src.count(old) == 1, "mutation anchor not unique: " + old
    ns = {"np": oracle_mod.np}
    exec(compile(src.replace(old, new), "<work_order variant>", "exec"), ns)  # noqa: S102
    return _OrderBound(ns["work_order"])


def test_unmutated_work_order_copy_passes_its_pins():
    bound = _work_order_variant("key=lambda x: -counts[x]", "key=lambda x: -counts[x]")
    pins.test_work_order_golden_fixture(bound)
    pins.test_work_order_properties(bound, 0)


@pytest.mark.parametrize("name", sorted(WORK_ORDER_MUTATIONS))
def test_planted_work_order_mistake_is_caught(name):
    bound = _work_order_variant(*WORK_ORDER_MUTATIONS[name])
    failures = 0
    for t in (lambda o: pins.test_work_order_golden_fixture(o),
              lambda o: pins.test_work_order_properties(o, 0)):
        try:
            t(bound)
        except AssertionError:
            failures += 1
    assert failures > 0, "no pin caught the planted mistake " + name
