"""Property-based check of the plan builder (hypothesis): for any parameter
list, rank count, HSDP group, persistence threshold and bucket sizes, the
C++ plan equals the oracle's field by field and its tiles cover shard and
persistent space exactly once.  Skipped where hypothesis is not installed."""
from __future__ import annotations

import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

from tests.test_abi_host import _check_tiles, _compare  # noqa: E402


@st.composite
def plans(draw):
    N = draw(st.sampled_from([1, 2, 3, 4, 5, 8, 16, 64]))
    divisors = [g for g in range(1, N + 1) if N % g == 0]
    group = draw(st.sampled_from([0] + divisors))
    numel = draw(st.lists(st.integers(0, 6000), min_size=0, max_size=25))
    ds = draw(st.permutations(list(range(len(numel))))) if draw(st.booleans()) else None
    return dict(numel=numel, N=N, group=group, ds_id=ds,
                threshold=draw(st.integers(0, 3000)), B=draw(st.integers(1, 20000)),
                G=draw(st.integers(1, 40000)), U=draw(st.integers(1, 20000)))


@settings(max_examples=150, deadline=None)
@given(plans())
def test_cpp_plan_equals_oracle_for_any_list(c):
    op, cp = _compare(c["numel"], c["N"], ds_id=c["ds_id"], threshold=c["threshold"], B=c["B"],
                      G=c["G"], U=c["U"], group=c["group"])
    _check_tiles(op, cp)
