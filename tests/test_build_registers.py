"""Every kernel of the built library compiles without register spills or a stack frame
(ptxas's own report of the build, `_build/ptxas.log`): a spill would put the rows that
the kernels keep in registers through local memory, and the shape tables were chosen so
that none does. Skipped when the library has not been built here."""
import os
import re

import pytest

LOG = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "row_wise_rmsnorm_gb300", "_build", "ptxas.log")


def test_no_spills_in_any_kernel():
    if not os.path.exists(LOG):
        pytest.skip("library not built")
    kernels, bad, cur = 0, [], None
    for line in open(LOG):
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            cur = m.group(1)
            kernels += 1
            continue
        m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and cur is not None:
            if any(int(v) for v in m.groups()):
                bad.append((cur, m.groups()))
            cur = None
    assert kernels > 0, "no kernels in the ptxas report"
    assert not bad, f"{len(bad)} kernels with a stack frame or spills, e.g. {bad[:3]}"
