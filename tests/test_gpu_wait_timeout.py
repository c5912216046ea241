"""Bounded waits give up: a wait on an mbarrier that nothing arrives on runs out after its poll
limit, the kernel reports SPEC_TREE_S_TIMEOUT through the status word and returns, and the
context stays usable (a build right after it is exact).  No copy is in flight during the wait,
and no fault, trap or hang is involved."""
import pytest
import torch

from dynamic_tree_speculative_gb300 import binding as B
from dynamic_tree_speculative_gb300 import workloads as WL

pytestmark = pytest.mark.gpu

import parity  # noqa: E402  (loads the native library; fails loudly if absent)


@pytest.mark.parametrize("polls", [1, 64])
def test_wait_gives_up_and_reports_timeout(polls):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    result = torch.full((4,), 7, dtype=torch.int32, device="cuda")
    B.spec_tree_wait_selftest(polls, status, result)
    torch.cuda.synchronize()
    assert int(status.item()) == B.S_TIMEOUT
    assert result.cpu().tolist() == [1, polls, 1, polls]
    # the context is intact: a small build and verify right after are exact
    out = parity.run_parity(WL.WORKLOADS["vicuna"].with_(B=2, V=4000, depth=3, R=10, K=4, W=2), 3)
    assert out["build_exact"] == 2


def test_wait_selftest_refuses_bad_arguments():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    result = torch.zeros(4, dtype=torch.int32, device="cuda")
    for polls in (0, (1 << 16) + 1):
        with pytest.raises(B.SpecTreeError):
            B.spec_tree_wait_selftest(polls, status, result)
