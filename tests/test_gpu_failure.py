"""Failure reporting without a GPU fault: a kernel waits on an mbarrier, or
on a global flag, that nothing signals.  The bounded wait must give up,
record FLASH_GAU_ETIMEOUT in the status word, and leave the context usable
(a forward afterwards still matches the oracle)."""

import numpy as np
import pytest
import torch

from efficient_attention_transformer_gb300 import binding as bd
from gpu_harness import Case, TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from efficient_attention_transformer_gb300.build import build
    build()


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_gives_up_and_reports(which):
    words = torch.zeros(2, dtype=torch.int32, device="cuda")
    st = bd.lib().flash_gau_selftest_bounded_wait(which, words.data_ptr(),
                                                  torch.cuda.current_stream().cuda_stream)
    assert st == bd.OK
    torch.cuda.synchronize()
    assert int(words[0]) == bd.ETIMEOUT
    assert int(words[1]) == 0
    # the context is intact: a forward still runs and matches the oracle
    case = Case(1, 256, 128, 256, 128, 128, True, "bf16", seed=151)
    O = case.run()
    ref, _ = case.reference()
    assert rel_err(O, ref) <= TOL["bf16"]
    assert case.status() == 0


def test_bounded_wait_rejects_bad_arguments():
    s = torch.cuda.current_stream().cuda_stream
    assert bd.lib().flash_gau_selftest_bounded_wait(0, None, s) == bd.EINVAL
    words = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert bd.lib().flash_gau_selftest_bounded_wait(2, words.data_ptr(), s) == bd.EINVAL
