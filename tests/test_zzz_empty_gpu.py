"""Empty problems on the GPU (N = 0 or B = 0, prefill, backward, host-buffer prefill and
decode): every entry point returns outputs of the right empty shape, launches nothing and
leaves the device error word clear.  The CPU twin of this test runs the same calls against
the library without a GPU."""
import pytest
import torch

import hierarchical_top_block_gb300 as pisa
from test_binding import _empty_calls


@pytest.mark.gpu
def test_empty_problems_on_the_gpu():
    torch.cuda.set_device(0)
    _empty_calls("cuda", host_prefill=True)
    torch.cuda.synchronize()
    assert pisa.pisa_get_last_device_error() == 0
