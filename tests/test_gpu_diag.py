"""The diagnostics the measurements are compared with: the MMA issue-rate probe."""
import numpy as np
import pytest

from qwtest import qw

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode,n", [(0, 64), (0, 128), (0, 256), (1, 128), (1, 256), (2, 256),
                                    (3, 256), (4, 256), (5, 256), (6, 256), (7, 256),
                                    (8 | 1, 256), (8 | 3, 256)])
def test_mma_rate_probe_runs_on_every_sm(mode, n):
    import torch
    Q = qw()
    cyc, ns = Q.mma_rate(mode, n, 1024)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert cyc.size == min(sms, Q.QW_MMA_PROBE_MAX_CTAS)
    assert np.all((cyc > 8) & (cyc < 100000)), cyc
    ghz = np.median(cyc / ns)
    assert 0.3 < ghz < 4.0, ghz
