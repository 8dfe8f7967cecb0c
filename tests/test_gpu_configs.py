"""The five benchmark workloads at full size, launched exactly as bench.py
launches them (automatic cluster width), compared with the oracle on every
segment."""
import pytest

from segmented_radix_top_gb300 import workloads as W
from tests.gpu_util import check_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg,kw", [(1, {}), (2, {}), (3, {}), (4, {}),
                                    (5, {"mode": "nondet"}), (5, {"mode": "det"})],
                         ids=["w1", "w2", "w3", "w4", "w5-nondet", "w5-det"])
def test_full_size_workload(cfg, kw):
    wl = W.by_number(cfg, **kw)
    check_workload(wl, where="workload %d %s" % (cfg, kw))
