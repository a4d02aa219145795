"""Host-side checks of bench.py (no GPU): the workloads its headline run
appends resolve, and the roofline arithmetic gives the compulsory bytes of the
headline workload (q, k, v in bf16, g and beta in fp32, bf16 o, fp32 final state)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from chunkwise_gated_delta_gdr_gb300 import inputs as gin  # noqa: E402


def test_other_workloads_resolve():
    names = set(bench.OTHER_WORKLOADS)
    assert len(names) == len(bench.OTHER_WORKLOADS)
    assert gin.HEADLINE not in names
    for name in names:
        assert bench.workload(name).name == name


def test_headline_algorithmic_bytes():
    w = bench.workload(None)
    assert w.name == gin.HEADLINE
    # 2 x 4096 x 12 x 128 x 2 (q, k) + 4096 x 12 x 128 x 2 (v) + 2 x 4096 x 12 x 4 (g, beta)
    # + 4096 x 12 x 128 x 2 (bf16 o) + 12 x 128 x 128 x 4 (final state)
    assert bench.algorithmic_bytes(w, 2) == 51511296
    assert bench.algorithmic_bytes(w, 4) == 51511296 + 4096 * 12 * 128 * 2


def test_skip_flag_parses(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py", "--skip-other-workloads", "--steps", "3"])
    args = bench.parse()
    assert args.skip_other_workloads and args.steps == 3 and args.workload is None
