"""Host logic of the timeline tool: the event report from a synthetic event array."""
import numpy as np

from sparse_top_mla_gb300 import timeline


def test_report_groups_exits_by_work_share():
    # four CTAs over 10 tiles of 4-tile items: ranges [0,2) [2,5) [5,7) [7,10), i.e. 2, 3, 2, 3
    # tiles in 1, 2, 1, 2 item segments
    n, total, tpi = 4, 10, 4
    rel = np.full((n, 256), np.nan)
    rel[:, 0] = 0.0
    rel[:, 2] = [10.0, 20.0, 30.0, 40.0]
    for c in range(n):
        rel[c, 8:8 + 24 * 3:24] = [1.0, 3.0 + c, 5.0 + 2 * c]  # S^T ready of tiles 0-2
    out = timeline.report(rel, total, tpi)
    assert "exit, 2 tiles in 1 item segment(s), 2 CTAs: 10.00 / 20.00 / 30.00" in out
    assert "exit, 3 tiles in 2 item segment(s), 2 CTAs: 20.00 / 30.00 / 40.00" in out
    assert "3 tiles in 1 item" not in out and "2 tiles in 2 item" not in out
    # mean period per CTA: (4 + 2c) / 2 = 2, 3, 4, 5
    assert "min 2.00 median 3.50 max 5.00" in out
    assert "tile 0: Sready=  1.00" in out
