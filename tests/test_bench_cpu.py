"""Host-side parts of bench.py that need no GPU: the oracle timings it reports
beside each further row's GPU figure."""
import sys

from conftest import ROOT

sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_row_cpu_baselines_small_case():
    """On a small shape every row gets a positive oracle figure with its unit,
    the thread count it used and a description of the sample."""
    rows = bench.row_cpu_baselines(H=2, T=64, d=32, dec_B=32, dec_H=2)
    assert set(rows) == {"softplus_gate", "short_conv", "backward", "decode"}
    units = {"softplus_gate": "tokens/s", "short_conv": "GB/s", "backward": "tokens/s",
             "decode": "GB/s"}
    for key, row in rows.items():
        assert row["kind"] == "oracle"
        assert row["unit"] == units[key]
        assert row["value"] > 0 and row["cores"] >= 1
        assert row["sample"]
    assert rows["decode"]["ms_per_step"] > 0
