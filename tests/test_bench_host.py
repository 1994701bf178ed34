"""Host-side pieces of bench.py that need no GPU: the committed DRAM-traffic
summary it reports as roofline.traffic, and the bytes it counts per run."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _summary(path):
    fields = {}
    for ln in open(path):
        if ":" in ln and not ln.startswith("#"):
            k, v = ln.split(":", 1)
            fields[k.strip()] = v.strip()
    return fields


def test_traffic_summary_is_current_and_close_to_the_algorithmic_bytes():
    # The ncu figure is reported only while the kernel sources are the ones it
    # was taken on; a kernel change without a new capture shows up here.
    import bench
    f = _summary(os.path.join(ROOT, "profiles", "lp_stream_kernel_large_dram.txt"))
    assert f["kernel_source_sha256"] == bench.kernel_source_hash(), "re-take the DRAM capture for the current kernel"
    traffic = bench.measured_traffic("large")
    alg = int(f["algorithmic_bytes_per_launch"])
    assert traffic == int(f["traffic_bytes_per_launch"])
    # the logits are read once; a few percent of writes (tile partials, counters)
    assert alg <= traffic <= 1.05 * alg
    # the scaling from the captured cut is the ratio of algorithmic bytes
    cut = int(f["cut dram__bytes_read.sum"]) + int(f["cut dram__bytes_write.sum"])
    scaled = cut * alg / int(f["cut algorithmic_bytes_per_launch"])
    assert abs(scaled - traffic) <= 1


def test_traffic_is_withheld_for_other_sources(monkeypatch):
    import bench
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 64)
    assert bench.measured_traffic("large") is None
    assert bench.measured_traffic("no_such_config") is None


@pytest.mark.parametrize("name", ["spec", "large", "decode"])
def test_algorithmic_bytes_counts_the_rows_the_oracle_emits(name):
    # In these workloads every group is read (it requests a record or has
    # drafts), so the rows read are exactly the rows the oracle emits: each
    # group's accepted prefix and the row after it.
    import bench
    import parity as PT
    import workloads as W
    w = W.decode() if name == "decode" else getattr(W, name)(groups=8)
    sizes = np.diff(w.group_indptr)
    assert ((w.requested != 0) | (sizes > 1)).all()
    orc = PT.run_oracle(w)
    ab = bench.algorithmic_bytes(w, orc["accepted"])
    assert ab["rows_read"] == int((orc["emitted_tokens"] >= 0).sum())
    assert ab["logit_bytes"] == ab["rows_read"] * w.V * w.elt
    assert ab["total"] > ab["logit_bytes"]


if __name__ == "__main__":
    sys.exit(pytest.main([__file__, "-q"]))
