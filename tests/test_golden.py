"""Figures the pages print, used as fixtures."""
import os

from gqa_split_kv_gb300.accounting import traffic_bytes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_fixture(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            vals[k] = int(v)
    return vals


def test_kv_bytes_of_the_gqa6_workload_match_the_pages_product():
    f = read_fixture("roofline_bytes_gqa6_ctx4096.txt")
    prod = f["keys"] * f["kv_heads"] * f["head_dim"] * f["tensors"] * f["bytes_per_element"]
    assert prod == f["product"]
    tb = traffic_bytes(1, 24, f["kv_heads"], f["head_dim"], [f["keys"]], S=1)
    assert tb["kv"] == f["product"]
