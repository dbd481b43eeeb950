"""The oracle's KV-size helper reproduces the worked examples printed on the KV-cache primer
page (cf-1.com/news/5988169, sections 3.2, 3.3 and 5.3)."""
import os

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_cache_bytes.txt")
UNITS = {"B": 1, "GiB": 1 << 30}


def _cases():
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("|")[0].strip()
            if not line or line.startswith("#"):
                continue
            *nums, expected, unit = line.split()
            yield [int(x) for x in nums], int(expected) * UNITS[unit]


def test_worked_examples():
    cases = list(_cases())
    assert len(cases) == 3
    for args, expected in cases:
        assert oracle.kv_cache_bytes(*args) == expected


def test_linear_in_each_factor():
    base = oracle.kv_cache_bytes(1, 32, 32, 128, 4096, 2)
    assert oracle.kv_cache_bytes(8, 32, 32, 128, 4096, 2) == 8 * base   # page: 8 requests -> 16 GB
    assert oracle.kv_cache_bytes(1, 32, 32, 128, 8192, 2) == 2 * base   # doubling length doubles it
