"""The pages' printed memory figures, recomputed as N * V * bytes * tensors.

These pin the logit-space byte accounting (decimal GB) used to report that the
fused path never holds an N x V buffer.
"""
import json
import os

import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_memory_figures.json")


def logit_space_bytes(N, V, bytes_per_elem, tensors=1):
    return N * V * bytes_per_elem * tensors


with open(GOLDEN) as fh:
    FIGS = json.load(fh)["figures"]


@pytest.mark.parametrize("fig", FIGS, ids=[f"{f['N']}x{f['V']}x{f['tensors']}" for f in FIGS])
def test_printed_figure(fig):
    gb = logit_space_bytes(fig["N"], fig["V"], fig["bytes_per_elem"], fig["tensors"]) / 1e9
    # the pages print two decimals (one for the 6.3 GB figure)
    digits = 1 if fig["printed_gb"] == 6.3 else 2
    assert round(gb, digits) == pytest.approx(fig["printed_gb"], abs=10 ** -digits * 0.51)
