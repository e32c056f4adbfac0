"""The roofline sweep tool on a GB300, on two small shapes.

It runs every FP32 entry point and the vendor library's product (the comparison column) and
checks each result against the product's; the test asserts that the run succeeds, that every
point is reported with a positive rate under its roof, and that no check reports a mismatch.
"""
from __future__ import annotations

import json

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def test_sweep_small_shapes(tmp_path, capsys):
    from roofline_driven_tiling_gb300 import sweep

    out = tmp_path / "sweep.jsonl"
    rc = sweep.main(["--shapes", "256x256x256,200x300x100", "--iters", "3", "--no-flush",
                     "--out", str(out)])
    assert rc == 0
    recs = [json.loads(line) for line in out.read_text().splitlines()]
    assert {tuple(r["shape"]) for r in recs} == {(256, 256, 256), (200, 300, 100)}
    assert {r["kernel"] for r in recs} == set(sweep.KERNELS)
    for r in recs:
        assert r["check"] != "MISMATCH", r
        assert r["tflops"] > 0 and r["ms_min"] <= r["ms_median"], r
        assert r["frac_of_roof"] < 1.0 or r["kernel"] == "tf32x3", r
    # The product's own point carries the tiling it took.
    assert all("plan" in r for r in recs if r["kernel"] == "ffma")
    assert "| 256x256x256 |" in capsys.readouterr().out
