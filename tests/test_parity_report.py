"""The parity report (tests/parity.py): every comparison is recorded with its
figures, failures included, and written as JSON lines to $FA_PARITY_REPORT."""
import json

import numpy as np
import pytest
import torch

import parity


def test_comparisons_are_recorded_and_written(tmp_path, monkeypatch):
    start = len(parity.RECORDS)
    o_ref = np.zeros((1, 1, 4, 8))
    lse_ref = np.zeros((1, 1, 4))
    parity.compare(torch.zeros(1, 1, 4, 8), torch.zeros(1, 1, 4), o_ref, lse_ref, "exact")
    with pytest.raises(AssertionError):
        parity.compare(torch.ones(1, 1, 4, 8), torch.zeros(1, 1, 4), o_ref, lse_ref, "off by one")
    ref = [np.ones((2, 3)), np.ones((2, 3)), np.ones((2, 3))]
    parity.compare_grads([torch.ones(2, 3)] * 3, ref, "grads")
    new = parity.RECORDS[start:]
    assert [r["case"] for r in new] == ["exact", "off by one", "grads dq", "grads dk", "grads dv"]
    assert [r["pass"] for r in new] == [True, False, True, True, True]
    assert new[1]["max_abs_dO"] == 1.0 and new[0]["max_abs_dO"] == 0.0
    assert new[2]["ref_max_abs"] == 1.0 and new[2]["max_abs"] == 0.0

    path = tmp_path / "report.jsonl"
    monkeypatch.setenv("FA_PARITY_REPORT", str(path))
    parity.write_report()
    lines = [json.loads(s) for s in path.read_text().splitlines()]
    assert len(lines) == len(parity.RECORDS) and lines[-1]["case"] == "grads dv"
    del parity.RECORDS[start:]  # these records are about the report, not about the kernels
