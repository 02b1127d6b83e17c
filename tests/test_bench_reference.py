"""The benchmark's reference arm (the oracle on the host cores) on CPU: it
does the warm-up steps it is given, times exactly the steps it is given, and
bounds each step to a sample of rows when whole steps would not fit its time
budget.  Small workloads; no GPU is used."""
import json

import bench
from sparse_attention_top_idx_gb300 import workloads as wl


def _small():
    return wl.make_workload("refarm", [300, 700, 300, 700, 300, 700], [1] * 6, topk=64, seed=11)


def test_whole_steps_when_they_fit():
    W = _small()
    rate, cores, r, el = bench.oracle_decode_steps(W, steps=2, warmup=3, budget_s=60.0)
    assert r == W.batch and rate > 0 and cores >= 1 and el > 0


def test_sampled_rows_when_whole_steps_do_not_fit():
    W = _small()
    # a budget far below one whole step: the sample shrinks to the fewest rows
    rate, cores, r, el = bench.oracle_decode_steps(W, steps=3, warmup=3, budget_s=1e-6)
    assert r == 1 and rate > 0
    # a budget for about half the rows: an even row count below the batch
    _, _, full_r, full_el = bench.oracle_decode_steps(W, steps=1, warmup=1, budget_s=60.0)
    assert full_r == W.batch
    _, _, r2, _ = bench.oracle_decode_steps(W, steps=4, warmup=1, budget_s=full_el * 5 * 0.5)
    assert 1 <= r2 <= W.batch and (r2 == 1 or r2 % 2 == 0)


def test_reference_line_reports_the_given_steps(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setattr(wl, "decode_batch", _small)
    args = bench.argparse.Namespace(steps=2, warmup=3, gpus=1)
    assert bench.run_reference(args) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] == line["cpu_baseline"]["value"] == line["e2e"]["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
