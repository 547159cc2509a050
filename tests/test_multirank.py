"""The benchmark's GPU arm times the one-GPU hot path only: with more than one rank, or
--gpus > 1, it refuses before any GPU or process-group work. The reference arm (the CPU oracle) runs on
rank 0 alone under torchrun; the other ranks exit without work. CPU only."""
import json

import bench


def test_gpu_arm_refuses_more_than_one_gpu_flag(monkeypatch, capsys):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    assert bench.main(["--gpus", "2"]) == 2
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "ours" and line["n_gpus"] == 2 and "one-GPU" in line["error"]


def test_gpu_arm_refuses_torchrun_ranks(monkeypatch, capsys):
    for rank, prints in ((0, True), (1, False)):
        monkeypatch.setenv("WORLD_SIZE", "2")
        monkeypatch.setenv("RANK", str(rank))
        assert bench.main(["--gpus", "2"]) == 2
        out = capsys.readouterr().out.strip()
        assert bool(out) == prints          # rank 0 alone says why
        if prints:
            assert "one-GPU" in json.loads(out)["error"]


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1"]) == 0
    assert capsys.readouterr().out == ""
