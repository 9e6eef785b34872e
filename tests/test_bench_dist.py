"""Host logic of the multi-rank benchmark path, on CPU with gloo (world size 2):
slowest-rank timing, whole-job rate, and the reference arm running on rank 0 only."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slow = bench.max_over_ranks(1.0 + rank * 2.5)
    dist.destroy_process_group()
    q.put((rank, slow, bench.whole_job_rate(100.0, world, slow)))


def test_max_over_ranks_gloo():
    import multiprocessing as mp
    import random
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = random.randint(20000, 40000)
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
    assert [r[1] for r in res] == [3.5, 3.5]
    assert all(abs(r[2] - 200.0 / 3.5) < 1e-12 for r in res)


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.25) == 4.25


def test_reference_arm_rank1_does_nothing():
    """Under torchrun, ranks other than 0 of the reference arm exit 0 without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_prints_json_line():
    import json
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GB/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_traffic_record_follows_code_not_comments(tmp_path, monkeypatch):
    """The recorded DRAM traffic is reported only while the GEMV kernel's code
    matches the capture: comment or whitespace edits keep the hash, a code edit
    changes it."""
    import shutil
    sys.path.insert(0, ROOT)
    import bench
    csrc = tmp_path / "q4_dequant_gemv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("q4k_gemv.cu", "q4k_dev.cuh", "ptx.cuh"):
        shutil.copy(os.path.join(ROOT, "q4_dequant_gemv_gb300", "csrc", f), csrc / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    src = (csrc / "q4k_gemv.cu").read_text()
    (csrc / "q4k_gemv.cu").write_text("// a new comment line\n" + src.replace("namespace q4k {", "namespace  q4k  {  /* c */"))
    assert bench.kernel_source_hash() == h0
    (csrc / "q4k_gemv.cu").write_text(src.replace("constexpr int kStages = 4;", "constexpr int kStages = 5;"))
    assert bench.kernel_source_hash() != h0
    # the device helpers shared by the kernel count as its code too
    (csrc / "q4k_gemv.cu").write_text(src)
    dev = (csrc / "q4k_dev.cuh").read_text()
    (csrc / "q4k_dev.cuh").write_text(dev.replace("constexpr int kI8Pair = 80;", "constexpr int kI8Pair = 96;"))
    assert bench.kernel_source_hash() != h0
