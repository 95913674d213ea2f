"""bench.py on CPU: the N > 1 path (independent replicas, one per GPU) with
two gloo ranks (the slowest rank's time and the sum of all ranks' tokens
make the whole-job throughput); the reference arm's JSON line (the CPU
oracle on bounded samples); the warm-up floor; and the library's arm
failing loudly, with no result line, where there is no GPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, lr = bench.dist_setup()
    assert (w, r, lr) == (world, rank, rank)
    local_ms = 100.0 + 50.0 * rank          # rank 1 is the slow one
    local_tokens = 16 * 1024 * 50
    bench.barrier(world)
    ms, tokens, value = bench.aggregate(local_ms, local_tokens, world)
    out.put((rank, ms, tokens, value))
    dist.destroy_process_group()


def test_replica_aggregation_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, tokens, value in res:
        assert ms == 150.0                    # max over ranks
        assert tokens == 2 * 16 * 1024 * 50   # sum over ranks
        assert abs(value - tokens / 0.150) < 1e-6 * value


def _run_bench(*args, timeout=300):
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    return subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], cwd=root,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_json_line_with_the_contract_keys():
    import json
    r = _run_bench("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    out = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in out, k
    assert out["impl"] == "reference"
    assert out["steps"] == 1 and out["warmup"] == 3 and out["n_gpus"] == 1
    assert out["value"] > 0 and out["higher_is_better"] is True
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["cores"] >= 1
    assert out["cpu_baseline"]["value"] == out["value"]
    assert out["e2e"] == dict(value=out["value"], unit=out["unit"], h2d_bytes_per_step=0, d2h_bytes_per_step=0)
    assert out["config"]["workload"]


def test_bench_rejects_fewer_than_three_warmup_steps():
    r = _run_bench("--impl", "reference", "--steps", "1", "--warmup", "2", timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the behaviour without a GPU")
def test_our_arm_fails_loudly_without_a_gpu():
    # no CPU fallback: without a device the library's arm exits non-zero and prints no result line
    r = _run_bench("--steps", "1", "--warmup", "3", "--no-cpu-baseline", timeout=120)
    assert r.returncode != 0
    assert not any(l.startswith("{") for l in r.stdout.splitlines())


def test_mfu_report_of_the_124m_step():
    import bench
    w = bench.WORKLOADS["gpt2-124M-B16-T1024"]
    assert bench.num_params(w) == 124_439_808          # the parameter count the 124M run log prints
    assert bench.flops_per_token(w) == 798_031_872.0   # 3 x (matmuls + causal attention), Vp = 50304
    peaks = dict(bf16=1772.9, bf16_sustained=1366.0, hbm_gbs=6338.5, source="measured")
    r = bench.mfu_report(919_310.0, w, peaks)
    assert abs(r["vs_bf16_burst"] - 0.4138) < 1e-4 and abs(r["vs_bf16_sustained"] - 0.5371) < 1e-4
    assert r["six_n"]["flops_per_token"] == 6 * 124_439_808
    assert abs(r["six_n"]["vs_bf16_burst"] - 919_310.0 * 6 * 124_439_808 / 1772.9e12) < 1e-4


def test_decode_step_bytes_at_position_530():
    import bench
    d = bench.DECODE
    matrices = 2 * (50304 * 768 + 12 * (2304 + 768 + 3072 + 3072) * 768)   # bf16 wte and the four Linears
    kv = 2 * 12 * 16 * 530 * (768 + 768)                                   # bf16 keys and values of rows 0..529
    new_row = 2 * 12 * 16 * 2304                                           # the new q, k, v row of every layer
    small = 4 * (12 * (2304 + 768 + 3072 + 768 + 4 * 768) + 2 * 768) + 4 * (16 + 1) * 768
    assert matrices == 247_136_256 and kv == 312_606_720
    assert bench.decode_step_bytes(d, 530) == matrices + kv + new_row + small == 561_165_312


def test_clock_sampler_summary_from_nvidia_smi_lines():
    import threading

    import bench

    class FakeProc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

        def kill(self):
            pass

    s = bench.ClockSampler(0)
    s.proc = FakeProc()
    s.t = threading.Thread(target=lambda: None)
    s.t.start()
    na = "Not Active"
    s.lines = [
        "0, 1942, 2032, 1010.5, 0x0000000000000004, %s, %s, %s, Active" % (na, na, na),
        "0, 1965, 2032, 1050.1, 0x0000000000000000, %s, %s, %s, %s" % (na, na, na, na),
        "0, 1905, 2032, 1094.2, 0x0000000000000004, %s, %s, %s, Active" % (na, na, na),
        "0, [N/A], 2032, 990.0, 0x0, %s, %s, %s, %s" % (na, na, na, na),   # unreadable: skipped
        "garbage",                                                         # short: skipped
    ]
    r = s.stop()
    assert r == dict(sm_mhz=1942.0, sm_max_mhz=2032.0, reasons=["sw_power_cap"], samples=3)
    s.lines.append("0, 1200, 2032, 700.0, 0x8, Active, %s, %s, %s" % (na, na, na))
    assert s.stop()["reasons"] == ["hw_slowdown", "sw_power_cap"]
    s.lines = []
    assert s.stop() is None


def test_traffic_is_reported_only_while_the_sources_are_unchanged(tmp_path, monkeypatch):
    import json

    import bench
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k() {}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = dict(sources=["k.cu"], digest=bench.source_digest(["k.cu"]), bytes_per_launch=12345)
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"attention_bwd": rec}))
    assert bench.load_traffic("attention_bwd") == 12345.0
    assert bench.load_traffic("layernorm_bwd") is None          # no record for this class
    src.write_text("__global__ void k() { }\n")                  # the kernel changed since the capture
    assert bench.load_traffic("attention_bwd") is None


def test_reference_arm_other_ranks_exit_without_work():
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1", MASTER_PORT="29599")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], cwd=root, env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
