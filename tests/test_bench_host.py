"""Host logic of bench.py: the multi-rank path (gloo, world size 2, on CPU), the
algorithmic byte/flop model, and the JSON contract of the reference arm."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from context_scan_gb300 import synth  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    w, r = bench.init_dist("gloo")
    bench.barrier()
    m = bench.reduce_max(1.0 + r)          # rank 1 is "slower"
    value = bench.aggregate(tokens_per_rank_step=100, steps=4, world=w, max_seconds=m)
    q.put((r, w, m, value, bench.rank_seed_offset(r)))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_max_and_weak_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    for r, w, m, value, off in out:
        assert w == 2
        assert m == 2.0                    # max over ranks
        assert value == 100 * 4 * 2 / 2.0  # all ranks' tokens / slowest rank's time
    assert out[0][4] != out[1][4]          # every rank draws its own batch


def test_algorithmic_model_matches_hand_count():
    w = synth.WORKLOADS["cp4_b2_h32_t32k"]
    tok_heads = 2 * 32768 * 32
    for pieces in (4, 8):
        plan = (pieces, 512 // pieces, 512 // pieces)
        stages, executed, method = bench.algorithmic(w, plan)
        # every token passes the forward once: piece 0 in phase 1, the rest in phase 2; q,k,v
        # bf16 (3*128*2) + g,beta bf16 (2*2) in, o fp32 (128*4) out
        fwd = stages["phase1"]["bytes"] + stages["phase2"]["bytes"]
        assert fwd >= tok_heads * (772 + 512) + tok_heads * (pieces - 2) // pieces * 516
        assert stages["phase2"]["bytes"] >= tok_heads * (pieces - 1) // pieces * (772 + 512)
        # the method's path total does not depend on how the library cuts the sequence:
        # summaries of 3 of the 4 segments (k, v, g, beta), the scan, the forward
        t_roof = method["bytes"] / 6791.4e9
        assert 520e-6 < t_roof < 540e-6
        assert method["bytes"] >= tok_heads * 3 // 4 * 516 + tok_heads * (772 + 512)
        # the WY stage: k, g, beta in; per chunk out, two bf16 factors, each 64 x 64 but for
        # its zero blocks above the diagonal: 16-column slabs of 64, 48, 32 and 16 rows
        factor = sum(64 - 16 * j for j in range(4)) * 16 * 2
        assert factor == 5120
        assert stages["wy"]["bytes"] == tok_heads * 260 + tok_heads // 64 * 2 * factor
        assert executed["bytes"] == sum(stages[k]["bytes"] for k in ("phase1", "scan", "phase2"))
    assert bench.algorithmic(w, (8, 64, 64))[2] == bench.algorithmic(w, (4, 128, 128))[2]
    # the unequal plan the library takes on 152 SMs: piece 0 of 154 chunks, two of 179; only
    # piece 1 is summarised, so the executed bytes are well below the method's (3/4 summarised)
    stages, executed, method = bench.algorithmic(w, (3, 154, 179))
    kv = 64 * 128 * 128 * 4
    hand = (64 * 154 * 64 * 1284 + 2 * kv + 64 * 179 * 64 * 516 + 2 * kv      # phase 1
            + 2 * kv + kv + kv + 4 * kv                                         # scan
            + 2 * 64 * 179 * 64 * 1284 + 3 * kv)                                # phase 2
    assert executed["bytes"] == hand
    assert 3.12e9 < executed["bytes"] < 3.15e9 < method["bytes"]
    # WY, piece 0's forward, the summaries, the scan, the second forward
    assert bench.launches_per_step(w, 8) == 5
    # CUDA-core shapes have no WY launch; one piece is a single forward
    assert bench.launches_per_step(synth.WORKLOADS["tiny_f32_k64_cp4"], 4) == 4
    assert bench.launches_per_step(synth.WORKLOADS["single_seg_h16_t8k"], 1) == 2


def test_wy_tail_rule_and_launch_count():
    # the last piece's WY tiles go beside the first phase when that phase leaves SMs idle and
    # the tiles fill at least one wave of WY CTAs (six per SM): the headline plan on 152 SMs
    w = synth.WORKLOADS["cp4_b2_h32_t32k"]
    plan = (3, 170, 171)
    assert bench.wy_tail_beside(w, plan, 152)
    # the first phase as one grid replaces its two launches, plus the WY grid for the tail
    assert bench.launches_per_step(w, 3, plan, 152) == 5
    # no idle SMs (128 chains on 128 SMs), or too few tiles (one 8K sequence of 16 heads)
    assert not bench.wy_tail_beside(w, plan, 128)
    # several waves, the last one partial: 512 chains on 152 SMs leave 96 idle in the fourth
    w4 = synth.WORKLOADS["cp2_b16_h32_t4k"]
    assert bench.wy_tail_beside(w4, (2, 32, 32), 152)
    assert bench.launches_per_step(w4, 2, (2, 32, 32), 152) == 5
    # ... but not when the last wave is all but full (4 idle)
    assert not bench.wy_tail_beside(synth.scaled(w4, B=4, H=37), (2, 32, 32), 152)
    w1 = synth.WORKLOADS["single_seg_h16_t8k"]
    assert not bench.wy_tail_beside(w1, (8, 16, 16), 152)
    # two pieces: the forward of piece 0 alone, then the tail's WY grid
    w2 = synth.scaled(w, B=1, H=16)
    assert bench.wy_tail_beside(w2, (2, 256, 256), 152)
    assert bench.launches_per_step(w2, 2, (2, 256, 256), 152) == 5
    # CUDA-core shapes never
    assert not bench.wy_tail_beside(synth.WORKLOADS["tiny_f32_k64_cp4"], (4, 1, 1), 152)
    # per-channel gates at bf16 inputs: the pre-pass, piece 0's forward, the summaries, the scan
    # and the second forward
    assert bench.launches_per_step(synth.WORKLOADS["kda_h16_t8k"], 8) == 5


def test_literal_flow_model_matches_hand_count():
    # every segment's summary (k, v, g, beta over all tokens; M and S written), the scan
    # (3 summaries read, h0 read, 4 H_in written), the forward (every token; H_in read,
    # h_final written)
    w = synth.WORKLOADS["cp4_b2_h32_t32k"]
    tok_heads = 2 * 32768 * 32
    kv = 64 * 128 * 128 * 4
    calls, total = bench.literal_algorithmic(w)
    assert calls["summary"]["bytes"] == tok_heads * 516 + 4 * 2 * kv
    assert calls["scan"]["bytes"] == 3 * 2 * kv + kv + 4 * kv
    assert calls["forward"]["bytes"] == tok_heads * 1284 + 4 * kv + kv
    assert total["bytes"] == sum(c["bytes"] for c in calls.values())


def test_state_grad_model_matches_hand_count():
    # the backward state-gradient kernel, counted by hand per chunk of 64 tokens and head at
    # K = V = 128, every product as a dense tile (the triangular C^T dO and A^T dR alike):
    # K K^T and Q K^T 2*(64*64*128*2) = 2.10 M, the inverse 0.17 M,
    # dR = Kd D + C^T dO 64*128*128*2 + 64*64*128*2 = 3.15 M, A^T dR 64*64*128*2 = 1.05 M,
    # the D update 2*(128*64*128*2) = 4.19 M: 10.66 M per chunk, 167 kFLOP per token-head
    w = synth.WORKLOADS["cp4_b2_h32_t32k"]
    tok_heads = 2 * 32768 * 32
    alg = bench.state_grad_algorithmic(w)
    per_chunk = 2 * 64 * 64 * 128 * 2 + 0.17e6 + 64 * 128 * 128 * 2 + 64 * 64 * 128 * 2 + \
        64 * 64 * 128 * 2 + 2 * 128 * 64 * 128 * 2
    assert abs(alg["flops"] - per_chunk * tok_heads / 64) < 1e3
    assert 166e3 < alg["flops"] / tok_heads < 168e3
    # q, k (2 x 128 bf16), g, beta (bf16) and dO (128 fp32) read once; dS (4 segments x 64
    # heads x 64 KiB) written
    assert alg["bytes"] == tok_heads * (512 + 4 + 512) + 4 * 64 * 128 * 128 * 4
    # fp32 CUDA-core peak from unit counts and the maximum SM clock
    assert abs(bench.FP32_ALU_TFLOPS - 80.55) < 0.01


@pytest.mark.parametrize("steps", [3])
def test_reference_arm_json_line(steps):
    env = dict(os.environ)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_f32_k64_cp4", "--steps", str(steps), "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_kernel_roofline_picks_the_binding_limit():
    # 1 TFLOP and 1 GB: at 100 TFLOP/s and 1000 GB/s the tensor rate binds (10 ms vs 1 ms)
    alg = {"flops": 1e12, "bytes": 1e9}
    r = bench.kernel_roofline(alg, 20.0, 1000.0, 100.0)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - 50.0) < 1e-6 and abs(r["frac"] - 0.5) < 1e-6
    # at 10 000 TFLOP/s the bytes bind (1 ms vs 0.1 ms)
    r = bench.kernel_roofline(alg, 2.0, 1000.0, 10000.0)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 500.0) < 1e-6 and abs(r["frac"] - 0.5) < 1e-6
    # no tensor rate: the fp32 CUDA-core peak
    r = bench.kernel_roofline(alg, 1000.0, 1000.0)
    assert r["bound"] == "alu" and abs(r["achieved"] - 1.0) < 1e-9
    assert abs(r["frac"] - 1.0 / bench.FP32_ALU_TFLOPS) < 1e-4   # frac is rounded to 4 places


def test_backward_piece_rule():
    from context_scan_gb300 import synth
    w = synth.WORKLOADS["cp4_b2_h32_t32k"]
    assert bench.bwd_pieces(w, 152) == 1          # 64 heads x 2 tiles = 128 chains: one wave
    small = synth.scaled(w, B=2, H=2, T=1024)     # 8 chains, 16 chunks
    assert bench.bwd_pieces(small, 152) == 16
    assert bench.bwd_pieces(synth.scaled(small, T=64 * 12), 152) == 4   # 12 chunks: 2-adic 4
    f32 = synth.scaled(small, in_dtype="f32")     # 32-column tiles: 16 chains
    assert bench.bwd_pieces(f32, 152) == 8


def test_record_traffic_one_launch_and_sum(tmp_path):
    # an ncu CSV of two launches, DRAM read and write bytes of each in the units ncu prints
    rows = [
        '"ID","Kernel Name","Grid Size","Metric Name","Metric Unit","Metric Value"',
        '"0","void k1(P)","(128, 1, 1)","dram__bytes_read.sum","Mbyte","10.5"',
        '"0","void k1(P)","(128, 1, 1)","dram__bytes_write.sum","byte","2,000"',
        '"1","void k2(P)","(144, 1, 1)","dram__bytes_read.sum","Kbyte","3"',
        '"1","void k2(P)","(144, 1, 1)","dram__bytes_write.sum","Gbyte","0.001"',
    ]
    csv_path = tmp_path / "t.csv"
    csv_path.write_text("==PROF== a line ncu prints\n" + "\n".join(rows) + "\n")

    def per_launch(path):
        return float([ln for ln in open(path) if ln.startswith("dram_bytes_per_launch:")][0]
                     .split(":")[1])

    one = bench.record_traffic(str(csv_path), "gdn_forward", "w", "cmd", grid="(144, 1, 1)",
                               out_dir=str(tmp_path))
    assert per_launch(one) == 3e3 + 1e6
    both = bench.record_traffic(str(csv_path), "gdn_varlen_forward", "w", "cmd", grid="sum",
                                out_dir=str(tmp_path))
    assert per_launch(both) == 10.5e6 + 2000 + 3e3 + 1e6
    assert "2 launches" in open(both).read()
    with pytest.raises(SystemExit):   # two launches and no grid: ambiguous
        bench.record_traffic(str(csv_path), "gdn_forward", "w", "cmd", out_dir=str(tmp_path))
