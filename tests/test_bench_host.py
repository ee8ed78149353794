"""Host logic of bench.py that needs no GPU: the algorithmic byte counts
behind every GB/s figure and the roofline's numerator, the MoE expert count
they use, the whole-job rate, and the traffic record lookup."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_dense_byte_counts():
    # NVFP4: M*K/2 code bytes + M*K/16 scale bytes + 4 (fp32 tensor scale)
    # + 2NK (bf16 x) + 4NM (fp32 y)
    assert bench.nvfp4_bytes(12288, 4096, 1) == 25165824 + 3145728 + 4 + 8192 + 49152 == 28368900
    assert bench.nvfp4_bytes(4096, 4096, 8) == 8388608 + 1048576 + 4 + 65536 + 131072
    # Q8_0: M*K int8 + M*K/32 fp16 scales + x + y (the LM head figures of
    # the committed DRAM summary)
    assert bench.q8_0_bytes(151936, 4096, 1) == 622329856 + 38895616 + 8192 + 607744 == 661841408
    assert bench.q8_0_bytes(32, 64, 2) == 2048 + 128 + 256 + 256


def test_moe_expert_bytes():
    # gate_up [2I][H] and down [H][I], NVFP4 each, plus two fp32 tensor scales
    H, I = 2048, 512
    gate_up = 2 * I * H // 2 + 2 * I * H // 16
    down = H * I // 2 + H * I // 16
    assert gate_up == 1048576 + 131072 and down == 524288 + 65536
    assert bench.moe_expert_bytes(H, I) == gate_up + down + 8 == 1769480


def test_moe_unique_experts_and_bytes():
    # token 0 picks experts 0 and 2; token 1 has a tie between experts 1
    # and 2 and picks both (2 slots): three distinct experts in all
    logits = np.array([[3.0, 1.0, 2.0, 0.0], [0.0, 2.0, 2.0, 1.0]], dtype=np.float32)
    assert bench.moe_unique_experts(logits, 2) == 3
    assert bench.moe_unique_experts(logits, 1) == 2  # experts 0 and 1 (the tie goes to the lower index)
    assert bench.moe_unique_experts(logits[:1], 4) == 4
    T, E, H, I = 2, 4, 32, 32
    assert bench.moe_bytes(T, E, H, I, 2, logits) == 3 * bench.moe_expert_bytes(H, I) + T * H * 2 + T * H * 4 + T * E * 4


def test_whole_job_rate():
    # every rank streams the step's bytes; the job's rate divides all ranks'
    # bytes by the slowest rank's time
    assert bench.whole_job_gbs(10**9, 2, 10, 4.0) == 5.0
    assert bench.whole_job_gbs(10**9, 1, 1, 0.5) == 2.0
    assert bench.max_over_ranks(1.25, 1, None) == 1.25


def test_step_rows_cover_the_workload():
    names = [n for n, _, _ in bench.rows_spec()]
    assert names == ["nvfp4 12288x4096 N=1", "nvfp4 4096x12288 N=1", "nvfp4 4096x4096 N=1",
                     "q8_0 12288x4096 N=1", "q8_0 4096x12288 N=1", "q8_0 151936x4096 N=1",
                     "nvfp4 4096x4096 N=4", "nvfp4 4096x4096 N=8", "nvfp4 12288x4096 N=4",
                     "nvfp4 12288x4096 N=8", "moe T=1", "moe T=16"]


def test_traffic_record_lookup():
    import json
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    rows = {n: (k, p) for n, k, p in bench.rows_spec() + bench.extra_rows_spec()}
    assert rec, "no traffic record"
    for name, ent in rec.items():
        assert name in rows, f"traffic record {name!r} is not a bench row"
        kind, p = rows[name]
        if kind == "q8_0":
            assert ent["algorithmic_bytes"] == bench.q8_0_bytes(p["M"], p["K"], p["N"])
        elif kind in ("nvfp4", "nvfp4_tiny"):
            assert ent["algorithmic_bytes"] == bench.nvfp4_bytes(p["M"], p["K"], p["N"])
        if kind not in ("moe", "moe_prefill"):  # every other row: the bench's own byte count of the row
            assert ent["algorithmic_bytes"] == bench.row_bytes(kind, p, None)
        # per-call means, each rounded to a byte
        assert abs(ent["dram_bytes_per_launch"] - (ent["dram_read"] + ent["dram_write"])) <= 1
        # the hash covers the named sources in a fixed order
        assert bench.source_sha(ent["sources"]) == bench.source_sha(list(reversed(ent["sources"])))
        assert bench.source_sha(ent["sources"]) != bench.source_sha(ent["sources"][:1])
    assert bench.profiled_traffic("no such kernel") is None


def test_rotating_copies_exceed_three_l2():
    l2 = 129 * 2**20
    for call_bytes, weight_bytes in ((28_368_900, 28_311_552), (661_841_408, 661_225_472), (14_170_000, 453e6)):
        r = bench.rotating_copies(call_bytes, weight_bytes, l2, 40e9)
        assert r >= 2 and (r - 1) * call_bytes > 3 * l2
    assert bench.rotating_copies(10**6, 10**10, l2, 40e9) == 4  # capped by the memory budget, at least 2


def test_moe_launch_count():
    # T = 1, 4 and 16 at top-8 with H = 2048, I = 512: the two batched kernels
    assert bench.moe_launches(1, 256, 2048, 512, 8) == 2
    assert bench.moe_launches(4, 256, 2048, 512, 8) == 2
    assert bench.moe_launches(16, 256, 2048, 512, 8) == 2
    # beyond the batched kernels' limits: route, gate_up, down, combine
    assert bench.moe_launches(32, 256, 2048, 512, 8) == 4
    assert bench.moe_launches(1, 256, 2048, 384, 8) == 4


def test_write_traffic_splits_rows_at_the_separator(tmp_path, monkeypatch):
    # a fake ncu CSV of --profile-all with two rows, two calls each: torch's
    # setup kernels are dropped, each row's bytes are halved
    rows = [("nvfp4 256x512 N=1", "nvfp4_tiny", dict(M=256, K=512, N=1)),
            ("q8_0 32x64 N=2", "q8_0", dict(M=32, K=64, N=2))]
    monkeypatch.setattr(bench, "rows_spec", lambda: rows[:1])
    monkeypatch.setattr(bench, "extra_rows_spec", lambda: rows[1:])
    hdr = ["ID", "Process ID", "Process Name", "Host Name", "Kernel Name", "Context", "Stream", "Block Size",
           "Grid Size", "Device", "CC", "Section Name", "Metric Name", "Metric Unit", "Metric Value"]
    launches = [("void at::native::fill", 5, 0), ("void bqd::nvfp4_dequant_kernel(int)", 7, 1),
                ("void bqd::gemv_direct_kernel<A>(int)", 100, 4), ("void bqd::gemv_direct_kernel<A>(int)", 102, 6),
                ("void bqd::nvfp4_dequant_kernel(int)", 7, 1), ("void at::native::copy", 9, 9),
                ("void bqd::gemv_kernel<B>(int)", 1000, 0), ("void bqd::gemv_kernel<B>(int)", 1000, 0)]
    lines = [",".join(f'"{c}"' for c in hdr)]
    for i, (k, rd, wr) in enumerate(launches):
        for m, v in (("dram__bytes_read.sum", rd), ("dram__bytes_write.sum", wr)):
            lines.append(",".join(f'"{c}"' for c in [i, 1, "python", "h", k, 1, 7, "(1, 1, 1)", "(1, 1, 1)", 0,
                                                    "10.3", "Command line profiler metrics", m, "byte", v]))
    csv_path = tmp_path / "all.csv"
    csv_path.write_text("\n".join(lines) + "\n")
    out = tmp_path / "traffic.json"
    bench.write_traffic(str(csv_path), 2, out_path=str(out))
    import json
    rec = json.loads(out.read_text())
    a, b = rec["nvfp4 256x512 N=1"], rec["q8_0 32x64 N=2"]
    assert (a["dram_read"], a["dram_write"], a["launches_per_call"]) == (101, 5, 1)
    assert (b["dram_read"], b["dram_write"], b["launches_per_call"]) == (1000, 0, 1)
    assert a["algorithmic_bytes"] == bench.nvfp4_bytes(256, 512, 1)
    assert b["algorithmic_bytes"] == bench.q8_0_bytes(32, 64, 2)
    assert a["kernels"] == ["gemv_direct_kernel<A>"] and b["kernels"] == ["gemv_kernel<B>"]


def test_traffic_record_sources_match_the_rows():
    # every record names the kernel sources its row runs (the files exist),
    # so that a change to any of them retires the record
    import json
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    rows = {n: (k, p) for n, k, p in bench.rows_spec() + bench.extra_rows_spec()}
    csrc = os.path.join(ROOT, "block_quantized_decode_nvfp4_gb300", "csrc")
    for name, ent in rec.items():
        kind, p = rows[name]
        assert ent["sources"] == bench.traffic_sources(kind, p), name
        assert all(os.path.exists(os.path.join(csrc, f)) for f in ent["sources"]), name
    assert bench.traffic_sources("fp8_b128", dict(M=4096, K=12288, N=1)) == bench.TRAFFIC_SOURCES["direct"]
    assert bench.traffic_sources("moe_prefill", dict(T=1024))[0] == "moe_prefill.cu"


# A small instance of every row kind and the library call its row makes.
SMALL_ROWS = {
    "nvfp4": (dict(M=32, K=64, N=1), "nvfp4_gemv"),
    "nvfp4_tiny": (dict(M=256, K=512, N=1), "nvfp4_gemv"),
    "nvfp4_silu": (dict(M=64, K=64, N=1), "nvfp4_gemv_silu_mul"),
    "nvfp4_add": (dict(M=32, K=64, N=1), "nvfp4_gemv_add"),
    "q8_0": (dict(M=32, K=64, N=2), "q8_0_gemv"),
    "q4_0": (dict(M=32, K=64, N=1), "q4_0_gemv"),
    "q4_1": (dict(M=32, K=64, N=1), "q4_1_gemv"),
    "fp8_b128": (dict(M=130, K=256, N=1), "fp8_b128_gemv"),
    "nvfp4_gemm": (dict(M=32, K=64, N=16), "nvfp4_gemm"),
    "nvfp4_gemm_grouped": (dict(E=4, M=32, K=64, N=64), "nvfp4_gemm_grouped"),
    "nvfp4_encode": (dict(M=32, K=64, N=1), "nvfp4_encode"),
    "q8_0_encode": (dict(M=32, K=64, N=1), "q8_0_encode"),
    "moe": (dict(T=2, E=8, H=64, I=64, topk=2), "moe_layer"),
    "moe_prefill": (dict(T=4, E=8, H=64, I=64, topk=2), "moe_prefill_layer"),
}


def test_every_row_kind_builds_and_calls_its_entry_point(monkeypatch):
    # Row construction and run() on the CPU: torch's cuda calls kept on the
    # host, the library replaced by a recorder; the call it records must be
    # an entry point of the package, and every row kind of the bench is here
    import torch
    import block_quantized_decode_nvfp4_gb300 as real
    kinds = {k for _, k, _ in bench.rows_spec() + bench.extra_rows_spec()}
    assert kinds <= set(SMALL_ROWS), kinds - set(SMALL_ROWS)
    monkeypatch.setattr(torch.Tensor, "cuda", lambda self, *a, **k: self)
    empty = torch.empty
    monkeypatch.setattr(torch, "empty", lambda *a, **k: empty(*a, **{n: v for n, v in k.items() if n != "device"}))
    calls = []

    class Recorder:
        def __getattr__(self, name):
            def f(*a, **k):
                calls.append(name)
                return 4096 if name.endswith("workspace_bytes") else None
            return f

    for kind, (p, entry) in SMALL_ROWS.items():
        row = bench.Row(f"small {kind}", kind, p, bench.host_inputs(kind, p), torch, Recorder())
        calls.clear()
        row.run()
        assert calls == [entry], (kind, calls)
        assert callable(getattr(real, entry)), entry
        assert row.bytes > 0 and row.weight_bytes > 0 and row.out_bytes > 0
