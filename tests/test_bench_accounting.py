"""The benchmark's algorithmic byte counts (the denominators of its GB/s
figures), checked against per-matrix counts derived by hand from the packed
format: N*K/8 bytes of words, N*(K/128)*2 bytes per fp16 metadata array, and
the bf16 activations in and out once.  CPU only."""
import bench


def test_weight_bytes_per_matrix():
    # 17408 x 5120: 11,141,120 B of words + 1,392,640 B of scales (+ the same of biases)
    assert bench.weight_bytes(17408, 5120, False) == 11_141_120 + 1_392_640
    assert bench.weight_bytes(17408, 5120, True) == 11_141_120 + 2 * 1_392_640
    # 5120 x 5120: 3,276,800 B of words + 409,600 B of scales
    assert bench.weight_bytes(5120, 5120, False) == 3_686_400


def test_decode_step_bytes():
    # per layer, x [K] in and y [N] out in bf16 for each of the four matrices
    gate = 12_533_760 + 5120 * 2 + 17408 * 2    # 12,578,816
    down = 12_533_760 + 17408 * 2 + 5120 * 2
    attn = 3_686_400 + 5120 * 2 + 5120 * 2      # 3,706,880
    assert gate == 12_578_816 and attn == 3_706_880
    assert bench.step_bytes(1) == 64 * (2 * gate + down + attn)
    # M tokens move M times the activations, the weights once
    assert bench.step_bytes(8) - bench.step_bytes(1) == 64 * 7 * 2 * (2 * (5120 + 17408) + (17408 + 5120) + 2 * 5120)
    # affine: one more metadata array per matrix
    assert bench.step_bytes(1, True) - bench.step_bytes(1) == 64 * (3 * 1_392_640 + 409_600)


def test_decode_chain_bytes():
    # per layer: all four matrices once; h and a in/out of the attention
    # product, a in and the FFN intermediate out of gate/up, the intermediate
    # in and h out of the down product (bf16, M = 1)
    w = 2 * 12_533_760 + 12_533_760 + 3_686_400
    act = 2 * (5120 + 5120) + 2 * (5120 + 17408) + 2 * (17408 + 5120)
    assert bench.chain_bytes(1) == 64 * (w + act)


def test_reference_arm_prints_the_contract_line():
    # the reference arm times the oracle on the host: one JSON line with the
    # GPU arm's metric and unit, marked as the reference, warm-up of at least 3
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, cwd=root, check=True, timeout=300).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["steps"] == 1 and d["warmup"] >= 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["config"]["workload"] == bench.WORKLOAD
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_clock_summary_reports_the_median_under_load():
    # nvidia-smi lines: sm, max sm, power, active mask, four reasons, utilization
    s = bench.ClockSampler(0)
    s.lines = ["345, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active, 0",
               "2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active, 100",
               "2055, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active, 99",
               "2040, 2070, 980.0, 0x0, Not Active, Not Active, Not Active, Not Active, 100",
               "garbage"]
    d = s.summary()
    assert d["samples"] == 4 and d["samples_under_load"] == 3
    assert d["sm_mhz"] == 2055 and d["sm_max_mhz"] == 2070
    assert d["reasons"] == ["sw_power_cap"]


def test_ffn_and_small_group_bytes():
    # FFN: gate and up 17408 x 5120 and down 5120 x 17408 once (12,533,760 B
    # each, symmetric), x and y [M, 5120] bf16, h [M, 17408] bf16 written and read
    for M in (1, 4, 8):
        assert bench.ffn_bytes(M) == 3 * 12_533_760 + M * 5120 * 2 * 2 + 2 * M * 17408 * 2
    # metadata per 64 / 32 weights: 80 / 160 fp16 scales per 5120-weight row
    assert bench.weight_bytes_g(17408, 5120, False, 64) == 11_141_120 + 17408 * 80 * 2
    assert bench.weight_bytes_g(17408, 5120, False, 32) == 11_141_120 + 17408 * 160 * 2
    assert bench.weight_bytes_g(17408, 5120, True, 128) == bench.weight_bytes(17408, 5120, True)
