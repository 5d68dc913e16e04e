"""The bench's roofline arithmetic against figures worked out by hand from the
layer's shapes, and its clock-sample filter (no GPU).

Per expert, NVFP4 storage is half a byte per weight, one E4M3 byte per 16
weights and one FP32 global scale per matrix: W13 (2I x H) and W2 (H x I) at
H = 2048, I = 512 take 1,048,576 + 131,072 + 4 and 524,288 + 65,536 + 4
bytes, 1,769,480 together.  The router costs 2HE FLOPs per token and each
routed pair 2H(2I) + 2IH = 6,291,456 FLOPs (gate/up, then down), the MLP of
the layer in "[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency", section
"Scope and related PRs"; top-10 over 512 experts with 8192 prefill tokens is
the workload of "[Perf][SM70] Optimize Qwen3.8 Flash Next prefill".
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from nvfp4_weight_mixture_gb300 import synth  # noqa: E402

PER_EXPERT = 1_048_576 + 131_072 + 4 + 524_288 + 65_536 + 4   # 1,769,480
W_R = 2048 * 512 * 2                                            # 2 MiB
PAIR_FLOPS = 2 * 2048 * 1024 + 2 * 512 * 2048                   # 6,291,456


def test_expert_bytes():
    wl = synth.WORKLOADS["decode_m1"]
    assert bench.w13_expert_bytes(wl) + bench.w2_expert_bytes(wl) == PER_EXPERT == 1_769_480


def test_decode_m1_layer():
    # ten touched experts, W_r, one token in and out
    b, f = bench.layer_accounting(synth.WORKLOADS["decode_m1"], 10, 10)
    assert b == 10 * PER_EXPERT + W_R + 4096 + 4096 == 19_800_144
    assert f == 2 * 2048 * 512 + 10 * PAIR_FLOPS == 65_011_712


def test_decode_m16_bias_layer():
    # the FP32 router bias adds E * 4 bytes
    b, f = bench.layer_accounting(synth.WORKLOADS["decode_m16_bias"], 65, 160)
    assert b == 65 * PER_EXPERT + W_R + 2 * 16 * 4096 + 512 * 4
    assert f == 16 * 2 * 2048 * 512 + 160 * PAIR_FLOPS


def test_prefill_m8192_layer_and_kernels():
    wl = synth.WORKLOADS["prefill_m8192"]
    b, f = bench.layer_accounting(wl, 512, 81920)
    assert b == 512 * PER_EXPERT + W_R + 2 * 8192 * 4096 == 975_179_776
    assert f == 8192 * 2 * 2048 * 512 + 81920 * PAIR_FLOPS == 532_575_944_704
    bound, b13, f13 = bench.kernel_accounting(wl, "w13", 512, 81920, decode=False)
    assert bound == "tensor" and f13 == 81920 * 2 * 2048 * 1024 == 343_597_383_680
    # W13 weights, x, h (FP16)
    assert b13 == 512 * 1_179_652 + 8192 * 4096 + 81920 * 1024
    bound, b2, f2 = bench.kernel_accounting(wl, "w2", 512, 81920, decode=False)
    assert bound == "tensor" and f2 == 81920 * 2 * 512 * 2048
    # W2 weights, h, FP16 partial rows
    assert b2 == 512 * 589_828 + 81920 * 1024 + 81920 * 4096
    bound, bc, _ = bench.kernel_accounting(wl, "combine", 512, 81920, decode=False)
    assert bound == "hbm" and bc == 81920 * 4096 + 8192 * 4096


def test_shared_expert_layer():
    # the shared expert is one more touched expert and one more pair per
    # token, plus the gate vector w_g (H FP16) and its 2H FLOPs per token
    wl = synth.WORKLOADS["prefill_m8192_zipf_shared"]
    b, f = bench.layer_accounting(wl, 149, 81920 + 8192)
    assert b == 149 * PER_EXPERT + W_R + 2 * 8192 * 4096 + 512 * 4 + 2048 * 2
    assert f == 8192 * 2 * 2048 * 512 + (81920 + 8192) * PAIR_FLOPS + 8192 * 2 * 2048


def test_clock_samples_outside_the_timed_region_are_dropped():
    import datetime
    def line(t, sm, reason="Not Active"):
        ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{ts}, {sm}, 2070, 900.5, 0x0, {reason}, Not Active, Not Active, Not Active"
    t0 = 1_800_000_000.0
    out = "\n".join([line(t0 - 0.2, 1000, "Active"),      # before: a slowdown, ignored
                     line(t0 + 0.05, 2070), line(t0 + 0.10, 2050), line(t0 + 0.15, 2070),
                     line(t0 + 0.6, 1200), "garbage line"])
    inside, every = bench.Clocks.parse(out, t0, t0 + 0.3)
    assert [s[0] for s in inside] == [2070.0, 2050.0, 2070.0]
    assert len(every) == 5 and "hw_slowdown" in every[0][2]
    assert all(not s[2] for s in inside)
