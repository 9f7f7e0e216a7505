"""The bench's host-side bookkeeping, on the CPU: the work per step of the
headline and Llama-2-7B workloads (written out here from the layer shapes),
the GEMM list of a step, the algorithmic bytes per GEMM launch, the host-link
floor, and the traffic record's hash check."""
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (in features, out features) of the five linears of one block
LLAMA70B = [(8192, 10240), (8192, 8192), (8192, 28672), (8192, 28672), (28672, 8192)]
LLAMA7B = [(4096, 12288), (4096, 4096), (4096, 11008), (4096, 11008), (11008, 4096)]


def test_headline_work_per_step():
    # fwd + dgrad + wgrad = 6 M N K per linear, two micro-batches of 4096 tokens
    want = 2 * sum(6 * 4096 * n * k for k, n in LLAMA70B)
    assert bench.LLAMA70B.flops_step() == pytest.approx(want, rel=1e-12)
    assert want / 1e12 == pytest.approx(42.06, abs=0.01)


def test_llama7b_work_per_step():
    # one micro-batch of 8192 tokens
    want = sum(6 * 8192 * n * k for k, n in LLAMA7B)
    assert bench.LLAMA7B.flops_step() == pytest.approx(want, rel=1e-12)
    assert want / 1e12 == pytest.approx(9.95, abs=0.01)


@pytest.mark.parametrize("wl,shapes,tokens", [(bench.LLAMA70B, LLAMA70B, 4096),
                                              (bench.LLAMA7B, LLAMA7B, 8192)])
def test_step_gemms_and_their_algorithmic_bytes(wl, shapes, tokens):
    g = bench.step_gemms(wl)
    assert len(g) == 3 * len(shapes)
    for (k, n), fwd, dgrad, wgrad in zip(shapes, g[0::3], g[1::3], g[2::3]):
        assert fwd[1:4] == (tokens, n, k) and fwd[5] == "bf16"          # Y = X W^T
        assert dgrad[1:4] == (tokens, k, n) and dgrad[5] == "bf16"      # dX = dY W
        assert wgrad[1:4] == (n, k, tokens) and wgrad[5] == "f32acc"    # dW += dY^T X
    # one byte per operand element read once; bf16 output written once, FP32
    # accumulation read and written
    per = []
    for k, n in shapes:
        m = tokens
        per += [m * k + n * k + 2 * m * n,
                m * n + k * n + 2 * m * k,
                n * m + k * m + 8 * n * k]
    assert bench.gemm_alg_bytes(wl) == pytest.approx(sum(per) / len(per), rel=1e-12)


def test_link_floor():
    link = {"h2d_gbs": 200.0, "d2h_gbs": 150.0, "h2d_concurrent_gbs": 100.0,
            "d2h_concurrent_gbs": 50.0}
    # 100 GB in, 100 GB out: both directions at their concurrent rates until
    # the input is done (1 s, 50 GB out), the other 50 GB out at 150 GB/s
    assert bench._link_floor_ms(100e9, 100e9, link) == pytest.approx(1000 + 1000 / 3)
    # only one direction: its concurrent rate until the empty other is done
    # (at once), then its one-way rate
    assert bench._link_floor_ms(200e9, 0, link) == pytest.approx(1000.0)


def test_traffic_record_is_tied_to_the_gemm_source():
    rec = json.load(open(os.path.join(ROOT, "profiles", "gemm_step_traffic.json")))
    for key in ("llama2-70b", "llama2-7b"):
        w = rec["workloads"][key]
        assert len(w["gemm_cu_sha256"]) == 64
        assert w["bytes_per_launch"] > w["algorithmic_bytes_per_launch"] > 0
        assert w["algorithmic_bytes_per_launch"] == round(bench.gemm_alg_bytes(bench.WORKLOADS[key]))
        got = bench._gemm_traffic(key)
        assert got in (None, w["bytes_per_launch"])   # None once gemm.cu has changed
    assert bench._gemm_traffic("no-such-workload") is None
