"""Host-side logic of bench.py, without a GPU: the algorithmic byte counts
each roofline divides by, the tensor classes they are split into, the
oracle sample, the all-cores oracle baseline (spawned workers) and the
source digests that key the committed DRAM traffic records."""
import json
import os

import pytest
import torch

import bench
from memory_efficient_optimizer_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N_8B = 8_030_261_248
N_1D = 65 * 4096  # 32 layers x 2 norms + the final norm


def test_llama3_8b_bytes_match_the_method_count():
    """Three reads of bf16 g, p read + write and the factored state: the
    method's 14 B per value plus the tiny row/col state."""
    wl = synth.workload("llama3_8b")
    step, impl, slots = bench.algorithmic_bytes(wl.shapes, 2, False)
    assert wl.numel == N_8B
    assert 14 * N_8B < step < 14 * N_8B * 1.001
    assert impl < step  # the fused pass reads g twice instead of three times
    assert slots["k_apply[rows_bf16]"] == 61_518_653_440


def test_tensor_classes_of_the_8b_list():
    classes = {bench.tensor_class(s, 2) for _, s in synth.workload("llama3_8b").shapes}
    assert classes == {"rows_bf16", "wide_bf16", "1d"}
    assert bench.tensor_class((4096, 14336), 2) == "wide_bf16"
    assert bench.tensor_class((4096, 4096), 4) == "vec_f32"
    assert bench.tensor_class((33, 7), 2) == "flat_bf16"
    assert bench.tensor_class((8, 1024, 1024), 4) == "flat_f32"
    assert bench.tensor_class((3, 4097), 4) == "elem_f32"
    assert bench.tensor_class((17, 100003), 2) == "elem_bf16"


def test_lamb_bytes():
    slots, design, one_pass = bench.lamb_bytes(N_8B, 2)
    assert slots == {"k_lamb_moments": 22 * N_8B, "k_lamb_update": 16 * N_8B}
    assert design == 38 * N_8B and one_pass == 26 * N_8B


def test_came_bytes():
    """Every Llama-3-8B matrix takes the row-panel pass (bf16, W in 2048 ..
    14336): g is read once there, pass b has nothing to do, and pass a only
    covers the 1D norms."""
    wl = synth.workload("llama3_8b_came")
    slots, design, one_pass = bench.came_bytes(wl.shapes, 2)
    nf = N_8B - N_1D
    assert slots["k_came_panel"] == 2 * nf
    assert slots["k_came_pass_a"] == 10 * N_1D
    assert "k_came_pass_b" not in slots
    assert slots["k_came_pass_c"] == 10 * nf + 30 * N_1D
    assert slots["k_came_pass_d"] == 12 * nf
    assert design == sum(slots.values()) and one_pass == 18 * N_8B
    # fp32 gradients and narrow or odd widths keep passes a and b
    slots32, _, _ = bench.came_bytes([("w", (64, 4096)), ("e", (33, 7))], 4)
    assert slots32["k_came_pass_b"] == 4 * (64 * 4096 + 33 * 7) and "k_came_panel" not in slots32
    assert bench.came_panel((3, 2056), 2) and bench.came_panel((5, 14336), 2)
    assert not bench.came_panel((5, 16384), 2) and not bench.came_panel((5, 2040), 2)


def test_oracle_sample_is_decoder_layer_0():
    wl = synth.workload("llama3_8b")
    idx = bench.oracle_sample(wl)
    assert [wl.shapes[k][0] for k in idx] == [f"layers.0.{n}" for n, _ in synth.llama_layer_shapes()]


def test_all_cores_baseline_runs_the_oracle_in_spawned_workers():
    wl = synth.workload("tiny")
    out = bench.cpu_baseline_all_cores(wl, "tiny", steps=1)
    assert out["kind"] == "oracle" and out["cores"] == 2 and out["value"] > 0
    assert "2 tensors (131,584 values)" in out["sample"]


def test_traffic_records_are_keyed_to_their_workload_and_kernel_sources():
    """Every committed DRAM traffic record is keyed "workload/kernel" (a launch
    slot moves different bytes in different workloads) and names a kernel
    whose source digest the bench can compute; the records of different
    kernel files differ, and a workload without a record gets none."""
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert {"llama3_8b/k_apply[rows_bf16]", "llama3_8b_lamb/k_lamb_moments", "llama3_8b_came/k_came_pass_d"} <= set(rec)
    for k in rec:
        wl, kernel = k.split("/")
        assert synth.workload(wl).numel > 0
    digests = {k: bench.kernel_source_digest(k.split("/")[1]) for k in rec}
    assert len({digests["llama3_8b/k_apply[rows_bf16]"], digests["llama3_8b_lamb/k_lamb_moments"],
                digests["llama3_8b_came/k_came_pass_d"]}) == 3
    for k, entry in rec.items():
        assert entry["dram_bytes_per_full_launch"] > 0
        assert len(entry["kernel_source_sha256"]) == 64
    assert bench.traffic_record("k_apply[rows_bf16]", "llama3_8b_beta1") is None
    assert bench.traffic_record("k_apply[rows_bf16]", None) is None


@pytest.mark.parametrize("name", ["llama3_8b", "llama3_8b_lamb", "llama3_8b_came", "llama3_8b_beta1_int8"])
def test_workloads_resolve_to_a_runner(name):
    wl = synth.workload(name)
    assert wl.optimizer in bench.ORACLE_TIMERS
    assert wl.numel == N_8B


def test_flat_views_share_one_buffer_with_256_byte_offsets():
    """The e2e gradient staging: one contiguous buffer, each view at a
    256-byte offset, shapes and dtypes kept, writes through a view land in the
    buffer."""
    like = [torch.zeros(3, 5, dtype=torch.bfloat16), torch.zeros(7, dtype=torch.float32), torch.zeros(0)]
    buf, views = bench.flat_views(like, "cpu")
    assert [v.shape for v in views] == [x.shape for x in like]
    assert [v.dtype for v in views] == [x.dtype for x in like]
    base = buf.data_ptr()
    assert [v.data_ptr() - base for v in views[:2]] == [0, 256]
    assert buf.numel() == 512
    views[1].fill_(1.0)
    assert buf[256:256 + 28].view(torch.float32).sum().item() == 7.0
